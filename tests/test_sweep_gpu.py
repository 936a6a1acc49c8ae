"""A seeded sweep of verification and SSD-round shapes against the oracle.

The hand-picked cases elsewhere pin the benchmark configurations and the
edge cases; this sweep draws 64 more shapes from a fixed seed, so that the
host's choices that depend on the sizes (chunk length and count, the
one-wave rule, the kernel-B cluster size and slice, the chunk-local draw,
ring or direct residual pass) meet combinations nobody picked: batch sizes
from 1 to 1216 across the cluster-size thresholds, K from 1 to 12, V from 1
to 152064, both dtypes, the three logit recipes, mixed temperatures,
drafts without probabilities (a third of the verification shapes) and
F from 1 to 12 (and below: 24 MSS shapes and 16 sampler shapes, with the
bars of tests/test_mss_gpu.py and tests/_sampler_case.py, and 16 outcome
prediction shapes with fan-outs and ties, keys exact).  Same bars as
tests/test_parity_gpu.py: every row the oracle
does not flag is exact, and at most 2 % of the rows (at least one) differ.
The flagged rows themselves are only counted: a flat row of 152064 logits
has many tokens of probability below 2e-6, and a draw of such a token is
flagged whatever U is (both ends of its CDF step lie within 1e-6 of U).
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_50_gb300 import workloads as wl
from tests.test_parity_gpu import (compare_ssd, compare_verify, differing_rows, gpu_ssd, gpu_verify,
                                    oracle_ssd, oracle_verify)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MAX_LOGITS = 60_000_000  # per case, so the oracle finishes each in a second or so


def _shapes(n=64, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(rng.choice([1, 2, 3, 7, 8, 9, 17, 31, 64, 100, 150, 256, 300, 600, 1216]))
        K = int(rng.integers(1, 13))
        band = int(rng.integers(0, 5))
        V = int([rng.integers(1, 300), rng.integers(300, 5000), rng.integers(5000, 70000),
                 128256, 152064][band])
        ssd = bool(rng.integers(0, 2))
        if B * (2 * K + 2) * V > MAX_LOGITS:
            continue
        dtype = wl.FP32 if rng.integers(0, 2) else wl.BF16
        kind = str(rng.choice(["normal", "boosted", "zipf"]))
        temps = tuple(sorted(set(float(t) for t in rng.choice([0.0, 0.5, 0.8, 1.0, 1.5],
                                                              int(rng.integers(1, 4))))))
        F = int(rng.integers(1, 13)) if ssd else 0
        nd = not ssd and len(out) % 3 == 1  # a third of the verification shapes: no draft logits
        out.append(dict(B=B, K=K, V=V, dtype=dtype, kind=kind, temps=temps, ssd=ssd, F=F, nd=nd,
                        seed=wl.SEED_BASE + 12000 + len(out)))
    return out


SHAPES = _shapes()


@pytest.fixture(scope="module")
def sv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_50_gb300 import _build
    _build.build()
    import speculative_decoding_verification_50_gb300 as m
    m.load_library()
    return m


@pytest.fixture(scope="module")
def olib():
    return oracle.load(oracle.build())


def _id(s):
    mode = f"ssdF{s['F']}" if s["ssd"] else ("verify-nodraft" if s["nd"] else "verify")
    return f"{mode}-B{s['B']}-K{s['K']}-V{s['V']}-{s['dtype']}-{s['kind']}"


@pytest.mark.parametrize("shape", SHAPES, ids=_id)
def test_sweep_matches_oracle(sv, olib, shape):
    extra = dict(boost_ids=min(8, shape["V"]), boost=6.0) if shape["kind"] == "boosted" else {}
    if shape["kind"] == "zipf":
        extra = dict(draft_scale=0.8)
    spec = wl.custom(_id(shape), B=shape["B"], K=shape["K"], V=shape["V"], dtype=shape["dtype"],
                     kind=shape["kind"], temps=shape["temps"], sigma_d=(0.3, 2.5), ssd=shape["ssd"],
                     F=shape["F"], seed=shape["seed"], **extra)
    data = wl.generate(spec)
    if shape["ssd"]:
        g = gpu_ssd(sv, data, shape["F"])
        o, keys, kl = oracle_ssd(olib, data, shape["F"])
        compare_ssd(olib, g, o, keys, kl, data["temperature"], _id(shape))
    elif shape["nd"]:  # q one-hot at each draft token (NO_DRAFT_PROBS)
        t = torch.from_numpy(np.ascontiguousarray(data["target"]))
        tgt = (t.view(torch.bfloat16) if shape["dtype"] == wl.BF16 else t).cuda()
        out = sv.specv_verify(tgt, None, torch.from_numpy(data["tokens"]).cuda(),
                              torch.from_numpy(data["temperature"]).cuda(),
                              torch.from_numpy(data["uniforms"]).cuda())
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in out.items()}
        o = oracle.verify(data["target"], None, data["tokens"], data["temperature"], data["uniforms"],
                          nthreads=0, lib=olib, no_draft=True)
        compare_verify(g, o, data["temperature"], _id(shape))
    else:
        g = gpu_verify(sv, data)
        o = oracle_verify(olib, data)
        compare_verify(g, o, data["temperature"], _id(shape))
    nd = differing_rows(g, o)
    assert nd <= max(1, shape["B"] // 50), nd


# ---- MSS nodes and the Saguaro sampler over seeded shapes -------------------

def _mss_shapes(n=24, seed=20261203):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(rng.choice([1, 3, 40, 300, 1300]))
        M = int(rng.integers(1, 9))
        band = int(rng.integers(0, 4))
        V = int([rng.integers(1, 300), rng.integers(300, 8000), rng.integers(8000, 70000), 152064][band])
        if 2 * B * V > 40_000_000:
            continue
        dtype = wl.FP32 if rng.integers(0, 2) else wl.BF16
        temps = tuple(sorted(set(float(t) for t in rng.choice([0.0, 0.6, 1.0, 1.4], int(rng.integers(1, 4))))))
        out.append(dict(B=B, M=M, V=V, dtype=dtype, temps=temps, naive=bool(rng.random() < 0.2),
                        ragged=bool(rng.random() < 0.3), seed=wl.SEED_BASE + 13000 + len(out)))
    return out


def _mss_id(s):
    return (f"mss-B{s['B']}-M{s['M']}-V{s['V']}-{s['dtype']}" + ("-naive" if s["naive"] else "") +
            ("-ragged" if s["ragged"] else ""))


@pytest.mark.parametrize("shape", _mss_shapes(), ids=_mss_id)
def test_sweep_mss_matches_oracle(sv, olib, shape):
    from tests.test_mss_gpu import compare, run_pair
    spec = wl.custom(_mss_id(shape), B=shape["B"], K=1, V=shape["V"], dtype=shape["dtype"],
                     temps=shape["temps"], sigma_d=(0.3, 2.5), seed=shape["seed"])
    data = wl.generate_mss(spec, shape["M"])
    nc = None
    if shape["ragged"]:  # per-node candidate counts 0..M
        nc = np.random.default_rng(shape["seed"]).integers(0, shape["M"] + 1, shape["B"]).astype(np.int32)
    g, o = run_pair(sv, olib, data, shape["dtype"] == wl.BF16, naive=shape["naive"], num_candidates=nc)
    compare(g, o, data, _mss_id(shape))


def _sampler_shapes(n=16, seed=20261204):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        rows = int(rng.choice([1, 5, 100, 1216, 2000]))
        band = int(rng.integers(0, 4))
        V = int([rng.integers(1, 300), rng.integers(300, 8000), rng.integers(8000, 70000), 152064][band])
        dtype = wl.FP32 if rng.integers(0, 2) else wl.BF16
        if dtype == wl.BF16:
            V += (-V) % 8  # contiguous rows stay 16-byte aligned (the vector paths)
        else:
            V += (-V) % 4
        if rows * V > 60_000_000:
            continue
        F = int(rng.integers(0, 17))
        C = float(np.round(rng.uniform(0.0, 1.0), 3)) if F else 1.0
        out.append(dict(rows=rows, V=V, dtype=dtype, F=F, C=C, sigma=float(rng.choice([1.0, 2.5, 4.0])),
                        seed=wl.SEED_BASE + 14000 + len(out)))
    return out


def _sampler_id(s):
    return f"sample-R{s['rows']}-V{s['V']}-{s['dtype']}-F{s['F']}-C{s['C']}"


@pytest.mark.parametrize("shape", _sampler_shapes(), ids=_sampler_id)
@pytest.mark.parametrize("layout", ["contiguous", "offset"])
def test_sweep_sampler_matches_oracle(sv, olib, shape, layout):
    """specv_saguaro_sample (one warp per row from 1216 rows of aligned rows,
    one CTA per row otherwise) against the oracle, on contiguous rows and on
    unaligned rows (one element into a wider buffer): error bits exact, tokens
    exact except draws within 1e-6 of a CDF step, sigma(token) within 1e-5."""
    from tests._sampler_case import near_boundary
    rng = np.random.default_rng(shape["seed"])
    rows, V, F, C = shape["rows"], shape["V"], shape["F"], shape["C"]
    z = (rng.standard_normal((rows, V)) * shape["sigma"]).astype(np.float32)
    T = rng.choice([0.0, 0.7, 1.0, 1.3], rows).astype(np.float32)
    U = rng.uniform(0, 1, rows).astype(np.float32)
    bf16 = shape["dtype"] == wl.BF16
    zz = wl.f32_to_bf16_bits(z) if bf16 else z
    if layout == "offset":  # rows one element into a wider buffer: unaligned, the element paths
        wide = np.zeros((rows, V + 1), zz.dtype)
        wide[:, 1:] = zz
        zt = torch.from_numpy(wide)
    else:
        zt = torch.from_numpy(np.ascontiguousarray(zz))
    zdev = (zt.view(torch.bfloat16) if bf16 else zt).cuda()
    if layout == "offset":
        zdev = zdev[:, 1:]
    g = sv.specv_saguaro_sample(zdev, torch.from_numpy(T).cuda(), F, C, torch.from_numpy(U).cuda())
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.saguaro_sample(zz, T, F, C, U, lib=olib)
    err = o["status"] & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err)
    differ = 0
    for b in np.nonzero(err == 0)[0]:
        if g["tokens"][b] != o["tokens"][b]:
            assert near_boundary(zz[b], float(T[b]), F, C, float(U[b]), int(o["tokens"][b]), olib), \
                (b, g["tokens"][b], o["tokens"][b], T[b])
            differ += 1
        else:
            assert abs(g["q"][b] - o["q"][b]) <= 1e-5, (b, g["q"][b], o["q"][b])
    assert differ <= max(1, rows // 50), differ
    print(f"[{_sampler_id(shape)} {layout}] differing rows {differ}/{rows}")


def _predict_shapes(n=16, seed=20261205):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(rng.choice([1, 3, 32, 100, 700]))
        K = int(rng.integers(1, 13))
        band = int(rng.integers(0, 4))
        V = int([rng.integers(1, 300), rng.integers(300, 8000), rng.integers(8000, 70000), 152064][band])
        if B * (K + 1) * V > 40_000_000:
            continue
        dtype = wl.FP32 if rng.integers(0, 2) else wl.BF16
        F = int(rng.integers(1, 33))
        fan = None
        if rng.random() < 0.4:  # a per-lookahead fan-out (any counts in 0..F)
            fan = [int(x) for x in rng.integers(0, F + 1, K + 1)]
        out.append(dict(B=B, K=K, V=V, dtype=dtype, F=F, fan=fan, grid=bool(rng.random() < 0.3),
                        seed=wl.SEED_BASE + 15000 + len(out)))
    return out


def _predict_id(s):
    return (f"predict-B{s['B']}-K{s['K']}-V{s['V']}-{s['dtype']}-F{s['F']}" +
            ("-fan" if s["fan"] else "") + ("-ties" if s["grid"] else ""))


@pytest.mark.parametrize("shape", _predict_shapes(), ids=_predict_id)
def test_sweep_predict_matches_oracle(sv, olib, shape):
    """specv_predict_outcomes (keys and key logits exact, ties included: some
    shapes draw logits on a coarse grid) and specv_check_hit on random
    outcomes against those keys."""
    rng = np.random.default_rng(shape["seed"])
    B, K, V, F = shape["B"], shape["K"], shape["V"], shape["F"]
    if shape["grid"]:
        z = (rng.integers(-4, 5, (B, K + 1, V)) * 0.5).astype(np.float32)
    else:
        z = (rng.standard_normal((B, K + 1, V)) * 2.0).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    zz = wl.f32_to_bf16_bits(z) if shape["dtype"] == wl.BF16 else z
    t = torch.from_numpy(np.ascontiguousarray(zz))
    dft = (t.view(torch.bfloat16) if shape["dtype"] == wl.BF16 else t).cuda()
    pr = sv.specv_predict_outcomes(dft, torch.from_numpy(tok).cuda(), F, fanout=shape["fan"])
    torch.cuda.synchronize()
    op = oracle.predict(zz, tok, F, nthreads=0, lib=olib, fanout=shape["fan"])
    keys = pr["keys"].cpu().numpy()
    assert np.array_equal(keys, op["keys"])
    assert np.array_equal(pr["key_logits"].cpu().numpy(), op["key_logits"])
    assert np.array_equal(pr["row_status"].cpu().numpy(), op["status"])
    n = rng.integers(-1, K + 2, B).astype(np.int32)
    outs = rng.integers(-1, V, (B, K + 1)).astype(np.int32)
    for b in range(0, B, 3):  # some outcomes that are keys
        if 0 <= n[b] <= K:
            outs[b, n[b]] = keys[b, n[b], 0]
    h = sv.specv_check_hit(pr["keys"], torch.from_numpy(n).cuda(), torch.from_numpy(outs).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy(), oracle.check_hit(op["keys"], n, outs, lib=olib))
