"""CUDA path against the CPU oracle, element by element, through the C ABI.

Bars (from the method's statement of parity):
  - accept lengths and tokens bit-exact, except rows the oracle flags as
    boundary cases (a uniform within 1e-6 of a ratio or CDF boundary), which
    are counted and reported;
  - greedy rows exact; outcome keys and hit flags exact;
  - p_i(x_i), q_i(x_i) within 1e-5 absolute (fp32 against fp64);
  - row-status error bits exact.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_50_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

PROB_TOL = 1e-5


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


def to_dev(a, dtype_name):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype_name == wl.BF16 and t.dtype == torch.int16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def gpu_verify(sv, data, target=None, draft=None):
    spec = data["spec"]
    tgt = to_dev(data["target"], spec.dtype) if target is None else target
    dft = to_dev(data["draft"], spec.dtype) if draft is None else draft
    out = sv.specv_verify(tgt, dft, to_dev(data["tokens"], None),
                          to_dev(data["temperature"], None), to_dev(data["uniforms"], None))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def differing_rows(g, o) -> int:
    """Rows whose accept length or tokens differ between the GPU and the oracle."""
    return int(((g["accept_len"] != o["accept_len"]) |
                (g["out_tokens"] != o["out_tokens"]).any(axis=1)).sum())


def compare_verify(g, o, temps, label=""):
    """Assert the parity bars; return the number of boundary rows."""
    err = o["status"] & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err), label
    bnd = o["boundary"].astype(bool)
    ok = ~bnd
    assert not (bnd & (temps == 0)).any(), "greedy rows are never boundary cases"
    mism = ok & ((g["accept_len"] != o["accept_len"]) |
                 (g["out_tokens"] != o["out_tokens"]).any(axis=1))
    if mism.any():
        b = int(np.argmax(mism))
        raise AssertionError(
            f"{label}: {int(mism.sum())} non-boundary rows differ; first b={b}: "
            f"gpu n={g['accept_len'][b]} toks={g['out_tokens'][b]} | oracle n={o['accept_len'][b]} "
            f"toks={o['out_tokens'][b]} T={temps[b]}")
    fb = ok & (err == 0)
    assert np.array_equal(g["row_status"][fb] & oracle.ROW_FALLBACK,
                          o["status"][fb] & oracle.ROW_FALLBACK), label
    good = err == 0
    dp = np.abs(g["p_draft"][good] - o["p"][good]).max(initial=0.0)
    dq = np.abs(g["q_draft"][good] - o["q"][good]).max(initial=0.0)
    assert dp <= PROB_TOL and dq <= PROB_TOL, (label, dp, dq)
    same = (g["accept_len"] == o["accept_len"]) & (g["out_tokens"] == o["out_tokens"]).all(axis=1)
    print(f"[{label}] boundary rows {int(bnd.sum())}/{len(bnd)} (of which identical anyway: "
          f"{int((bnd & same).sum())}); max |dp| {dp:.2e} |dq| {dq:.2e}")
    return int(bnd.sum())


def oracle_verify(olib, data):
    return oracle.verify(data["target"], data["draft"], data["tokens"], data["temperature"],
                         data["uniforms"], nthreads=0, lib=olib)


@pytest.mark.parametrize("name", ["cfg1", "cfg2a", "cfg2b", "cfg3"])
def test_verify_configs(sv, olib, name):
    data = wl.generate(wl.SPECS[name])
    g = gpu_verify(sv, data)
    o = oracle_verify(olib, data)
    nb = compare_verify(g, o, data["temperature"], name)
    print(f"{name}: boundary rows {nb}/{len(o['boundary'])}, mean accept "
          f"{o['accept_len'].mean():.3f}")
    assert nb <= max(1, len(o["boundary"]) // 50)


def test_ssd_round_cfg4(sv, olib):
    """Config 4: verify on the SSD draft layout [B, K+1, V], predict F=6 keys
    at every lookahead, hit check against the realised outcome."""
    spec = wl.SPECS["cfg4"]
    data = wl.generate(spec)
    tgt = to_dev(data["target"], spec.dtype)
    dft = to_dev(data["draft"], spec.dtype)
    assert dft.shape[1] == spec.K + 1
    g = gpu_verify(sv, data, tgt, dft)
    o = oracle_verify(olib, data)
    compare_verify(g, o, data["temperature"], "cfg4")
    tok = to_dev(data["tokens"], None)
    pr = sv.specv_predict_outcomes(dft, tok, spec.F)
    hit = sv.specv_check_hit(pr["keys"], to_dev(g["accept_len"], None), to_dev(g["out_tokens"], None))
    torch.cuda.synchronize()
    op = oracle.predict(data["draft"], data["tokens"], spec.F, nthreads=0, lib=olib)
    assert np.array_equal(pr["keys"].cpu().numpy(), op["keys"])
    assert np.array_equal(pr["key_logits"].cpu().numpy(), op["key_logits"])
    assert np.array_equal(pr["row_status"].cpu().numpy(), op["status"])
    # the hit flag of the GPU outcome, recomputed by the oracle's definition
    oh = oracle.check_hit(op["keys"], g["accept_len"], g["out_tokens"], lib=olib)
    assert np.array_equal(hit.cpu().numpy(), oh)
    print(f"cfg4: hit rate {oh.mean():.3f}")


def test_cfg5_full_size(sv, olib):
    """Config 5 at full size (B=256, K=8, V=152064 fp32) in the launch
    configuration the benchmark times: every row against the oracle, the
    boundary rows of the whole batch counted and bounded."""
    spec = wl.SPECS["cfg5"]
    data = wl.generate(spec)
    g = gpu_verify(sv, data)
    B, K = spec.B, spec.K
    n = g["accept_len"]
    assert ((n >= 0) & (n <= K)).all()
    assert (g["row_status"] & oracle.ROW_ERRORS == 0).all()
    for b in range(B):
        assert (g["out_tokens"][b, :n[b]] == data["tokens"][b, :n[b]]).all()
        assert 0 <= g["out_tokens"][b, n[b]] < spec.V
        assert (g["out_tokens"][b, n[b] + 1:] == -1).all()
    o = oracle_verify(olib, data)
    nb = compare_verify(g, o, data["temperature"], "cfg5")
    nd = differing_rows(g, o)
    print(f"cfg5: boundary rows {nb}/{B}, differing rows {nd}; mean accept {n.mean():.3f}")
    assert nd <= max(1, B // 50)


def test_predict_full_size_cfg5_layout(sv, olib):
    """Outcome prediction at V=152064 fp32 with K+1 draft rows, F=6 and F=32."""
    spec = wl.custom("pred5", B=8, K=8, V=152064, dtype=wl.FP32, kind="zipf",
                     draft_scale=0.8, ssd=True, seed=wl.SEED_BASE + 5100)
    data = wl.generate(spec)
    dft = to_dev(data["draft"], spec.dtype)
    tok = to_dev(data["tokens"], None)
    for F in (6, 32):
        pr = sv.specv_predict_outcomes(dft, tok, F)
        torch.cuda.synchronize()
        op = oracle.predict(data["draft"], data["tokens"], F, nthreads=0, lib=olib)
        assert np.array_equal(pr["keys"].cpu().numpy(), op["keys"]), F
        assert np.array_equal(pr["key_logits"].cpu().numpy(), op["key_logits"]), F


# ---------------------------------------------------------------------------
# sizes that span several tiles, ragged tails, every cluster width, layouts

RAGGED = [
    # (B, K, V, dtype, temps)  -- V sets the cluster width: ceil(V/8192), <= 16
    (3, 2, 1, wl.FP32, (1.0,)),
    (3, 2, 2, wl.BF16, (0.7,)),
    (4, 3, 3, wl.FP32, (0.0, 1.0)),
    (4, 3, 33, wl.BF16, (0.0, 0.6, 1.0)),
    (5, 4, 4097, wl.FP32, (0.0, 0.6, 1.0)),
    (5, 4, 8193, wl.BF16, (0.3, 1.5)),
    (4, 5, 20001, wl.FP32, (1.0,)),
    (4, 5, 70003, wl.BF16, (0.8,)),
    (3, 6, 131071, wl.FP32, (0.5, 1.0)),
    (3, 7, 152064, wl.BF16, (0.0, 1.0)),
    (4, 32, 4096, wl.FP32, (1.0,)),
    (2, 1, 128256, wl.BF16, (1.0,)),
]


@pytest.mark.parametrize("B,K,V,dtype,temps", RAGGED)
def test_verify_ragged(sv, olib, B, K, V, dtype, temps):
    spec = wl.custom(f"rag{V}", B=B, K=K, V=V, dtype=dtype, temps=temps,
                     sigma_d=(0.3, 2.0), seed=wl.SEED_BASE + 7000 + V)
    data = wl.generate(spec)
    g = gpu_verify(sv, data)
    o = oracle_verify(olib, data)
    compare_verify(g, o, data["temperature"], f"V={V}")


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
@pytest.mark.parametrize("V", [1000, 4101, 40000])
def test_verify_padded_and_sliced_layouts(sv, olib, dtype, V):
    """Row stride > V (16-byte aligned rows: vector path with a ragged tail)
    and a batch slice of a larger tensor (unaligned rows: element path)."""
    spec = wl.custom(f"pad{V}", B=6, K=3, V=V, dtype=dtype, temps=(0.0, 0.9),
                     seed=wl.SEED_BASE + 7500 + V)
    data = wl.generate(spec)
    pad = (-V) % 16 + 16
    for layout in ("padded", "offset"):
        if layout == "padded":
            t = np.zeros(data["target"].shape[:2] + (V + pad,), data["target"].dtype)
            d = np.zeros(data["draft"].shape[:2] + (V + pad,), data["draft"].dtype)
            t[..., :V] = data["target"]
            d[..., :V] = data["draft"]
            tt, dd = to_dev(t, dtype)[..., :V], to_dev(d, dtype)[..., :V]
        else:
            t = np.zeros(data["target"].shape[:2] + (V + 1,), data["target"].dtype)
            d = np.zeros(data["draft"].shape[:2] + (V + 1,), data["draft"].dtype)
            t[..., 1:] = data["target"]
            d[..., 1:] = data["draft"]
            tt, dd = to_dev(t, dtype)[..., 1:], to_dev(d, dtype)[..., 1:]
        g = gpu_verify(sv, data, tt, dd)
        o = oracle_verify(olib, data)
        compare_verify(g, o, data["temperature"], f"{layout} V={V}")


def _edge_batch(dtype):
    """Hand-built rows: identical logits, -inf masks, q(x)=0, zero residual,
    bad token / NaN / +inf / bad temperature, ties, extreme temperatures."""
    rng = np.random.default_rng(99)
    K, V = 3, 50
    B = 12
    zt = (rng.standard_normal((B, K + 1, V)) * 2).astype(np.float32)
    zd = (zt[:, :K] + rng.standard_normal((B, K, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    temp = np.ones(B, np.float32)
    u = rng.random((B, K + 1), dtype=np.float32)
    zd[0] = zt[0, :K]                       # identical: every draft accepted
    zt[1, :, 10:] = -np.inf                 # target masked outside [0, 10)
    zd[2, 0, tok[2, 0]] = -np.inf           # q(x_1) = 0: reject at once
    zd[3, 0] = zt[3, 0]                     # zero residual -> fallback to p
    zt[3, 0, tok[3, 0]] = -np.inf
    zd[3, 0, tok[3, 0]] = -np.inf
    tok[4, 1] = V                           # bad token
    zt[5, 2, 7] = np.nan                    # NaN
    zd[6, 1, 3] = np.inf                    # +inf
    temp[7] = -0.5                          # bad temperature
    temp[8] = 0.0                           # greedy with ties
    zt[8, :, :] = 0.0
    zd[8, :, :] = 0.0
    tok[8] = 0
    temp[9] = 0.05                          # very low temperature
    temp[10] = 7.0                          # very high temperature
    zt[11, 1, :] = -np.inf                  # a target row with no finite logit
    if dtype == wl.BF16:
        zt = wl.f32_to_bf16_bits(zt)
        zd = wl.f32_to_bf16_bits(zd)
    spec = wl.custom("edge", B=B, K=K, V=V, dtype=dtype)
    return dict(spec=spec, target=zt, draft=zd, tokens=tok, temperature=temp, uniforms=u)


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
def test_verify_edge_cases(sv, olib, dtype):
    data = _edge_batch(dtype)
    g = gpu_verify(sv, data)
    o = oracle_verify(olib, data)
    compare_verify(g, o, data["temperature"], "edge")
    assert o["accept_len"][0] == 3 and g["accept_len"][0] == 3
    assert g["accept_len"][2] == 0
    assert g["row_status"][3] & oracle.ROW_FALLBACK
    assert g["row_status"][4] == oracle.ROW_BAD_TOKEN
    assert g["row_status"][5] == oracle.ROW_NONFINITE
    assert g["row_status"][6] == oracle.ROW_NONFINITE
    assert g["row_status"][7] == oracle.ROW_BAD_TEMP
    assert g["row_status"][11] == oracle.ROW_NONFINITE
    assert g["out_tokens"][8].tolist() == [0, 0, 0, 0]


def test_empty_batch(sv):
    z = torch.zeros((0, 4, 16), device="cuda")
    out = sv.specv_verify(z, z[:, :3], torch.zeros((0, 3), dtype=torch.int32, device="cuda"),
                          torch.zeros(0, device="cuda"), torch.zeros((0, 4), device="cuda"))
    assert out["accept_len"].numel() == 0
    assert sv.last_launch_count() == 0


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
def test_predict_edge_cases(sv, olib, dtype):
    """Ties (bf16 grid values), F > V-1, exclusion, bad token, NaN row."""
    rng = np.random.default_rng(5)
    B, K, V, F = 4, 3, 37, 8
    z = (rng.integers(-2, 3, (B, K + 1, V)) * 0.5).astype(np.float32)
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    tok[1, 2] = -3
    z[2, 1, 5] = np.nan
    zz = wl.f32_to_bf16_bits(z) if dtype == wl.BF16 else z
    dft = to_dev(zz, dtype)
    for F_ in (F, 1, 32):
        pr = sv.specv_predict_outcomes(dft, to_dev(tok, None), F_)
        torch.cuda.synchronize()
        op = oracle.predict(zz, tok, F_, lib=olib)
        assert np.array_equal(pr["keys"].cpu().numpy(), op["keys"]), F_
        assert np.array_equal(pr["key_logits"].cpu().numpy(), op["key_logits"]), F_
        assert np.array_equal(pr["row_status"].cpu().numpy(), op["status"]), F_
    small = to_dev(zz[:, :, :4], dtype)
    pr = sv.specv_predict_outcomes(small, to_dev(np.clip(tok, 0, 3), None), 6)
    op = oracle.predict(np.ascontiguousarray(zz[:, :, :4]), np.clip(tok, 0, 3), 6, lib=olib)
    assert np.array_equal(pr["keys"].cpu().numpy(), op["keys"])


def test_check_hit_matches_definition(sv, olib):
    rng = np.random.default_rng(8)
    B, K, F = 200, 4, 3
    keys = rng.integers(0, 20, (B, K + 1, F)).astype(np.int32)
    n = rng.integers(-1, K + 2, B).astype(np.int32)
    toks = rng.integers(-1, 20, (B, K + 1)).astype(np.int32)
    h = sv.specv_check_hit(to_dev(keys, None), to_dev(n, None), to_dev(toks, None))
    torch.cuda.synchronize()
    assert np.array_equal(h.cpu().numpy(), oracle.check_hit(keys, n, toks, lib=olib))


def test_repeated_calls_are_deterministic(sv):
    data = wl.generate(wl.SPECS["cfg3"])
    a = gpu_verify(sv, data)
    b = gpu_verify(sv, data)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


# ---------------------------------------------------------------------------
# the fused SSD round: verification + top-F keys + hit in one pass

def oracle_ssd(olib, data, F, fanout=None):
    o = oracle_verify(olib, data)
    op = oracle.predict(data["draft"], data["tokens"], F, nthreads=0, lib=olib, fanout=fanout)
    o["status"] = o["status"] | op["status"]
    err = (o["status"] & oracle.ROW_ERRORS) != 0
    # a flagged batch row of an SSD round has no outcome (header contract)
    o["accept_len"][err] = 0
    o["out_tokens"][err] = -1
    o["p"][err] = 0.0
    o["q"][err] = 0.0
    o["boundary"][err] = 0
    keys, kl = op["keys"].copy(), op["key_logits"].copy()
    keys[err] = -1
    kl[err] = -np.inf
    return o, keys, kl


def gpu_ssd(sv, data, F, target=None, draft=None, fanout=None):
    spec = data["spec"]
    tgt = to_dev(data["target"], spec.dtype) if target is None else target
    dft = to_dev(data["draft"], spec.dtype) if draft is None else draft
    out = sv.specv_ssd_round(tgt, dft, to_dev(data["tokens"], None),
                             to_dev(data["temperature"], None), to_dev(data["uniforms"], None), F,
                             fanout=fanout)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def compare_ssd(olib, g, o, keys, kl, temps, label):
    nb = compare_verify(g, o, temps, label)
    assert np.array_equal(g["keys"], keys), label
    assert np.array_equal(g["key_logits"], kl), label
    # the hit flag of the GPU's own outcome, by the oracle's definition
    assert np.array_equal(g["hit"], oracle.check_hit(keys, g["accept_len"], g["out_tokens"], lib=olib)), label
    return nb


def test_ssd_round_cfg4_fused(sv, olib):
    spec = wl.SPECS["cfg4"]
    data = wl.generate(spec)
    g = gpu_ssd(sv, data, spec.F)
    o, keys, kl = oracle_ssd(olib, data, spec.F)
    compare_ssd(olib, g, o, keys, kl, data["temperature"], "ssd cfg4")
    print(f"ssd cfg4: hit rate {g['hit'].mean():.3f}")


def test_ssd_round_cfg5_full_size(sv, olib):
    """Config 5 sizes with K+1 draft rows and F=6, the benchmark's workload:
    every row, key and hit flag against the oracle."""
    import dataclasses
    spec = dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-ssd", ssd=True, F=6)
    data = wl.generate(spec)
    g = gpu_ssd(sv, data, spec.F)
    o, keys, kl = oracle_ssd(olib, data, spec.F)
    nb = compare_ssd(olib, g, o, keys, kl, data["temperature"], "ssd cfg5")
    nd = differing_rows(g, o)
    print(f"ssd cfg5: boundary rows {nb}/{spec.B}, differing rows {nd}; hit rate {g['hit'].mean():.3f}")
    assert nd <= max(1, spec.B // 50)


@pytest.mark.parametrize("a,r,budget", [(0.6, 1.0, 30), (0.9, 0.5, 12), (0.3, 2.0, 5)])
def test_ssd_round_geometric_fanout(sv, olib, a, r, budget):
    """Config 4 with the Theorem 12 fan-out: F_k keys at lookahead k (the rest
    -1) and the hit flag against those keys."""
    spec = wl.SPECS["cfg4"]
    data = wl.generate(spec)
    fan, _ = sv.specv_geometric_fanout(spec.K, a, r, budget)
    F = max(1, max(fan))
    g = gpu_ssd(sv, data, F, fanout=fan)
    o, keys, kl = oracle_ssd(olib, data, F, fanout=fan)
    compare_ssd(olib, g, o, keys, kl, data["temperature"], f"ssd fanout {fan}")
    for k, f in enumerate(fan):
        assert (g["keys"][:, k, f:] == -1).all()
    pr = sv.specv_predict_outcomes(to_dev(data["draft"], spec.dtype), to_dev(data["tokens"], None),
                                   F, fanout=fan)
    torch.cuda.synchronize()
    op = oracle.predict(data["draft"], data["tokens"], F, nthreads=0, lib=olib, fanout=fan)
    assert np.array_equal(pr["keys"].cpu().numpy(), op["keys"])
    assert np.array_equal(pr["key_logits"].cpu().numpy(), op["key_logits"])
    print(f"fanout {fan}: hit rate {g['hit'].mean():.3f}")


def test_ssd_round_cfg5_geometric_fanout(sv, olib):
    """Config 5 sizes, K+1 draft rows, Theorem 12 fan-out over a budget of 48
    keys (a = 0.5, r = 1): every row against the oracle."""
    import dataclasses
    spec = dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-ssd", ssd=True, F=6)
    data = wl.generate(spec)
    fan, _ = sv.specv_geometric_fanout(spec.K, 0.5, 1.0, 48)
    F = max(fan)
    g = gpu_ssd(sv, data, F, fanout=fan)
    o, keys, kl = oracle_ssd(olib, data, F, fanout=fan)
    nb = compare_ssd(olib, g, o, keys, kl, data["temperature"], "ssd cfg5 fanout")
    nd = differing_rows(g, o)
    print(f"ssd cfg5 fanout: boundary rows {nb}/{spec.B}, differing rows {nd}")
    assert nd <= max(1, spec.B // 50)


@pytest.mark.parametrize("B,K,V,dtype,F", [
    (3, 2, 5, wl.FP32, 3),
    (4, 3, 33, wl.BF16, 6),
    (4, 4, 4097, wl.FP32, 1),
    (3, 5, 20001, wl.BF16, 32),
    (3, 3, 70003, wl.FP32, 8),
    (2, 2, 152064, wl.BF16, 6),
])
def test_ssd_round_ragged(sv, olib, B, K, V, dtype, F):
    spec = wl.custom(f"ssd{V}", B=B, K=K, V=V, dtype=dtype, temps=(0.0, 0.7, 1.0),
                     sigma_d=(0.3, 2.0), ssd=True, F=F, seed=wl.SEED_BASE + 8000 + V)
    data = wl.generate(spec)
    g = gpu_ssd(sv, data, F)
    o, keys, kl = oracle_ssd(olib, data, F)
    compare_ssd(olib, g, o, keys, kl, data["temperature"], f"ssd V={V}")


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
@pytest.mark.parametrize("V", [1000, 4101, 40000])
def test_ssd_round_padded_and_sliced_layouts(sv, olib, dtype, V):
    """The fused SSD round on row stride > V (16-byte aligned rows, a ragged
    tail) and on a slice of a wider tensor (unaligned rows: the element path
    of both kernels, the keys from the register path's candidates)."""
    spec = wl.custom(f"ssdpad{V}", B=6, K=3, V=V, dtype=dtype, temps=(0.0, 0.9), ssd=True, F=6,
                     sigma_d=(0.3, 2.0), seed=wl.SEED_BASE + 8500 + V)
    data = wl.generate(spec)
    pad = (-V) % 16 + 16
    for layout in ("padded", "offset"):
        lo, w = (0, V + pad) if layout == "padded" else (1, V + 1)
        t = np.zeros(data["target"].shape[:2] + (w,), data["target"].dtype)
        d = np.zeros(data["draft"].shape[:2] + (w,), data["draft"].dtype)
        t[..., lo:lo + V] = data["target"]
        d[..., lo:lo + V] = data["draft"]
        tt, dd = to_dev(t, dtype)[..., lo:lo + V], to_dev(d, dtype)[..., lo:lo + V]
        g = gpu_ssd(sv, data, spec.F, tt, dd)
        o, keys, kl = oracle_ssd(olib, data, spec.F)
        compare_ssd(olib, g, o, keys, kl, data["temperature"], f"ssd {layout} V={V}")


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
def test_ssd_round_edge_cases(sv, olib, dtype):
    base = _edge_batch(wl.FP32)
    zt, zd = base["target"], base["draft"]
    K = zd.shape[1]
    rng = np.random.default_rng(3)
    extra = (zt[:, K:K + 1] + rng.standard_normal((zt.shape[0], 1, zt.shape[2]))).astype(np.float32)
    zd = np.concatenate([zd, extra], axis=1)
    zd[0, K, 4] = np.nan  # NaN only in draft row K: flags the batch row in an SSD round
    if dtype == wl.BF16:
        zt, zd = wl.f32_to_bf16_bits(zt), wl.f32_to_bf16_bits(zd)
    data = dict(base, target=zt, draft=zd, spec=wl.custom("edge", B=zt.shape[0], K=K, V=zt.shape[2], dtype=dtype))
    g = gpu_ssd(sv, data, 4)
    o, keys, kl = oracle_ssd(olib, data, 4)
    compare_ssd(olib, g, o, keys, kl, data["temperature"], "ssd edge")
    assert g["row_status"][0] == oracle.ROW_NONFINITE and (g["keys"][0] == -1).all()


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
def test_extreme_temperatures(sv, olib, dtype):
    """Temperatures far from 1 (0.001, 0.02, 20, 10000): the exponent
    (z - max) log2(e)/T spans hundreds, or nearly vanishes.  Same bars."""
    spec = wl.custom(f"temps{dtype}", B=32, K=4, V=20000, dtype=dtype,
                     temps=(0.001, 0.02, 20.0, 10000.0), sigma_d=(0.3, 2.0),
                     seed=wl.SEED_BASE + 33000)
    data = wl.generate(spec)
    g = gpu_verify(sv, data)
    o = oracle_verify(olib, data)
    compare_verify(g, o, data["temperature"], f"temps {dtype}")
    ssd = wl.custom(f"temps-ssd{dtype}", B=16, K=4, V=20000, dtype=dtype, F=6, ssd=True,
                    temps=(0.001, 20.0, 10000.0), sigma_d=(0.3, 2.0), seed=wl.SEED_BASE + 33100)
    d2 = wl.generate(ssd)
    g2 = gpu_ssd(sv, d2, 6)
    o2, keys, kl = oracle_ssd(olib, d2, 6)
    compare_ssd(olib, g2, o2, keys, kl, d2["temperature"], f"temps ssd {dtype}")


def test_maximum_sizes(sv, olib):
    """The largest K and F the library takes (32, 32) in an SSD round, MSS
    with 32 candidates, and a batch of 8192 rows (16384 units) against the
    oracle."""
    spec = wl.custom("maxkf", B=3, K=32, V=4097, dtype=wl.BF16, F=32, ssd=True,
                     temps=(0.0, 1.0, 1.5), sigma_d=(0.2, 0.6), seed=wl.SEED_BASE + 35000)
    data = wl.generate(spec)
    g = gpu_ssd(sv, data, 32)
    o, keys, kl = oracle_ssd(olib, data, 32)
    compare_ssd(olib, g, o, keys, kl, data["temperature"], "K=32 F=32")

    ms = wl.custom("maxm", B=16, K=1, V=300, dtype=wl.FP32, temps=(0.0, 1.0),
                   sigma_d=(1.0, 3.0), seed=wl.SEED_BASE + 35100)
    m = wl.generate_mss(ms, 32)
    nc = np.random.default_rng(1).integers(0, 33, 16).astype(np.int32)
    r = sv.specv_mss_verify(to_dev(m["target"], wl.FP32), to_dev(m["draft"], wl.FP32),
                            to_dev(m["candidates"], None), to_dev(m["temperature"], None),
                            to_dev(m["uniforms"], None), num_candidates=to_dev(nc, None))
    torch.cuda.synchronize()
    om = oracle.mss(m["target"], m["draft"], m["candidates"], m["temperature"], m["uniforms"],
                    num_cands=nc, nthreads=0, lib=olib)
    ok = om["boundary"] == 0
    assert np.array_equal(r["out_token"].cpu().numpy()[ok], om["token"][ok])
    assert np.array_equal(r["accepted"].cpu().numpy()[ok], om["accepted"][ok])
    assert np.abs(r["accept_prob"].cpu().numpy() - om["accept_prob"]).max() <= 1e-5

    big = wl.custom("bigb", B=8192, K=1, V=64, dtype=wl.FP32, temps=(0.0, 0.8, 1.0),
                    sigma_d=(0.5, 2.0), seed=wl.SEED_BASE + 35200)
    db = wl.generate(big)
    gb = gpu_verify(sv, db)
    ob = oracle_verify(olib, db)
    compare_verify(gb, ob, db["temperature"], "B=8192")
