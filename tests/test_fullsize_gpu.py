"""The benchmark's other config 5 workloads at full size, in the launch
configuration bench.py times (inputs laid out by bench.py's own code):
the Saguaro sampler over the 2304 draft rows of a round (16-trip chunks, the
32-tile chunk-local draw), per-row draft counts over packed rows, and
verification without draft logits.  Sampled rows against the oracle, the
same bars as the smaller cases (tokens and accept lengths exact except
boundary rows, probabilities within 1e-5, error bits exact)."""
import dataclasses

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


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_sampler_full_size_sampled(sv, olib, bench):
    spec, _ = bench.WORKLOADS["cfg5-sample"]
    F, C = bench.SAGUARO["cfg5-sample"]
    lay = bench.lay_out(wl.generate(spec), spec, "sample")
    z, T, U = lay["draft"], lay["temperature"], lay["uniforms"]
    g = sv.specv_saguaro_sample(dev(z), dev(T), F, C, dev(U))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    n = z.shape[0]
    assert n == 2304 and (g["row_status"] & oracle.ROW_ERRORS == 0).all()
    assert ((g["tokens"] >= 0) & (g["tokens"] < spec.V)).all()
    rows = np.random.default_rng(11).choice(n, 32, replace=False)
    o = oracle.saguaro_sample(z[rows], T[rows], F, C, U[rows], lib=olib)
    for k, b in enumerate(rows):
        if g["tokens"][b] == o["tokens"][k]:
            assert abs(g["q"][b] - o["q"][k]) <= PROB_TOL, (b, g["q"][b], o["q"][k])
            continue
        q = oracle.saguaro_probs(z[b], float(T[b]), F, C, lib=olib)
        cs = np.cumsum(q)
        t = int(o["tokens"][k])
        lo = cs[t - 1] if t > 0 else 0.0
        assert min(abs(U[b] - lo), abs(cs[t] - U[b])) < 1e-6, (b, g["tokens"][b], t)


def test_ragged_full_size_sampled(sv, olib, bench):
    spec, _ = bench.WORKLOADS["cfg5-ragged"]
    data = wl.generate(spec)
    lay = bench.lay_out(data, spec, "ragged")
    K, B = spec.K, spec.B
    cu = lay["cu"]
    g = sv.specv_verify_ragged(dev(lay["target"]), dev(lay["draft"]), dev(cu), dev(lay["tokens"]),
                               dev(lay["temperature"]), dev(lay["uniforms"]), K)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    kb = np.diff(np.concatenate([[0], cu]))
    assert (g["accept_len"] <= kb).all() and (g["row_status"] & oracle.ROW_ERRORS == 0).all()
    rows = np.sort(np.random.default_rng(12).choice(B, 16, replace=False))
    sub = {k: data[k][rows] for k in ("target", "draft", "tokens", "temperature", "uniforms")}
    kr = kb[rows]
    cu_s = np.cumsum(kr).astype(np.int32)
    tgt = np.concatenate([sub["target"][i, :kr[i] + 1] for i in range(len(rows))])
    dft = np.concatenate([sub["draft"][i, :kr[i]] for i in range(len(rows))])
    tok = np.concatenate([sub["tokens"][i, :kr[i]] for i in range(len(rows))]).astype(np.int32)
    uni = np.concatenate([np.append(sub["uniforms"][i, :kr[i]], sub["uniforms"][i, -1])
                          for i in range(len(rows))]).astype(np.float32)
    o = oracle.verify_ragged(tgt, dft, cu_s, tok, sub["temperature"], uni, K, nthreads=0, lib=olib)
    ok = o["boundary"] == 0
    assert np.array_equal(g["accept_len"][rows][ok], o["accept_len"][ok])
    assert np.array_equal(g["out_tokens"][rows][ok], o["out_tokens"][ok])
    c0 = np.concatenate([[0], cu[:-1]])
    gp = np.concatenate([g["p_draft"][c0[b]:cu[b]] for b in rows])
    gq = np.concatenate([g["q_draft"][c0[b]:cu[b]] for b in rows])
    assert np.abs(gp - o["p"]).max(initial=0) <= PROB_TOL
    assert np.abs(gq - o["q"]).max(initial=0) <= PROB_TOL


def test_no_draft_full_size_sampled(sv, olib, bench):
    spec, _ = bench.WORKLOADS["cfg5-nodraft"]
    data = wl.generate(spec)
    g = sv.specv_verify(dev(data["target"]), None, dev(data["tokens"]),
                        dev(data["temperature"]), dev(data["uniforms"]))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    assert (g["row_status"] & oracle.ROW_ERRORS == 0).all()
    rows = np.random.default_rng(13).choice(spec.B, 16, replace=False)
    o = oracle.verify(data["target"][rows], None, data["tokens"][rows], data["temperature"][rows],
                      data["uniforms"][rows], nthreads=0, lib=olib, no_draft=True)
    ok = o["boundary"] == 0
    assert np.array_equal(g["accept_len"][rows][ok], o["accept_len"][ok])
    assert np.array_equal(g["out_tokens"][rows][ok], o["out_tokens"][ok])
    assert np.abs(g["p_draft"][rows] - o["p"]).max() <= PROB_TOL
    assert (g["q_draft"] == 1.0).all()
