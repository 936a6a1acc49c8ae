"""Multi-step speculative sampling at token-tree nodes ("Lecture 5 -
Speculative Decoding and SpecInfer" §6.4), CUDA path against the oracle.

Bars: status bits exact; the accepted candidate and the token exact except
on draws the oracle flags as boundary cases or where a tested candidate's
accept probability lies within ACC_TOL of its uniform (the library forms
p_j(x_j)/q(x_j) = max(0, t_j - c_j) / D_j from fp32 logits, the oracle
p_j by fp64 arrays); accept probabilities within ACC_TOL.

ACC_TOL = 1e-5, the bar for probabilities: t_j = p(x_j)/q(x_j) comes from
fp32 logits with a few ulps of error (relative 1e-7), c_j and D_j are
float-float sums of fp32 terms (relative 1e-7), so |delta a_j| <= 1e-7
(t_j + c_j + a_j D_j) / D_j, below 1e-5 while t_j, c_j <= 10 and D_j >= 0.2
(measured: below 3e-6).  A uniform within ACC_TOL of a_j may decide either
way, like a boundary row.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_50_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


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


def to_dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if bf16:
        t = t.view(torch.bfloat16)
    return t.cuda()


ACC_TOL = 1e-5


def run_pair(sv, olib, data, bf16, naive=False, num_candidates=None):
    nc_dev = to_dev(num_candidates) if num_candidates is not None else None
    g = sv.specv_mss_verify(to_dev(data["target"], bf16), to_dev(data["draft"], bf16),
                            to_dev(data["candidates"]), to_dev(data["temperature"]),
                            to_dev(data["uniforms"]), num_candidates=nc_dev, naive=naive)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.mss(data["target"], data["draft"], data["candidates"], data["temperature"],
                   data["uniforms"], num_cands=num_candidates, naive=naive, nthreads=0, lib=olib)
    return g, o


def compare(g, o, data, label):
    err = o["status"] & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err), label
    B, M = data["candidates"].shape
    near = 0
    worst = 0.0
    for b in range(B):
        if err[b]:
            assert g["out_token"][b] == -1 and g["accepted"][b] == -1, (label, b)
            continue
        tol = ACC_TOL
        worst = max(worst, float(np.abs(g["accept_prob"][b] - o["accept_prob"][b]).max()))
        assert np.abs(g["accept_prob"][b] - o["accept_prob"][b]).max() <= tol, \
            (label, b, g["accept_prob"][b], o["accept_prob"][b])
        if g["out_token"][b] == o["token"][b] and g["accepted"][b] == o["accepted"][b]:
            continue
        u = data["uniforms"][b, :M]
        close = np.abs(u - o["accept_prob"][b]) <= tol
        assert o["boundary"][b] or close.any(), \
            (label, b, g["out_token"][b], o["token"][b], g["accepted"][b], o["accepted"][b])
        near += 1
    assert near <= max(1, B // 50), (label, near)
    print(f"[{label}] max |d accept_prob| {worst:.2e}, near-boundary nodes {near}")


@pytest.mark.parametrize("V,dtype", [(37, wl.FP32), (4097, wl.BF16), (20001, wl.FP32),
                                     (152064, wl.FP32), (128256, wl.BF16)])
@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("naive", [False, True])
def test_mss_matches_oracle(sv, olib, V, dtype, M, naive):
    spec = wl.custom(f"mss{V}", B=40, K=1, V=V, dtype=dtype, temps=(0.0, 0.6, 1.0, 1.0),
                     sigma_d=(0.3, 2.5), seed=wl.SEED_BASE + 12000 + V)
    data = wl.generate_mss(spec, M)
    # some nodes whose first candidates are rejected more often: noisier drafts
    g, o = run_pair(sv, olib, data, dtype == wl.BF16, naive=naive)
    compare(g, o, data, f"V={V} M={M} naive={naive}")
    if not naive:
        acc = g["accepted"][(o["status"] & oracle.ROW_ERRORS) == 0]
        print(f"V={V} M={M}: accepted hist {np.bincount(acc + 1, minlength=M + 1).tolist()}")


def test_mss_law_is_target(sv, olib):
    """Theorem 4.2 on the GPU: 60k nodes sharing one (p, q) pair on V = 6
    with three candidates drawn i.i.d. from q; the empirical token law
    matches p (chi-square), and MSS accepts at least as often as the exact
    naive-sampling rate."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(21)
    n, V, M = 60000, 6, 3
    zt = np.array([1.2, 0.3, -0.5, 2.0, 0.0, -1.0], np.float32)
    zd = np.array([0.2, 1.5, -0.2, 0.8, 0.9, -2.0], np.float32)
    p = oracle.row_probs(zt, 1.0, lib=olib)
    q = oracle.row_probs(zd, 1.0, lib=olib)
    cands = rng.choice(V, size=(n, M), p=q).astype(np.int32)
    U = rng.uniform(0, 1, (n, M + 1)).astype(np.float32)
    g = sv.specv_mss_verify(to_dev(np.tile(zt, (n, 1))), to_dev(np.tile(zd, (n, 1))),
                            to_dev(cands), to_dev(np.ones(n, np.float32)), to_dev(U))
    torch.cuda.synchronize()
    tok = g["out_token"].cpu().numpy()
    acc = g["accepted"].cpu().numpy()
    counts = np.bincount(tok, minlength=V)
    assert chisquare(counts, p * n).pvalue > 1e-3, counts
    ns_rate = np.mean([p[np.unique(c)].sum() for c in cands[:5000]])
    assert (acc >= 0).mean() >= ns_rate - 0.01


def test_mss_counts_and_bad_inputs(sv, olib):
    """Per-node candidate counts (0..M), counts outside [0, M], candidates
    outside [0, V) and an empty batch."""
    spec = wl.custom("mssbad", B=8, K=1, V=300, dtype=wl.FP32, temps=(1.0,),
                     seed=wl.SEED_BASE + 12500)
    data = wl.generate_mss(spec, 3)
    data["candidates"][5, 1] = 300
    nc = np.array([0, 1, 2, 3, -1, 3, 4, 2], np.int32)
    g, o = run_pair(sv, olib, data, False, num_candidates=nc)
    compare(g, o, data, "counts")
    st = g["row_status"]
    assert st[4] & sv.ROW_BAD_COUNT and st[6] & sv.ROW_BAD_COUNT
    assert st[5] & oracle.ROW_BAD_TOKEN
    assert g["accepted"][0] == -1 and g["out_token"][0] >= 0  # no candidates: a draw from p
    assert (g["accept_prob"][1, 1:] == 0).all()  # untested slots stay 0
    empty = torch.empty((0, 300), dtype=torch.float32, device="cuda")
    e = sv.specv_mss_verify(empty, empty, torch.empty((0, 3), dtype=torch.int32, device="cuda"),
                            torch.empty(0, device="cuda"), torch.empty((0, 4), device="cuda"))
    assert e["accepted"].numel() == 0


def test_mss_cfg5_sizes(sv, olib):
    """The benchmark's MSS workload (2048 nodes, three candidates, V = 152064
    fp32, config 5 logits, T = 1) in the launch configuration bench.py
    times; every node against the oracle."""
    spec = wl.SPECS["cfg5"]
    data = wl.generate_mss(spec, 3, B=2048)
    g = sv.specv_mss_verify(to_dev(data["target"]), to_dev(data["draft"]),
                            to_dev(data["candidates"]), to_dev(data["temperature"]),
                            to_dev(data["uniforms"]))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.mss(data["target"], data["draft"], data["candidates"], data["temperature"],
                   data["uniforms"], nthreads=0, lib=olib)
    compare(g, o, data, "cfg5 all nodes")
    print("cfg5 nodes: accepted hist", np.bincount(g["accepted"] + 1, minlength=4).tolist())


@pytest.mark.parametrize("V,dtype", [(20001, wl.FP32), (4097, wl.BF16)])
@pytest.mark.parametrize("naive", [False, True])
def test_mss_unaligned_rows(sv, olib, V, dtype, naive):
    """Rows whose stride is not a multiple of 16 bytes take the register
    path (element loads, every pass read directly)."""
    spec = wl.custom(f"mssu{V}", B=24, K=1, V=V, dtype=dtype, temps=(0.0, 0.7, 1.0),
                     sigma_d=(0.5, 2.5), seed=wl.SEED_BASE + 34000 + V)
    data = wl.generate_mss(spec, 3)
    bf = dtype == wl.BF16

    def padded(a):  # stride V + 1 elements
        t = to_dev(np.pad(a, ((0, 0), (0, 1))), bf)
        return t[:, :V]

    g = sv.specv_mss_verify(padded(data["target"]), padded(data["draft"]),
                            to_dev(data["candidates"]), to_dev(data["temperature"]),
                            to_dev(data["uniforms"]), naive=naive)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.mss(data["target"], data["draft"], data["candidates"], data["temperature"],
                   data["uniforms"], naive=naive, nthreads=0, lib=olib)
    compare(g, o, data, f"unaligned V={V} naive={naive}")
