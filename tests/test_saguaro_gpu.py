"""Saguaro sampling ("Speculative Speculative Decoding" §4.2.1), CUDA path
against the oracle: the draft-side sampler sigma_{F,C}, and an SSD round whose
drafts came from it (q = sigma in the accept test and the residual).  Tokens
exact except draws within 1e-6 of a CDF boundary; probabilities within 1e-5."""
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


def to_dev(a, dtype_name=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype_name == wl.BF16 and t.dtype == torch.int16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def near_boundary(z, T, F, C, U, tok, olib):
    """The draw lies within 1e-6 of a cumulative-sum boundary of sigma."""
    if T == 0:
        return False
    q = oracle.saguaro_probs(z, T, F, C, lib=olib)
    cs = np.cumsum(q)
    lo = cs[tok - 1] if tok > 0 else 0.0
    return abs(U - lo) < 1e-6 or abs(cs[tok] - U) < 1e-6


@pytest.mark.parametrize("V,dtype", [(37, wl.FP32), (4097, wl.BF16), (20001, wl.FP32),
                                     (152064, wl.FP32), (128256, wl.BF16)])
@pytest.mark.parametrize("F,C", [(0, 1.0), (1, 0.25), (6, 47 / 147), (32, 0.0)])
def test_sampler_matches_oracle(sv, olib, V, dtype, F, C):
    rng = np.random.default_rng(V + 7 * F)
    B = 24
    z = rng.normal(0, 2.5, (B, V)).astype(np.float32)
    z[1, : min(V, 40)] += 6.0  # a few dominant tokens (the top-F carry most mass)
    zz = wl.f32_to_bf16_bits(z) if dtype == wl.BF16 else z
    T = rng.choice([0.0, 0.7, 1.0, 1.5], B).astype(np.float32)
    U = rng.uniform(0, 1, B).astype(np.float32)
    g = sv.specv_saguaro_sample(to_dev(zz, dtype), to_dev(T), F, C, to_dev(U))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.saguaro_sample(zz, T, F, C, U, lib=olib)
    err = o["status"] & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err)
    ok = err == 0
    for b in np.nonzero(ok)[0]:
        if g["tokens"][b] != o["tokens"][b]:
            assert near_boundary(zz[b], float(T[b]), F, C, float(U[b]), int(o["tokens"][b]), olib), \
                (b, g["tokens"][b], o["tokens"][b], T[b])
        else:
            assert abs(g["q"][b] - o["q"][b]) <= PROB_TOL, (b, g["q"][b], o["q"][b])
    assert (g["tokens"][~ok] == -1).all()


@pytest.mark.parametrize("V", [6_000_000, 8_000_000])
def test_sampler_long_rows_few_batch_rows(sv, olib, V):
    """Two rows of millions of logits: one CTA per row while its segment table
    fits in shared memory (V = 6e6), a cluster per row beyond (V = 8e6)."""
    rng = np.random.default_rng(V // 1000)
    z = rng.normal(0, 2.0, (2, V)).astype(np.float32)
    z[1, :6] = 20.0  # the top keys hold most of row 1's mass: the whole-row pass
    T = np.array([1.0, 0.8], np.float32)
    U = np.array([0.37, 0.81], np.float32)
    g = sv.specv_saguaro_sample(to_dev(z), to_dev(T), 6, 0.3, to_dev(U))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.saguaro_sample(z, T, 6, 0.3, U, lib=olib)
    assert (g["row_status"] & oracle.ROW_ERRORS == 0).all()
    for b in range(2):
        if g["tokens"][b] != o["tokens"][b]:
            assert near_boundary(z[b], float(T[b]), 6, 0.3, float(U[b]), int(o["tokens"][b]), olib)
        else:
            assert abs(g["q"][b] - o["q"][b]) <= PROB_TOL


def test_sampler_law_small_vocab(sv, olib):
    """Empirical law of GPU draws on V = 6 with C = 0.2, F = 2 against sigma
    (chi-square over 60k draws across many rows of one logit vector)."""
    from scipy.stats import chisquare
    z = np.array([2.0, 1.5, 0.0, -0.5, 1.0, -2.0], np.float32)
    n = 60000
    U = np.random.default_rng(9).uniform(0, 1, n).astype(np.float32)
    g = sv.specv_saguaro_sample(to_dev(np.tile(z, (n, 1))), to_dev(np.ones(n, np.float32)),
                                2, 0.2, to_dev(U))
    torch.cuda.synchronize()
    counts = np.bincount(g["tokens"].cpu().numpy(), minlength=6)
    q = oracle.saguaro_probs(z, 1.0, 2, 0.2, lib=olib)
    assert chisquare(counts, q * n).pvalue > 1e-3


@pytest.mark.parametrize("Fs,C,fanout", [(1, 0.3, None), (4, 47 / 147, None), (6, 0.0, None),
                                         (6, 0.3, [6, 4, 2, 1, 0])])
def test_ssd_round_with_saguaro_drafts(sv, olib, Fs, C, fanout):
    """Config 4 with drafts from sigma_{Fs,C}: accept lengths, tokens, p/q,
    keys and hit against the oracle's verify(saguaro=...) + predict + hit.
    With a fan-out whose later lookaheads keep fewer keys than F_s, the
    statistics kernel must still keep F_s candidates there for the weights."""
    spec = wl.SPECS["cfg4"]
    data = wl.generate(spec)
    F = spec.F
    # draft tokens drawn from sigma on the host by the oracle (a valid input)
    B, K = data["tokens"].shape
    tok = data["tokens"].copy()
    rng = np.random.default_rng(Fs)
    for i in range(K):
        s = oracle.saguaro_sample(np.ascontiguousarray(data["draft"][:, i]), data["temperature"],
                                  Fs, C, rng.uniform(0, 1, B).astype(np.float32), lib=olib)
        tok[:, i] = np.where(s["tokens"] >= 0, s["tokens"], tok[:, i])
    out = sv.specv_ssd_round(to_dev(data["target"], spec.dtype), to_dev(data["draft"], spec.dtype),
                             to_dev(tok), to_dev(data["temperature"]), to_dev(data["uniforms"]), F,
                             saguaro=(Fs, C), fanout=fanout)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items()}
    o = oracle.verify(data["target"], data["draft"], tok, data["temperature"], data["uniforms"],
                      nthreads=0, lib=olib, saguaro=(Fs, C))
    op = oracle.predict(data["draft"], tok, F, nthreads=0, lib=olib, fanout=fanout)
    status = o["status"] | op["status"]
    err = status & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err)
    ok = (err == 0) & ~o["boundary"].astype(bool)
    assert np.array_equal(g["accept_len"][ok], o["accept_len"][ok])
    assert np.array_equal(g["out_tokens"][ok], o["out_tokens"][ok])
    good = err == 0
    assert np.abs(g["p_draft"][good] - o["p"][good]).max() <= PROB_TOL
    assert np.abs(g["q_draft"][good] - o["q"][good]).max() <= PROB_TOL
    assert np.array_equal(g["keys"][good], op["keys"][good])
    oh = oracle.check_hit(np.where(good[:, None, None], op["keys"], -1), g["accept_len"],
                          g["out_tokens"], lib=olib)
    assert np.array_equal(g["hit"], oh)
    print(f"saguaro Fs={Fs} C={C:.3f}: hit rate {g['hit'].mean():.3f}, mean accept "
          f"{g['accept_len'].mean():.2f}")


def test_ssd_round_cfg5_with_saguaro(sv, olib):
    """Config 5 sizes, Saguaro drafts (F_s = 6, C = 0.3), the benchmark's
    cfg5-ssd-saguaro workload: every row, key and hit flag against the
    oracle's verify(saguaro=...) + predict + hit."""
    spec = dataclasses.replace(wl.SPECS["cfg5"], name="cfg5-ssd", ssd=True, F=6)
    data = wl.generate(spec)
    out = sv.specv_ssd_round(to_dev(data["target"]), to_dev(data["draft"]), to_dev(data["tokens"]),
                             to_dev(data["temperature"]), to_dev(data["uniforms"]), 6,
                             saguaro=(6, 0.3))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in out.items()}
    o = oracle.verify(data["target"], data["draft"], data["tokens"], data["temperature"],
                      data["uniforms"], nthreads=0, lib=olib, saguaro=(6, 0.3))
    op = oracle.predict(data["draft"], data["tokens"], 6, nthreads=0, lib=olib)
    err = (o["status"] | op["status"]) & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err)
    good = err == 0
    ok = good & ~o["boundary"].astype(bool)
    assert np.array_equal(g["accept_len"][ok], o["accept_len"][ok])
    assert np.array_equal(g["out_tokens"][ok], o["out_tokens"][ok])
    differ = int((good & ((g["accept_len"] != o["accept_len"]) |
                          (g["out_tokens"] != o["out_tokens"]).any(axis=1))).sum())
    assert differ <= max(1, spec.B // 50), differ
    assert np.abs(g["p_draft"][good] - o["p"][good]).max() <= PROB_TOL
    assert np.abs(g["q_draft"][good] - o["q"][good]).max() <= PROB_TOL
    assert np.array_equal(g["keys"][good], op["keys"][good])
    oh = oracle.check_hit(np.where(good[:, None, None], op["keys"], -1), g["accept_len"],
                          g["out_tokens"], lib=olib)
    assert np.array_equal(g["hit"], oh)
    print(f"saguaro cfg5: boundary rows {int(o['boundary'].sum())}/{spec.B}, differing rows {differ}, "
          f"hit rate {g['hit'].mean():.3f}")
