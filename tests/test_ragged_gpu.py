"""Per-row draft counts and drafts without probabilities, CUDA path against
the oracle ("Speculative Decoding" dl-note, Appendix: cu_num_draft_tokens and
NO_DRAFT_PROBS).  Same bars as tests/test_parity_gpu.py: tokens and accept
lengths exact except oracle-flagged boundary rows, p/q within 1e-5, error
bits exact."""
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


def pack(data, kb):
    """Pack a strided batch into the per-row-count layout with K_b drafts."""
    B = len(kb)
    cu = np.cumsum(kb).astype(np.int32)
    tgt = np.concatenate([data["target"][b, :kb[b] + 1] for b in range(B)])
    dft = np.concatenate([data["draft"][b, :kb[b]] for b in range(B)] +
                         [np.zeros((0, data["target"].shape[-1]), data["target"].dtype)])
    tok = np.concatenate([data["tokens"][b, :kb[b]] for b in range(B)] + [np.zeros(0, np.int32)])
    uni = np.concatenate([np.append(data["uniforms"][b, :kb[b]], data["uniforms"][b, -1])
                          for b in range(B)]).astype(np.float32)
    return cu, tgt, dft, tok.astype(np.int32), uni


def compare_rows(g, o, kb, cu, temps, label):
    err = o["status"] & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err), label
    ok = ~o["boundary"].astype(bool)
    assert not (o["boundary"].astype(bool) & (temps == 0)).any()
    mism = ok & ((g["accept_len"] != o["accept_len"]) |
                 (g["out_tokens"] != o["out_tokens"]).any(axis=1))
    assert not mism.any(), (label, np.nonzero(mism)[0][:5], g["out_tokens"][mism][:3],
                            o["out_tokens"][mism][:3])
    for b in range(len(kb)):
        if err[b]:
            continue
        c0 = 0 if b == 0 else int(cu[b - 1])
        sl = slice(c0, c0 + int(kb[b]))
        assert np.abs(g["p_draft"][sl] - o["p"][sl]).max(initial=0) <= PROB_TOL, (label, b)
        assert np.abs(g["q_draft"][sl] - o["q"][sl]).max(initial=0) <= PROB_TOL, (label, b)
    print(f"[{label}] boundary rows {int(o['boundary'].sum())}/{len(kb)}")


def run_pair(sv, olib, data, kb, K, dtype, no_draft, label):
    cu, tgt, dft, tok, uni = pack(data, kb)
    temps = data["temperature"]
    g = sv.specv_verify_ragged(to_dev(tgt, dtype), None if no_draft else to_dev(dft, dtype),
                               to_dev(cu), to_dev(tok), to_dev(temps), to_dev(uni), K)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.verify_ragged(tgt, None if no_draft else dft, cu, tok, temps, uni, K,
                             nthreads=0, lib=olib, no_draft=no_draft)
    compare_rows(g, o, kb, cu, temps, label)
    return g, o


@pytest.mark.parametrize("B,K,V,dtype", [
    (6, 3, 37, wl.FP32),
    (8, 4, 4097, wl.BF16),
    (5, 6, 20001, wl.FP32),
    (4, 8, 131071, wl.BF16),
    (300, 4, 50000, wl.FP32),  # clusters of 2: bonus and no-draft draws from one chunk
])
@pytest.mark.parametrize("no_draft", [False, True])
def test_ragged_rows(sv, olib, B, K, V, dtype, no_draft):
    spec = wl.custom(f"rag{V}", B=B, K=K, V=V, dtype=dtype, temps=(0.0, 0.7, 1.0),
                     sigma_d=(0.3, 2.0), seed=wl.SEED_BASE + 9000 + V)
    data = wl.generate(spec)
    kb = np.random.default_rng(V).integers(0, K + 1, B)
    kb[0], kb[-1] = 0, K  # a row with no drafts and a full row
    g, o = run_pair(sv, olib, data, kb, K, dtype, no_draft, f"ragged V={V} nd={no_draft}")
    assert (g["accept_len"] <= kb).all()
    for b in range(B):
        assert (g["out_tokens"][b, g["accept_len"][b] + 1:] == -1).all()


@pytest.mark.parametrize("dtype", [wl.FP32, wl.BF16])
def test_no_draft_probs_strided(sv, olib, dtype):
    """The strided layout without draft logits (draft = None)."""
    spec = wl.custom("nd", B=12, K=4, V=8193, dtype=dtype, temps=(0.0, 0.6, 1.0),
                     sigma_d=(0.3, 2.0), seed=wl.SEED_BASE + 9500)
    data = wl.generate(spec)
    # drafts the target often accepts: its own argmax half the time
    tok = data["tokens"].copy()
    zt = data["target"].astype(np.float32) if dtype == wl.FP32 else \
        wl.bf16_bits_to_f32(data["target"])
    tok[::2] = np.argmax(zt[::2, :spec.K], axis=-1)
    g = sv.specv_verify(to_dev(data["target"], dtype), None, to_dev(tok),
                        to_dev(data["temperature"]), to_dev(data["uniforms"]))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.verify(data["target"], None, tok, data["temperature"], data["uniforms"],
                      nthreads=0, lib=olib, no_draft=True)
    err = o["status"] & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err)
    ok = ~o["boundary"].astype(bool)
    assert np.array_equal(g["accept_len"][ok], o["accept_len"][ok])
    assert np.array_equal(g["out_tokens"][ok], o["out_tokens"][ok])
    assert np.abs(g["p_draft"] - o["p"]).max() <= PROB_TOL
    assert (g["q_draft"] == 1.0).all()
    # a rejected no-draft row never emits the rejected token as its bonus
    for b in range(spec.B):
        n = g["accept_len"][b]
        if n < spec.K:
            assert g["out_tokens"][b, n] != tok[b, n]


def test_ragged_bad_counts_are_flagged(sv, olib):
    """Counts outside [0, K] or past num_draft_tokens flag the row (read nowhere);
    the other rows are unaffected."""
    spec = wl.custom("ragbad", B=5, K=3, V=300, dtype=wl.FP32, temps=(1.0,),
                     seed=wl.SEED_BASE + 9700)
    data = wl.generate(spec)
    kb = np.array([2, 3, 1, 0, 2])
    cu, tgt, dft, tok, uni = pack(data, kb)
    bad = cu.copy()
    bad[2] = bad[1] + 5         # K_2 = 5 > K
    dev_cu = to_dev(bad)
    g = sv.specv_verify_ragged(to_dev(tgt), to_dev(dft), dev_cu, to_dev(tok),
                               to_dev(data["temperature"]), to_dev(uni), spec.K,
                               num_draft_tokens=int(cu[-1]))
    torch.cuda.synchronize()
    st = g["row_status"].cpu().numpy()
    assert st[2] & sv.ROW_BAD_COUNT and g["accept_len"].cpu().numpy()[2] == 0
    assert (g["out_tokens"].cpu().numpy()[2] == -1).all()
    # row 3 now ends before it starts: flagged, not read
    assert st[3] & sv.ROW_BAD_COUNT
    o = oracle.verify_ragged(tgt, dft, cu, tok, data["temperature"], uni, spec.K, lib=olib)
    for b in (0, 1, 4):  # rows whose own counts are intact verify as before
        assert st[b] == o["status"][b]
        assert g["accept_len"].cpu().numpy()[b] == o["accept_len"][b]
        assert (g["out_tokens"].cpu().numpy()[b] == o["out_tokens"][b]).all()
    # a buffer that holds fewer packed rows than the counts need
    g2 = sv.specv_verify_ragged(to_dev(tgt), to_dev(dft), to_dev(cu), to_dev(tok),
                                to_dev(data["temperature"]), to_dev(uni), spec.K,
                                num_draft_tokens=int(cu[2]))
    torch.cuda.synchronize()
    st2 = g2["row_status"].cpu().numpy()
    assert not (st2[:4] & sv.ROW_BAD_COUNT).any() and st2[4] & sv.ROW_BAD_COUNT


def test_ragged_cfg3_sizes(sv, olib):
    """Config 3 sizes (B=64, K=4, V=128256 bf16, mixed temperatures) with
    per-row draft counts 0..4: every row against the oracle."""
    spec = wl.SPECS["cfg3"]
    data = wl.generate(spec)
    kb = np.random.default_rng(3).integers(0, spec.K + 1, spec.B)
    run_pair(sv, olib, data, kb, spec.K, spec.dtype, False, "ragged cfg3")


def test_no_draft_rejections_draw_from_one_chunk(sv, olib):
    """Without draft probabilities a rejection's residual is p_n less the
    rejected token; at B=300, V=50000 fp32 (clusters of 2, chunks shorter
    than a CTA's slice) it is drawn from the one chunk that holds U * R, the
    token's mass taken from its chunk.  Rows whose rejected token holds most
    of the mass (p = 0.8, drafted and rejected by u = 0.95) read the whole
    row instead; at p = 0.3 the chunk's mass loses 0.3 of the row's to the
    correction.  Every row against the oracle."""
    B, K, V = 300, 3, 50000
    spec = wl.custom("ndlocal", B=B, K=K, V=V, dtype=wl.FP32, temps=(0.7, 1.0),
                     sigma_d=(0.3, 2.0), seed=wl.SEED_BASE + 9600)
    data = wl.generate(spec)
    zt = data["target"].copy()
    tok = data["tokens"].copy()
    u = data["uniforms"].copy()
    rng = np.random.default_rng(96)
    dom = rng.choice(B, 60, replace=False)
    for i, b in enumerate(dom):  # a drafted token of p = 0.8 (or 0.3) at position 0, rejected
        x = int(rng.integers(0, V))
        T = float(data["temperature"][b])
        others = np.delete(zt[b, 0].astype(np.float64), x) / T
        lse = others.max() + np.log(np.exp(others - others.max()).sum())
        pt = 0.8 if i % 2 == 0 else 0.3
        zt[b, 0, x] = np.float32(T * (lse + np.log(pt / (1.0 - pt))))
        tok[b, 0] = x
        u[b, 0] = 0.95
    g = sv.specv_verify(to_dev(zt), None, to_dev(tok), to_dev(data["temperature"]), to_dev(u))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.verify(zt, None, tok, data["temperature"], u, nthreads=0, lib=olib, no_draft=True)
    err = o["status"] & oracle.ROW_ERRORS
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err)
    ok = ~o["boundary"].astype(bool)
    assert np.array_equal(g["accept_len"][ok], o["accept_len"][ok])
    assert np.array_equal(g["out_tokens"][ok], o["out_tokens"][ok])
    fb = ok & (err == 0)
    assert np.array_equal(g["row_status"][fb] & oracle.ROW_FALLBACK, o["status"][fb] & oracle.ROW_FALLBACK)
    assert np.abs(g["p_draft"] - o["p"]).max() <= PROB_TOL
    differ = int(((g["accept_len"] != o["accept_len"]) | (g["out_tokens"] != o["out_tokens"]).any(axis=1)).sum())
    assert differ <= max(1, B // 50), differ
    rej = (o["accept_len"][dom] == 0).mean()
    assert rej > 0.9, rej  # the dominant rows do reject at position 0
    for b in range(B):
        n = g["accept_len"][b]
        if n < K:
            assert g["out_tokens"][b, n] != tok[b, n]
    print(f"no-draft local draw: boundary rows {int(o['boundary'].sum())}/{B}, differing {differ}")
