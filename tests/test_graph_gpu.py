"""The library's calls enqueue only kernels on the caller's stream (no
allocation, no synchronisation), so a caller can capture a whole round in a
CUDA graph and replay it: here an SSD round (config 4's shapes, bf16, with
the outcome keys and the hit check) and the Saguaro sampler on 1216 rows
(the warp-per-row decision), each captured once and replayed on new inputs
copied into the captured buffers, against direct calls on the same inputs."""
import numpy as np
import pytest

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


def _dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(torch.bfloat16) if bf16 else t).cuda()


def _same(a, b):
    for k in a:
        x, y = a[k].cpu(), b[k].cpu()
        assert torch.equal(x, y), k


def test_ssd_round_replays_in_a_cuda_graph(sv):
    spec = wl.SPECS["cfg4"]
    runs = [wl.generate(spec), wl.generate(wl.custom("graph", B=spec.B, K=spec.K, V=spec.V, dtype=spec.dtype,
                                                        temps=(0.0, 0.7, 1.0), sigma_d=(0.3, 2.0), F=spec.F,
                                                        ssd=True, seed=wl.SEED_BASE + 34000))]
    bf16 = spec.dtype == wl.BF16
    ins = [_dev(runs[0][k], bf16 and k in ("target", "draft")) for k in ("target", "draft", "tokens",
                                                                       "temperature", "uniforms")]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sv.specv_ssd_round(*ins, spec.F)  # first call outside the capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = sv.specv_ssd_round(*ins, spec.F)
    for d in runs:
        for t, k in zip(ins, ("target", "draft", "tokens", "temperature", "uniforms")):
            t.copy_(_dev(d[k], bf16 and k in ("target", "draft")))
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.clone() for k, v in out.items()}
        ref = sv.specv_ssd_round(*[_dev(d[k], bf16 and k in ("target", "draft"))
                                   for k in ("target", "draft", "tokens", "temperature", "uniforms")], spec.F)
        torch.cuda.synchronize()
        _same(got, ref)


def test_sampler_replays_in_a_cuda_graph(sv):
    rng = np.random.default_rng(17)
    rows, V = 1216, 152064  # 8 rows per SM of 152: the warp-per-row decision
    z = [rng.normal(0, 2.5, (rows, V)).astype(np.float32) for _ in range(2)]
    T = rng.choice([0.0, 0.7, 1.0], rows).astype(np.float32)
    U = [rng.uniform(0, 1, rows).astype(np.float32) for _ in range(2)]
    zd, Td, Ud = _dev(z[0]), _dev(T), _dev(U[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        sv.specv_saguaro_sample(zd, Td, 6, 0.3, Ud)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = sv.specv_saguaro_sample(zd, Td, 6, 0.3, Ud)
    for zi, ui in zip(z, U):
        zd.copy_(_dev(zi))
        Ud.copy_(_dev(ui))
        g.replay()
        torch.cuda.synchronize()
        got = {k: v.clone() for k, v in out.items()}
        ref = sv.specv_saguaro_sample(_dev(zi), Td, 6, 0.3, _dev(ui))
        torch.cuda.synchronize()
        _same(got, ref)
