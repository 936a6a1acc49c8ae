"""specv_verify_noalloc: verification with the library's built-in scratch.

Some callers cannot allocate device memory where they call the library (a
server that reserved all free GPU memory for its KV cache, or a host language
without a CUDA allocator binding).  For them the library offers one entry point
that takes no workspace and uses a fixed scratch array in device memory.  These
tests call it through the C ABI twice in a row, on two different workloads, and
check each result against the workspace entry point specv_verify on the same
inputs.  The file sorts last so that a run stopping at its first failure has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest

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


def _dev(data):
    spec = data["spec"]

    def logits(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return (t.view(torch.bfloat16) if spec.dtype == wl.BF16 else t).cuda()

    return (logits(data["target"]), logits(data["draft"]), torch.from_numpy(data["tokens"]).cuda(),
            torch.from_numpy(data["temperature"]).cuda(), torch.from_numpy(data["uniforms"]).cuda())


def _numpy(out):
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(sv):
    cases = [
        wl.generate(wl.SPECS["cfg3"]),  # bf16, mixed greedy / temperature rows
        wl.generate(wl.SPECS["cfg5"]),  # fp32, B=256, K=8, V=152064: the size the header cites
    ]
    for data in cases:
        args = _dev(data)
        ref = _numpy(sv.specv_verify(*args))
        got = _numpy(sv.specv_verify_noalloc(*args))  # consecutive scratch reuse
        assert sv.last_launch_count() == 2
        for k in ("accept_len", "out_tokens", "row_status"):
            assert np.array_equal(got[k], ref[k]), k
        for k in ("p_draft", "q_draft"):
            assert np.abs(got[k] - ref[k]).max() <= PROB_TOL, k


def test_noalloc_covers_config5_at_full_size(sv):
    """The header's size claim: B=256, K=8, V=152064 fp32 fits the scratch."""
    lib = sv.load_library()
    need = lib.specv_verify_workspace_bytes(256, 8, 152064, sv.SPECV_FP32)
    assert 0 < need <= (8 << 20), need


def test_noalloc_rejects_calls_beyond_its_scratch(sv):
    lib = sv.load_library()
    a = sv.VerifyArgs()
    a.B, a.K, a.V, a.dtype = 4096, 32, 1_000_000, sv.SPECV_FP32
    for f in ("target_logits", "draft_logits", "draft_tokens", "temperature", "uniforms",
              "accept_len", "out_tokens"):
        setattr(a, f, 0x10000)
    a.target_row_stride = a.draft_row_stride = a.V
    a.target_batch_stride, a.draft_batch_stride = 33 * a.V, 32 * a.V
    assert lib.specv_verify_workspace_bytes(a.B, a.K, a.V, a.dtype) > (8 << 20)
    assert lib.specv_verify_noalloc(ctypes.byref(a), None) == sv.SPECV_ERR_UNSUPPORTED
    assert b"scratch" in lib.specv_last_error()
