"""GB300 (sm_103a) speculative-sampling verification and SSD outcome prediction.

Thin Python binding over the C ABI of ``libspecv.so`` (declared in
``include/specv.h``): it marshals torch tensors into pointers, sizes and
strides and passes the current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; there is no Python or CPU fallback, and a
missing library raises.

Entry points (same names as the C ABI):
  specv_verify(target, draft, draft_tokens, temperature, uniforms, ...)
  specv_ssd_round(target, draft, draft_tokens, temperature, uniforms, F, ...)
  specv_predict_outcomes(draft, draft_tokens, F, ...)
  specv_check_hit(keys, accept_len, out_tokens, ...)
"""
from __future__ import annotations

import ctypes
import os

from . import workloads  # noqa: F401  (seeded inputs; no method arithmetic)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecv.so")

SPECV_OK, SPECV_ERR_INVALID_ARG, SPECV_ERR_UNSUPPORTED, SPECV_ERR_CUDA, SPECV_ERR_WORKSPACE = range(5)
SPECV_BF16, SPECV_FP32 = 0, 1
ROW_BAD_TOKEN, ROW_NONFINITE, ROW_BAD_TEMP, ROW_FALLBACK, ROW_DEVICE_TIMEOUT = 1, 2, 4, 8, 16
ROW_BAD_COUNT = 32
SPECV_NO_DRAFT_PROBS = 1
SPECV_MSS_NAIVE = 1

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


class VerifyArgs(ctypes.Structure):
    _fields_ = [("B", _I32), ("K", _I32), ("V", _I32), ("dtype", _I32),
                ("target_logits", _P), ("target_batch_stride", _I64), ("target_row_stride", _I64),
                ("draft_logits", _P), ("draft_batch_stride", _I64), ("draft_row_stride", _I64),
                ("draft_tokens", _P), ("temperature", _P), ("uniforms", _P),
                ("accept_len", _P), ("out_tokens", _P), ("p_draft", _P), ("q_draft", _P),
                ("row_status", _P), ("cu_num_draft_tokens", _P), ("num_draft_tokens", _I32),
                ("flags", _I32)]


class SsdArgs(ctypes.Structure):
    _fields_ = [("verify", VerifyArgs), ("F", _I32), ("keys", _P), ("key_logits", _P),
                ("hit", _P), ("fanout", _P), ("saguaro_F", _I32), ("saguaro_C", ctypes.c_float)]


class SaguaroArgs(ctypes.Structure):
    _fields_ = [("B", _I32), ("V", _I32), ("dtype", _I32), ("logits", _P), ("row_stride", _I64),
                ("temperature", _P), ("F", _I32), ("C", ctypes.c_float), ("uniforms", _P),
                ("tokens", _P), ("q", _P), ("row_status", _P)]


class MssArgs(ctypes.Structure):
    _fields_ = [("B", _I32), ("M", _I32), ("V", _I32), ("dtype", _I32),
                ("target_logits", _P), ("target_row_stride", _I64),
                ("draft_logits", _P), ("draft_row_stride", _I64),
                ("candidates", _P), ("num_candidates", _P), ("temperature", _P), ("uniforms", _P),
                ("flags", _I32), ("accepted", _P), ("out_token", _P), ("accept_prob", _P),
                ("row_status", _P)]


class PredictArgs(ctypes.Structure):
    _fields_ = [("B", _I32), ("K", _I32), ("V", _I32), ("F", _I32), ("dtype", _I32),
                ("draft_logits", _P), ("draft_batch_stride", _I64), ("draft_row_stride", _I64),
                ("draft_tokens", _P), ("keys", _P), ("key_logits", _P), ("row_status", _P),
                ("fanout", _P)]


class SpecvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"specv status {status}: {msg}")
        self.status = status


_lib = None
_lib_path = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libspecv.so (built by __graft_entry__.build()); raise if absent."""
    global _lib, _lib_path
    if _lib is not None and path == _lib_path:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    lib.specv_verify_workspace_bytes.restype = ctypes.c_size_t
    lib.specv_verify_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
    lib.specv_verify.restype = ctypes.c_int
    lib.specv_verify.argtypes = [ctypes.POINTER(VerifyArgs), _P, ctypes.c_size_t, _P]
    lib.specv_verify_noalloc.restype = ctypes.c_int
    lib.specv_verify_noalloc.argtypes = [ctypes.POINTER(VerifyArgs), _P]
    lib.specv_ssd_workspace_bytes.restype = ctypes.c_size_t
    lib.specv_ssd_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32]
    lib.specv_ssd_round.restype = ctypes.c_int
    lib.specv_ssd_round.argtypes = [ctypes.POINTER(SsdArgs), _P, ctypes.c_size_t, _P]
    lib.specv_predict_workspace_bytes.restype = ctypes.c_size_t
    lib.specv_predict_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32, _I32]
    lib.specv_predict_outcomes.restype = ctypes.c_int
    lib.specv_predict_outcomes.argtypes = [ctypes.POINTER(PredictArgs), _P, ctypes.c_size_t, _P]
    lib.specv_saguaro_workspace_bytes.restype = ctypes.c_size_t
    lib.specv_saguaro_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
    lib.specv_saguaro_sample.restype = ctypes.c_int
    lib.specv_saguaro_sample.argtypes = [ctypes.POINTER(SaguaroArgs), _P, ctypes.c_size_t, _P]
    lib.specv_mss_workspace_bytes.restype = ctypes.c_size_t
    lib.specv_mss_workspace_bytes.argtypes = [_I32, _I32, _I32, _I32]
    lib.specv_mss_verify.restype = ctypes.c_int
    lib.specv_mss_verify.argtypes = [ctypes.POINTER(MssArgs), _P, ctypes.c_size_t, _P]
    lib.specv_geometric_fanout.restype = ctypes.c_int
    lib.specv_geometric_fanout.argtypes = [_I32, ctypes.c_double, ctypes.c_double, _I32, _I32,
                                           _P, _P]
    lib.specv_check_hit.restype = ctypes.c_int
    lib.specv_check_hit.argtypes = [_I32, _I32, _I32, _P, _P, _P, _P, _P]
    lib.specv_status_string.restype = ctypes.c_char_p
    lib.specv_status_string.argtypes = [ctypes.c_int]
    lib.specv_last_error.restype = ctypes.c_char_p
    lib.specv_last_error.argtypes = []
    lib.specv_last_launch_count.restype = _I32
    lib.specv_last_launch_count.argtypes = []
    lib.specv_set_split_event.restype = None
    lib.specv_set_split_event.argtypes = [_P]
    _lib, _lib_path = lib, path
    return lib


def _check(rc: int) -> None:
    if rc != SPECV_OK:
        lib = load_library()
        raise SpecvError(rc, lib.specv_last_error().decode() or lib.specv_status_string(rc).decode())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return SPECV_BF16
    if t.dtype == torch.float32:
        return SPECV_FP32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def specv_set_split_event(event) -> None:
    """Record `event` (a torch.cuda.Event, already recorded once so that it
    exists, or None) between the library's two kernels on later calls from
    this thread (measurement hook; see include/specv.h)."""
    handle = None if event is None else ctypes.c_void_p(event.cuda_event)
    load_library().specv_set_split_event(handle)


def last_launch_count() -> int:
    """Kernel launches enqueued by the most recent call on this thread."""
    return int(load_library().specv_last_launch_count())


def _verify_args(target, draft, draft_tokens, temperature, uniforms, draft_rows, accept_len,
                 out_tokens, p_draft, q_draft, row_status):
    import torch
    B, K = draft_tokens.shape
    V = target.shape[-1]
    assert target.dim() == 3 and target.shape[0] == B and target.shape[1] >= K + 1
    assert target.stride(-1) == 1
    if draft is not None:  # None: no draft probabilities (SPECV_NO_DRAFT_PROBS)
        assert draft.dim() == 3 and draft.shape[0] == B and draft.shape[1] >= draft_rows
        assert draft.shape[-1] == V and draft.stride(-1) == 1 and target.dtype == draft.dtype
    assert uniforms.shape == (B, K + 1) and temperature.shape == (B,)
    dev = target.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, K + 1), dtype=torch.int32, device=dev)
    if p_draft is None:
        p_draft = torch.empty((B, K), dtype=torch.float32, device=dev)
    if q_draft is None:
        q_draft = torch.empty((B, K), dtype=torch.float32, device=dev)
    if row_status is None:
        row_status = torch.empty(B, dtype=torch.int32, device=dev)
    args = VerifyArgs(B, K, V, _dtype_code(target),
                      target.data_ptr(), target.stride(0), target.stride(1),
                      None if draft is None else draft.data_ptr(),
                      0 if draft is None else draft.stride(0), 0 if draft is None else draft.stride(1),
                      draft_tokens.data_ptr(), temperature.data_ptr(), uniforms.data_ptr(),
                      accept_len.data_ptr(), out_tokens.data_ptr(),
                      p_draft.data_ptr(), q_draft.data_ptr(), row_status.data_ptr(),
                      None, 0, SPECV_NO_DRAFT_PROBS if draft is None else 0)
    outs = dict(accept_len=accept_len, out_tokens=out_tokens, p_draft=p_draft,
                q_draft=q_draft, row_status=row_status)
    return args, outs


def specv_verify(target, draft, draft_tokens, temperature, uniforms, *, accept_len=None,
                 out_tokens=None, p_draft=None, q_draft=None, row_status=None,
                 workspace=None, stream=None) -> dict:
    """Verify B batch rows on the GPU (see include/specv.h, specv_verify).

    target [B, >=K+1, V], draft [B, >=K, V] (bf16 or fp32, CUDA, last dim
    contiguous) or None for drafts without probabilities (SPECV_NO_DRAFT_PROBS);
    draft_tokens int32 [B, K]; temperature fp32 [B]; uniforms fp32 [B, K+1].
    Outputs are allocated when not given.  Returns a dict with accept_len,
    out_tokens, p_draft, q_draft, row_status.
    """
    import torch
    lib = load_library()
    B, K = draft_tokens.shape
    args, outs = _verify_args(target, draft, draft_tokens, temperature, uniforms, K, accept_len,
                              out_tokens, p_draft, q_draft, row_status)
    need = lib.specv_verify_workspace_bytes(B, K, target.shape[-1], args.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=target.device)
    _check(lib.specv_verify(ctypes.byref(args), _ptr(workspace), workspace.numel(), _stream(stream)))
    return outs


def specv_verify_ragged(target, draft, cu_num_draft_tokens, draft_tokens, temperature, uniforms,
                        K: int, *, num_draft_tokens: int | None = None, accept_len=None,
                        out_tokens=None, p_draft=None, q_draft=None, row_status=None,
                        workspace=None, stream=None) -> dict:
    """Verification with a per-row draft count (see include/specv.h,
    cu_num_draft_tokens): rows packed along one axis.

    target [N + B, V] (K_b + 1 rows per batch row, in order), draft [N, V] or
    None (no draft probabilities), cu_num_draft_tokens int32 [B] (inclusive
    prefix sums, on the device), draft_tokens int32 [N], temperature fp32 [B],
    uniforms fp32 [N + B]; K = the largest count allowed.  N defaults to
    draft_tokens.numel().  Returns accept_len [B], out_tokens [B, K+1],
    p_draft / q_draft [N], row_status [B].
    """
    import torch
    lib = load_library()
    B = cu_num_draft_tokens.shape[0]
    N = draft_tokens.numel() if num_draft_tokens is None else int(num_draft_tokens)
    V = target.shape[-1]
    assert target.dim() == 2 and target.stride(-1) == 1 and target.shape[0] >= N + B
    if draft is not None:
        assert draft.dim() == 2 and draft.stride(-1) == 1 and draft.shape[0] >= N
        assert draft.shape[-1] == V and draft.dtype == target.dtype
    assert draft_tokens.numel() >= N and uniforms.numel() >= N + B and temperature.shape == (B,)
    dev = target.device
    i32 = dict(dtype=torch.int32, device=dev)
    accept_len = torch.empty(B, **i32) if accept_len is None else accept_len
    out_tokens = torch.empty((B, K + 1), **i32) if out_tokens is None else out_tokens
    p_draft = torch.zeros(max(N, 1), dtype=torch.float32, device=dev) if p_draft is None else p_draft
    q_draft = torch.zeros(max(N, 1), dtype=torch.float32, device=dev) if q_draft is None else q_draft
    row_status = torch.empty(B, **i32) if row_status is None else row_status
    args = VerifyArgs(B, K, V, _dtype_code(target), target.data_ptr(), 0, target.stride(0),
                      None if draft is None else draft.data_ptr(), 0,
                      0 if draft is None else draft.stride(0),
                      draft_tokens.data_ptr(), temperature.data_ptr(), uniforms.data_ptr(),
                      accept_len.data_ptr(), out_tokens.data_ptr(), p_draft.data_ptr(),
                      q_draft.data_ptr(), row_status.data_ptr(), cu_num_draft_tokens.data_ptr(),
                      N, SPECV_NO_DRAFT_PROBS if draft is None else 0)
    need = lib.specv_verify_workspace_bytes(B, K, V, args.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check(lib.specv_verify(ctypes.byref(args), _ptr(workspace), workspace.numel(), _stream(stream)))
    return dict(accept_len=accept_len, out_tokens=out_tokens, p_draft=p_draft, q_draft=q_draft,
                row_status=row_status)


def specv_verify_noalloc(target, draft, draft_tokens, temperature, uniforms, *, accept_len=None,
                         out_tokens=None, p_draft=None, q_draft=None, row_status=None,
                         stream=None) -> dict:
    """specv_verify without a workspace: the library's built-in scratch is used
    (for callers that cannot allocate device memory where they call it; see
    include/specv.h).  Calls that may overlap on the GPU must be serialised."""
    lib = load_library()
    B, K = draft_tokens.shape
    args, outs = _verify_args(target, draft, draft_tokens, temperature, uniforms, K, accept_len,
                              out_tokens, p_draft, q_draft, row_status)
    _check(lib.specv_verify_noalloc(ctypes.byref(args), _stream(stream)))
    return outs


def _fanout_arg(fanout, K: int):
    """A host int32 array [K+1] kept alive by the caller, or None."""
    if fanout is None:
        return None, None
    vals = [int(x) for x in fanout]
    assert len(vals) == K + 1, "fanout needs K+1 entries"
    arr = (_I32 * (K + 1))(*vals)
    return arr, ctypes.cast(arr, _P)


def specv_ssd_round(target, draft, draft_tokens, temperature, uniforms, F: int, *,
                    accept_len=None, out_tokens=None, p_draft=None, q_draft=None,
                    row_status=None, keys=None, key_logits=None, hit=None, workspace=None,
                    fanout=None, saguaro=None, stream=None) -> dict:
    """One fused SSD round (see include/specv.h, specv_ssd_round): verification,
    top-F outcome keys at every lookahead and the hit flag, in one pass.

    draft must hold K+1 rows per batch row.  Returns the specv_verify outputs
    plus keys int32 [B, K+1, F], key_logits fp32 [B, K+1, F], hit uint8 [B].
    fanout (optional, K+1 ints in [0, F], e.g. from specv_geometric_fanout)
    keeps only the first fanout[k] keys at lookahead k.  saguaro=(F_s, C): the
    drafts were sampled from sigma_{F_s,C} (specv_saguaro_sample), so the
    accept test and the residual use it as q.
    """
    import torch
    lib = load_library()
    B, K = draft_tokens.shape
    args, outs = _verify_args(target, draft, draft_tokens, temperature, uniforms, K + 1,
                              accept_len, out_tokens, p_draft, q_draft, row_status)
    dev = target.device
    if keys is None:
        keys = torch.empty((B, K + 1, F), dtype=torch.int32, device=dev)
    if key_logits is None:
        key_logits = torch.empty((B, K + 1, F), dtype=torch.float32, device=dev)
    if hit is None:
        hit = torch.empty(B, dtype=torch.uint8, device=dev)
    need = lib.specv_ssd_workspace_bytes(B, K, target.shape[-1], F, args.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    fan_keep, fan_ptr = _fanout_arg(fanout, K)
    sg_F, sg_C = saguaro if saguaro else (0, 1.0)
    sargs = SsdArgs(args, F, keys.data_ptr(), key_logits.data_ptr(), hit.data_ptr(), fan_ptr,
                    int(sg_F), float(sg_C))
    _check(lib.specv_ssd_round(ctypes.byref(sargs), _ptr(workspace), workspace.numel(),
                               _stream(stream)))
    outs.update(keys=keys, key_logits=key_logits, hit=hit)
    return outs


def specv_predict_outcomes(draft, draft_tokens, F: int, *, keys=None, key_logits=None,
                           row_status=None, workspace=None, fanout=None, stream=None) -> dict:
    """Top-F outcome keys per lookahead (see include/specv.h).

    draft [B, >=K+1, V] (bf16 or fp32, CUDA); draft_tokens int32 [B, K].
    Returns keys int32 [B, K+1, F], key_logits fp32, row_status int32 [B].
    """
    import torch
    lib = load_library()
    B, K = draft_tokens.shape
    V = draft.shape[-1]
    assert draft.dim() == 3 and draft.shape[0] == B and draft.shape[1] >= K + 1
    assert draft.stride(-1) == 1
    dev = draft.device
    if keys is None:
        keys = torch.empty((B, K + 1, F), dtype=torch.int32, device=dev)
    if key_logits is None:
        key_logits = torch.empty((B, K + 1, F), dtype=torch.float32, device=dev)
    if row_status is None:
        row_status = torch.empty(B, dtype=torch.int32, device=dev)
    code = _dtype_code(draft)
    need = lib.specv_predict_workspace_bytes(B, K, V, F, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    fan_keep, fan_ptr = _fanout_arg(fanout, K)
    args = PredictArgs(B, K, V, F, code, draft.data_ptr(), draft.stride(0), draft.stride(1),
                       draft_tokens.data_ptr(), keys.data_ptr(), key_logits.data_ptr(),
                       row_status.data_ptr(), fan_ptr)
    _check(lib.specv_predict_outcomes(ctypes.byref(args), _ptr(workspace), workspace.numel(),
                                      _stream(stream)))
    return dict(keys=keys, key_logits=key_logits, row_status=row_status)


def specv_saguaro_sample(logits, temperature, F: int, C: float, uniforms, *, tokens=None, q=None,
                         row_status=None, workspace=None, stream=None) -> dict:
    """Draft-side Saguaro sampling (see include/specv.h): one token per row of
    logits [B, V] (bf16 or fp32, CUDA) from sigma_{F,C}(z/T) by inverse CDF of
    uniforms [B].  Returns tokens int32 [B], q fp32 [B], row_status int32 [B]."""
    import torch
    lib = load_library()
    assert logits.dim() == 2 and logits.stride(-1) == 1
    B, V = logits.shape
    dev = logits.device
    tokens = torch.empty(B, dtype=torch.int32, device=dev) if tokens is None else tokens
    q = torch.empty(B, dtype=torch.float32, device=dev) if q is None else q
    row_status = torch.empty(B, dtype=torch.int32, device=dev) if row_status is None else row_status
    code = _dtype_code(logits)
    need = lib.specv_saguaro_workspace_bytes(B, V, int(F), code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    args = SaguaroArgs(B, V, code, logits.data_ptr(), logits.stride(0), temperature.data_ptr(),
                       int(F), float(C), uniforms.data_ptr(), tokens.data_ptr(), q.data_ptr(),
                       row_status.data_ptr())
    _check(lib.specv_saguaro_sample(ctypes.byref(args), _ptr(workspace), workspace.numel(),
                                    _stream(stream)))
    return dict(tokens=tokens, q=q, row_status=row_status)


def specv_mss_verify(target, draft, candidates, temperature, uniforms, *, num_candidates=None,
                     naive: bool = False, accepted=None, out_token=None, accept_prob=None,
                     row_status=None, workspace=None, stream=None) -> dict:
    """Multi-step speculative sampling at B token-tree nodes (see
    include/specv.h): target, draft [B, V] (bf16 or fp32, CUDA; rows may be
    strided), candidates int32 [B, M], num_candidates int32 [B] or None,
    temperature fp32 [B], uniforms fp32 [B, M+1].  naive=True: naive sampling.
    Returns accepted int32 [B], out_token int32 [B], accept_prob fp32 [B, M],
    row_status int32 [B]."""
    import torch
    lib = load_library()
    assert target.dim() == 2 and draft.dim() == 2 and target.shape == draft.shape
    assert target.stride(-1) == 1 and draft.stride(-1) == 1 and target.dtype == draft.dtype
    B, V = target.shape
    M = candidates.shape[1]
    dev = target.device
    i32 = dict(dtype=torch.int32, device=dev)
    accepted = torch.empty(B, **i32) if accepted is None else accepted
    out_token = torch.empty(B, **i32) if out_token is None else out_token
    accept_prob = (torch.empty((B, M), dtype=torch.float32, device=dev)
                   if accept_prob is None else accept_prob)
    row_status = torch.empty(B, **i32) if row_status is None else row_status
    code = _dtype_code(target)
    need = lib.specv_mss_workspace_bytes(B, M, V, code)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    args = MssArgs(B, M, V, code, target.data_ptr(), target.stride(0), draft.data_ptr(),
                   draft.stride(0), candidates.data_ptr(),
                   num_candidates.data_ptr() if num_candidates is not None else None,
                   temperature.data_ptr(), uniforms.data_ptr(),
                   SPECV_MSS_NAIVE if naive else 0, accepted.data_ptr(), out_token.data_ptr(),
                   accept_prob.data_ptr(), row_status.data_ptr())
    _check(lib.specv_mss_verify(ctypes.byref(args), _ptr(workspace), workspace.numel(),
                                _stream(stream)))
    return dict(accepted=accepted, out_token=out_token, accept_prob=accept_prob,
                row_status=row_status)


def specv_geometric_fanout(K: int, a: float, r: float, budget: int, max_f: int = 32) -> tuple:
    """Theorem 12 fan-out (see include/specv.h): (integer F_k list, real F_k list)."""
    lib = load_library()
    fk = (_I32 * (K + 1))()
    real = (ctypes.c_double * (K + 1))()
    _check(lib.specv_geometric_fanout(int(K), float(a), float(r), int(budget), int(max_f),
                                      ctypes.cast(fk, _P), ctypes.cast(real, _P)))
    return list(fk), list(real)


def specv_check_hit(keys, accept_len, out_tokens, *, hit=None, stream=None):
    """hit[b] = out_tokens[b, n_b] in keys[b, n_b, :] (uint8 [B])."""
    import torch
    lib = load_library()
    B, K1, F = keys.shape
    assert accept_len.shape == (B,) and out_tokens.shape == (B, K1)
    if hit is None:
        hit = torch.empty(B, dtype=torch.uint8, device=keys.device)
    _check(lib.specv_check_hit(B, K1 - 1, F, _ptr(keys), _ptr(accept_len), _ptr(out_tokens),
                               _ptr(hit), _stream(stream)))
    return hit
