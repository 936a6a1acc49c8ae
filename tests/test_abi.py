"""C-ABI library: loads, exports every declared symbol, validates on the host.

No test here launches a kernel: every call is rejected by host-side argument
checks before any CUDA call, so these run without a GPU.
"""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_50_gb300 as sv
from speculative_decoding_verification_50_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return sv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(specv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_entry_points():
    names = declared_functions()
    for n in ("specv_verify", "specv_predict_outcomes", "specv_check_hit"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(5):
        assert lib.specv_status_string(code)
    assert lib.specv_status_string(99) == b"unknown status"


def _args(**kw):
    a = sv.VerifyArgs()
    a.B, a.K, a.V, a.dtype = 2, 3, 100, sv.SPECV_FP32
    for f in ("target_logits", "draft_logits", "draft_tokens", "temperature", "uniforms",
              "accept_len", "out_tokens"):
        setattr(a, f, 0x10000)
    a.target_batch_stride, a.target_row_stride = 400, 100
    a.draft_batch_stride, a.draft_row_stride = 300, 100
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,code", [
    (dict(K=0), sv.SPECV_ERR_INVALID_ARG),
    (dict(K=33), sv.SPECV_ERR_INVALID_ARG),
    (dict(V=0), sv.SPECV_ERR_INVALID_ARG),
    (dict(B=-1), sv.SPECV_ERR_INVALID_ARG),
    (dict(dtype=7), sv.SPECV_ERR_INVALID_ARG),
    (dict(target_logits=None), sv.SPECV_ERR_INVALID_ARG),
    (dict(uniforms=None), sv.SPECV_ERR_INVALID_ARG),
    (dict(target_row_stride=99), sv.SPECV_ERR_INVALID_ARG),
    (dict(target_batch_stride=399), sv.SPECV_ERR_INVALID_ARG),
    (dict(draft_batch_stride=299), sv.SPECV_ERR_INVALID_ARG),
    (dict(draft_tokens=0x10002), sv.SPECV_ERR_INVALID_ARG),
])
def test_verify_rejects_bad_arguments(lib, kw, code):
    a = _args(**kw)
    rc = lib.specv_verify(ctypes.byref(a), ctypes.c_void_p(0x100000), 1 << 20, None)
    assert rc == code
    assert lib.specv_last_error()


def test_verify_null_args(lib):
    assert lib.specv_verify(None, None, 0, None) == sv.SPECV_ERR_INVALID_ARG


def test_verify_workspace_checks(lib):
    a = _args()
    need = lib.specv_verify_workspace_bytes(2, 3, 100, sv.SPECV_FP32)
    assert need >= 2 * 4 * 48 and need % 256 == 0
    assert lib.specv_verify(ctypes.byref(a), None, need, None) == sv.SPECV_ERR_WORKSPACE
    assert lib.specv_verify(ctypes.byref(a), ctypes.c_void_p(0x100000), need - 1, None) == sv.SPECV_ERR_WORKSPACE
    assert lib.specv_verify(ctypes.byref(a), ctypes.c_void_p(0x100010), need, None) == sv.SPECV_ERR_WORKSPACE


def test_empty_batch_is_a_no_op(lib):
    a = _args(B=0, target_logits=None)
    assert lib.specv_verify(ctypes.byref(a), None, 0, None) == sv.SPECV_OK
    assert lib.specv_last_launch_count() == 0
    assert lib.specv_verify_workspace_bytes(0, 3, 100, 1) == 0


def test_predict_rejects_bad_arguments(lib):
    p = sv.PredictArgs(2, 3, 100, 6, sv.SPECV_BF16, 0x10000, 400, 100, 0x10000, 0x10000, 0, 0)
    for field, val in (("F", 0), ("F", 33), ("K", 0), ("V", 0), ("dtype", 5),
                       ("keys", None), ("draft_batch_stride", 399), ("draft_row_stride", 50)):
        q = sv.PredictArgs.from_buffer_copy(p)
        setattr(q, field, val)
        assert lib.specv_predict_outcomes(ctypes.byref(q), None, 0, None) == sv.SPECV_ERR_INVALID_ARG, field
    q = sv.PredictArgs.from_buffer_copy(p)
    q.row_status = 0x10000
    assert lib.specv_predict_outcomes(ctypes.byref(q), None, 0, None) == sv.SPECV_ERR_WORKSPACE


def test_check_hit_rejects_bad_arguments(lib):
    P = ctypes.c_void_p(0x10000)
    assert lib.specv_check_hit(2, 0, 6, P, P, P, P, None) == sv.SPECV_ERR_INVALID_ARG
    assert lib.specv_check_hit(2, 3, 0, P, P, P, P, None) == sv.SPECV_ERR_INVALID_ARG
    assert lib.specv_check_hit(2, 3, 6, None, P, P, P, None) == sv.SPECV_ERR_INVALID_ARG
    assert lib.specv_check_hit(0, 3, 6, None, None, None, None, None) == sv.SPECV_OK


def test_product_path_never_touches_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_verification_50_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "specv_oracle" not in text, f


def test_struct_layouts_match_the_header(tmp_path):
    """The binding's ctypes structs have the C header's sizes and offsets."""
    import subprocess
    src = tmp_path / "layout.c"
    src.write_text(r'''
#include <stddef.h>
#include <stdio.h>
#include "specv.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n",
         sizeof(specv_verify_args),
         offsetof(specv_verify_args, target_logits), offsetof(specv_verify_args, draft_tokens),
         offsetof(specv_verify_args, row_status), sizeof(specv_ssd_args),
         offsetof(specv_ssd_args, keys), sizeof(specv_predict_args),
         offsetof(specv_predict_args, row_status), offsetof(specv_ssd_args, fanout),
         offsetof(specv_predict_args, fanout), offsetof(specv_ssd_args, saguaro_C),
         sizeof(specv_saguaro_args), offsetof(specv_saguaro_args, C),
         offsetof(specv_saguaro_args, row_status), sizeof(specv_mss_args),
         offsetof(specv_mss_args, candidates), offsetof(specv_mss_args, flags),
         offsetof(specv_mss_args, row_status));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    want = [ctypes.sizeof(sv.VerifyArgs), sv.VerifyArgs.target_logits.offset,
            sv.VerifyArgs.draft_tokens.offset, sv.VerifyArgs.row_status.offset,
            ctypes.sizeof(sv.SsdArgs), sv.SsdArgs.keys.offset, ctypes.sizeof(sv.PredictArgs),
            sv.PredictArgs.row_status.offset, sv.SsdArgs.fanout.offset,
            sv.PredictArgs.fanout.offset, sv.SsdArgs.saguaro_C.offset,
            ctypes.sizeof(sv.SaguaroArgs), sv.SaguaroArgs.C.offset,
            sv.SaguaroArgs.row_status.offset, ctypes.sizeof(sv.MssArgs),
            sv.MssArgs.candidates.offset, sv.MssArgs.flags.offset, sv.MssArgs.row_status.offset]
    assert got == want


def test_ssd_round_rejects_bad_arguments(lib):
    a = _args()
    s = sv.SsdArgs(a, 6, 0x10000, 0, 0x10000)
    for field, val in (("F", 0), ("F", 33), ("keys", None), ("hit", None)):
        q = sv.SsdArgs.from_buffer_copy(s)
        setattr(q, field, val)
        assert lib.specv_ssd_round(ctypes.byref(q), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG, field
    q = sv.SsdArgs.from_buffer_copy(s)
    q.verify.draft_batch_stride = 300  # needs K+1 = 4 draft rows of stride 100
    assert lib.specv_ssd_round(ctypes.byref(q), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG


def test_unsupported_vocabulary_size(lib):
    V = 2_000_000_000  # per-CTA segment table of the decision kernel would not fit
    a = _args(V=V, target_row_stride=V, draft_row_stride=V,
              target_batch_stride=4 * V, draft_batch_stride=3 * V)
    assert lib.specv_verify(ctypes.byref(a), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_UNSUPPORTED


def test_ssd_round_and_predict_reject_bad_fanout(lib):
    a = _args()
    for bad in ([1, 2, 7, 1], [1, -1, 0, 0]):  # F = 6: entries must lie in [0, 6]
        arr = (ctypes.c_int32 * 4)(*bad)
        s = sv.SsdArgs(a, 6, 0x10000, 0, 0x10000, ctypes.cast(arr, ctypes.c_void_p))
        assert lib.specv_ssd_round(ctypes.byref(s), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG
        p = sv.PredictArgs(2, 3, 100, 6, sv.SPECV_BF16, 0x10000, 400, 100, 0x10000, 0x10000, 0, 0,
                           ctypes.cast(arr, ctypes.c_void_p))
        assert lib.specv_predict_outcomes(ctypes.byref(p), None, 0, None) == sv.SPECV_ERR_INVALID_ARG


def test_geometric_fanout_matches_the_oracle(lib):
    """Host-only entry point: the library's Theorem 12 fan-out equals the
    oracle's, real values to 1e-12 and integers exactly (up to exact ties of
    fractional parts, where either choice is the same reading)."""
    import numpy as np
    import oracle
    olib = oracle.load()
    rng = np.random.default_rng(21)
    for _ in range(300):
        K = int(rng.integers(1, 33))
        a = float(rng.uniform(0.01, 0.99))
        r = float(rng.uniform(0.1, 4.0))
        budget = int(rng.integers(0, 400))
        max_f = int(rng.integers(0, 33))
        fk, real = sv.specv_geometric_fanout(K, a, r, budget, max_f)
        ofk, oreal = oracle.geometric_fanout(K, a, r, budget, max_f, lib=olib)
        np.testing.assert_allclose(real, oreal, rtol=1e-12, atol=1e-12)
        if list(fk) != list(ofk):
            frac = np.sort(oreal - np.floor(oreal))
            assert np.min(np.diff(frac)) < 1e-9, (K, a, r, budget, fk, ofk)
    fk, real = sv.specv_geometric_fanout(4, 0.7, 1.0, 24)
    assert fk == [6, 5, 4, 4, 5] and abs(sum(real) - 24) < 1e-12


def test_geometric_fanout_rejects_bad_arguments(lib):
    out = (ctypes.c_int32 * 40)()
    ptr = ctypes.cast(out, ctypes.c_void_p)
    for args in ((0, 0.5, 1.0, 10, 8), (33, 0.5, 1.0, 10, 8), (4, 0.0, 1.0, 10, 8),
                 (4, 1.0, 1.0, 10, 8), (4, 0.5, 0.0, 10, 8), (4, 0.5, 1.0, -1, 8),
                 (4, 0.5, 1.0, 10, 33)):
        assert lib.specv_geometric_fanout(*args, ptr, None) == sv.SPECV_ERR_INVALID_ARG, args
    assert lib.specv_geometric_fanout(4, 0.5, 1.0, 10, 8, None, None) == sv.SPECV_ERR_INVALID_ARG
    assert lib.specv_geometric_fanout(4, 0.5, 1.0, 10, 8, ptr, None) == sv.SPECV_OK


def test_verify_flags_and_packed_rows_are_checked(lib):
    # unknown flag bits
    assert lib.specv_verify(ctypes.byref(_args(flags=2)), ctypes.c_void_p(0x100000), 1 << 20,
                            None) == sv.SPECV_ERR_INVALID_ARG
    # SPECV_NO_DRAFT_PROBS needs draft_logits NULL, and NULL needs the flag
    assert lib.specv_verify(ctypes.byref(_args(flags=sv.SPECV_NO_DRAFT_PROBS)),
                            ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG
    assert lib.specv_verify(ctypes.byref(_args(draft_logits=None)), ctypes.c_void_p(0x100000),
                            1 << 20, None) == sv.SPECV_ERR_INVALID_ARG
    # packed rows: a negative row count, a misaligned count array
    assert lib.specv_verify(ctypes.byref(_args(cu_num_draft_tokens=0x10000, num_draft_tokens=-1)),
                            ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG
    assert lib.specv_verify(ctypes.byref(_args(cu_num_draft_tokens=0x10002, num_draft_tokens=4)),
                            ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG
    # packed rows ignore the batch strides (0 is fine); the workspace check comes next
    a = _args(cu_num_draft_tokens=0x10000, num_draft_tokens=4, target_batch_stride=0,
              draft_batch_stride=0)
    assert lib.specv_verify(ctypes.byref(a), None, 0, None) == sv.SPECV_ERR_WORKSPACE


def test_ssd_round_refuses_verification_only_modes(lib):
    a = _args(draft_batch_stride=400)
    s = sv.SsdArgs(a, 6, 0x10000, 0, 0x10000)
    s.verify.flags = sv.SPECV_NO_DRAFT_PROBS
    s.verify.draft_logits = None
    assert lib.specv_ssd_round(ctypes.byref(s), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG
    s = sv.SsdArgs(a, 6, 0x10000, 0, 0x10000)
    s.verify.cu_num_draft_tokens = 0x10000
    s.verify.num_draft_tokens = 4
    assert lib.specv_ssd_round(ctypes.byref(s), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_UNSUPPORTED


def test_saguaro_arguments_are_checked(lib):
    P = 0x10000
    base = sv.SaguaroArgs(4, 100, sv.SPECV_FP32, P, 100, P, 6, 0.25, P, P, 0, 0)
    for field, val in (("F", -1), ("F", 33), ("C", 1.5), ("C", -0.1), ("V", 0), ("dtype", 9),
                       ("logits", None), ("tokens", None), ("row_stride", 99), ("logits", 0x10002)):
        a = sv.SaguaroArgs.from_buffer_copy(base)
        setattr(a, field, val)
        assert lib.specv_saguaro_sample(ctypes.byref(a), ctypes.c_void_p(0x100000), 1 << 20,
                                        None) == sv.SPECV_ERR_INVALID_ARG, field
    a = sv.SaguaroArgs.from_buffer_copy(base)
    assert lib.specv_saguaro_sample(ctypes.byref(a), None, 0, None) == sv.SPECV_ERR_WORKSPACE
    assert lib.specv_saguaro_workspace_bytes(4, 100, 6, sv.SPECV_FP32) > 0
    a.B = 0
    assert lib.specv_saguaro_sample(ctypes.byref(a), None, 0, None) == sv.SPECV_OK
    # an SSD round whose Saguaro F exceeds its key width, or C outside [0, 1]
    s = sv.SsdArgs(_args(draft_batch_stride=400), 6, 0x10000, 0, 0x10000, None, 7, 0.5)
    assert lib.specv_ssd_round(ctypes.byref(s), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG
    s = sv.SsdArgs(_args(draft_batch_stride=400), 6, 0x10000, 0, 0x10000, None, 3, 1.5)
    assert lib.specv_ssd_round(ctypes.byref(s), ctypes.c_void_p(0x100000), 1 << 20, None) == sv.SPECV_ERR_INVALID_ARG


def test_mss_arguments_are_checked(lib):
    P = 0x10000
    base = sv.MssArgs(4, 3, 100, sv.SPECV_FP32, P, 100, P, 100, P, None, P, P, 0, P, P, None, None)
    for field, val in (("M", 0), ("M", 33), ("V", 0), ("dtype", 9), ("flags", 2),
                       ("target_logits", None), ("draft_logits", None), ("candidates", None),
                       ("uniforms", None), ("accepted", None), ("out_token", None),
                       ("target_row_stride", 99), ("draft_row_stride", 99),
                       ("candidates", 0x10002), ("num_candidates", 0x10002)):
        a = sv.MssArgs.from_buffer_copy(base)
        setattr(a, field, val)
        assert lib.specv_mss_verify(ctypes.byref(a), ctypes.c_void_p(0x100000), 1 << 20,
                                    None) == sv.SPECV_ERR_INVALID_ARG, field
    a = sv.MssArgs.from_buffer_copy(base)
    assert lib.specv_mss_verify(ctypes.byref(a), None, 0, None) == sv.SPECV_ERR_WORKSPACE
    assert lib.specv_mss_workspace_bytes(4, 3, 100, sv.SPECV_FP32) > 0
    assert lib.specv_mss_workspace_bytes(4, 0, 100, sv.SPECV_FP32) == 0
    a.B = 0
    assert lib.specv_mss_verify(ctypes.byref(a), None, 0, None) == sv.SPECV_OK
    a.flags = sv.SPECV_MSS_NAIVE
    assert lib.specv_mss_verify(ctypes.byref(a), None, 0, None) == sv.SPECV_OK
    assert lib.specv_mss_verify(None, None, 0, None) == sv.SPECV_ERR_INVALID_ARG


def test_missing_library_fails_loudly():
    """Without libspecv.so the product raises: there is no CPU fallback."""
    import subprocess
    import sys
    code = ("import torch, speculative_decoding_verification_50_gb300 as sv\n"
            "sv.load_library.__defaults__ = ('/nonexistent/libspecv.so',)\n"
            "z = torch.zeros(1, 2, 8); t = torch.zeros(1, 1, dtype=torch.int32)\n"
            "sv.specv_verify(z, z[:, :1], t, torch.ones(1), torch.zeros(1, 2))\n")
    p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert p.returncode != 0
    assert "libspecv.so is missing" in p.stderr, p.stderr[-1000:]
