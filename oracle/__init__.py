"""CPU oracle for speculative-sampling verification and SSD outcome prediction.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import or run anything in this package; the
product library never does, and it shares no code with the CUDA path.

The arithmetic lives in ``specv_oracle.c`` (plain fp64 loops, OpenMP over
batch rows); this module compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "specv_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libspecv_oracle.so")

BF16, FP32 = 0, 1
ROW_BAD_TOKEN, ROW_NONFINITE, ROW_BAD_TEMP, ROW_FALLBACK = 1, 2, 4, 8
ROW_BAD_COUNT = 32  # a per-row draft count outside [0, Kmax]
ROW_ERRORS = ROW_BAD_TOKEN | ROW_NONFINITE | ROW_BAD_TEMP | ROW_BAD_COUNT


_P = ctypes.c_void_p
_I = ctypes.c_int
_L = ctypes.c_int64


def build(src: str = SRC, out: str = LIB_PATH, openmp: bool = True,
          force: bool = False) -> str:
    """Compile the oracle into a shared library and return its path."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
            "-fPIC", "-shared", src, "-o", out, "-lm"]
    if openmp:
        try:
            subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                           capture_output=True)
            return out
        except subprocess.CalledProcessError:
            pass
    subprocess.run(base, check=True, capture_output=True)
    return out


_LIBS: dict = {}


def load(path: str | None = None) -> ctypes.CDLL:
    path = path or build()
    if path in _LIBS:
        return _LIBS[path]
    lib = ctypes.CDLL(path)
    lib.specv_oracle_verify.restype = _I
    lib.specv_oracle_verify.argtypes = [_I, _I, _I, _I, _P, _L, _L, _P, _L, _L,
                                        _P, _P, _P, _I, _I, ctypes.c_double,
                                        _P, _P, _P, _P, _P, _P, _P, _I]
    lib.specv_oracle_saguaro_probs.restype = _I
    lib.specv_oracle_saguaro_probs.argtypes = [_I, _I, _P, ctypes.c_double, _I, ctypes.c_double, _P]
    lib.specv_oracle_saguaro_sample.restype = _I
    lib.specv_oracle_saguaro_sample.argtypes = [_I, _I, _I, _P, _L, _P, _I, ctypes.c_double, _P,
                                                _P, _P, _P]
    lib.specv_oracle_verify_ragged.restype = _I
    lib.specv_oracle_verify_ragged.argtypes = [_I, _I, _I, _I, _P, _L, _P, _L, _P, _P, _P, _P,
                                               _I, _P, _P, _P, _P, _P, _P, _P, _I]
    lib.specv_oracle_predict.restype = _I
    lib.specv_oracle_predict.argtypes = [_I, _I, _I, _I, _I, _P, _L, _L, _P, _P, _P,
                                         _P, _P, _I]
    lib.specv_oracle_geometric_fanout.restype = _I
    lib.specv_oracle_geometric_fanout.argtypes = [_I, ctypes.c_double, ctypes.c_double, _I, _I,
                                                  _P, _P]
    lib.specv_oracle_check_hit.restype = None
    lib.specv_oracle_check_hit.argtypes = [_I, _I, _I, _P, _P, _P, _P]
    lib.specv_oracle_row_probs.restype = _I
    lib.specv_oracle_row_probs.argtypes = [_I, _I, _P, ctypes.c_double, _P]
    lib.specv_oracle_mss.restype = _I
    lib.specv_oracle_mss.argtypes = [_I, _I, _I, _I, _P, _L, _P, _L, _P, _P, _P, _P, _I,
                                     _P, _P, _P, _P, _P, _I]
    lib.specv_oracle_mss_law.restype = _I
    lib.specv_oracle_mss_law.argtypes = [_I, _P, _P, _P, _I, _I, _P, _P]
    _LIBS[path] = lib
    return lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return FP32
    if a.dtype in (np.int16, np.uint16):
        return BF16
    raise TypeError(f"logits must be float32 or int16 bf16 bits, got {a.dtype}")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_P)


def _strides(a: np.ndarray):
    it = a.itemsize
    return a.strides[0] // it, a.strides[1] // it


def verify(target, draft, tokens, temperature, uniforms, nthreads: int = 1,
           lib=None, no_draft: bool = False, saguaro=None) -> dict:
    """Run the oracle's verification on B batch rows.

    target [B, >=K+1, V], draft [B, >=K, V] (fp32 or int16 bf16 bits, rows
    contiguous along V), tokens int32 [B, K], temperature fp32 [B], uniforms
    fp32 [B, K+1].  Returns accept_len, out_tokens, p (=p_i(x_i)),
    q (=q_i(x_i)), alpha (=sum_v min(p_i, q_i)), status, boundary.
    no_draft: the draft distributions are one-hot at the sent tokens (the
    draft tensor is then ignored; pass the target).
    saguaro=(F, C): the drafts were sampled from sigma_{F,C}(z/T), so that is q.
    """
    lib = lib or load()
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B, K = tokens.shape
    V = target.shape[-1]
    if no_draft:
        draft = target
    assert target.strides[-1] == target.itemsize and draft.strides[-1] == draft.itemsize
    assert target.dtype == draft.dtype
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    out = dict(
        accept_len=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, K + 1), np.int32),
        p=np.zeros((B, K), np.float64),
        q=np.zeros((B, K), np.float64),
        alpha=np.zeros((B, K), np.float64),
        status=np.zeros(B, np.int32),
        boundary=np.zeros(B, np.int32),
    )
    tbs, trs = _strides(target)
    dbs, drs = _strides(draft)
    rc = lib.specv_oracle_verify(
        B, K, V, _dtype_code(target), _ptr(target), tbs, trs, _ptr(draft), dbs,
        drs, _ptr(tokens), _ptr(temperature), _ptr(uniforms), int(bool(no_draft)),
        int(saguaro[0]) if saguaro else 0, float(saguaro[1]) if saguaro else 1.0,
        _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["p"]),
        _ptr(out["q"]), _ptr(out["alpha"]), _ptr(out["status"]),
        _ptr(out["boundary"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle verify: bad sizes")
    return out


def saguaro_probs(z, T: float, F: int, C: float, lib=None) -> np.ndarray:
    """The oracle's sigma_{F,C}(z/T) of one logit row."""
    lib = lib or load()
    z = np.ascontiguousarray(z)
    p = np.zeros(z.shape[-1], np.float64)
    rc = lib.specv_oracle_saguaro_probs(z.shape[-1], _dtype_code(z), _ptr(z), float(T), int(F),
                                        float(C), _ptr(p))
    if rc & ROW_ERRORS:
        raise ValueError(f"row status {rc}")
    return p


def saguaro_sample(z, temperature, F: int, C: float, uniforms, lib=None) -> dict:
    """[SSD] §4.2.1 draft-side sampling: tokens [B] drawn from sigma_{F,C}(z/T)
    by inverse CDF of uniforms [B], with q = sigma(token) and row status."""
    lib = lib or load()
    z = np.ascontiguousarray(z)
    B, V = z.shape
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    out = dict(tokens=np.zeros(B, np.int32), q=np.zeros(B, np.float64),
               status=np.zeros(B, np.int32))
    rc = lib.specv_oracle_saguaro_sample(B, V, _dtype_code(z), _ptr(z), V, _ptr(temperature),
                                         int(F), float(C), _ptr(uniforms), _ptr(out["tokens"]),
                                         _ptr(out["q"]), _ptr(out["status"]))
    if rc != 0:
        raise ValueError("oracle saguaro_sample: bad arguments")
    return out


def verify_ragged(target, draft, cu, tokens, temperature, uniforms, Kmax: int,
                  nthreads: int = 1, lib=None, no_draft: bool = False) -> dict:
    """Verification with K_b = cu[b] - cu[b-1] drafts per row, packed rows.

    target [cu[-1] + B, V] (K_b + 1 rows per batch row, in order), draft
    [cu[-1], V] (ignored with no_draft), cu int32 [B] inclusive prefix sums,
    tokens int32 [cu[-1]], temperature fp32 [B], uniforms fp32 [cu[-1] + B].
    Returns accept_len [B], out_tokens [B, Kmax+1], p/q/alpha [cu[-1]],
    status [B], boundary [B].
    """
    lib = lib or load()
    cu = np.ascontiguousarray(cu, dtype=np.int32)
    B = cu.shape[0]
    T = int(cu[-1]) if B else 0
    target = np.ascontiguousarray(target)
    draft = target if no_draft else np.ascontiguousarray(draft)
    V = target.shape[-1]
    assert target.dtype == draft.dtype
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32)
    out = dict(
        accept_len=np.zeros(B, np.int32),
        out_tokens=np.zeros((B, Kmax + 1), np.int32),
        p=np.zeros(max(T, 1), np.float64),
        q=np.zeros(max(T, 1), np.float64),
        alpha=np.zeros(max(T, 1), np.float64),
        status=np.zeros(B, np.int32),
        boundary=np.zeros(B, np.int32),
    )
    rc = lib.specv_oracle_verify_ragged(
        B, Kmax, V, _dtype_code(target), _ptr(target), V, _ptr(draft), V, _ptr(cu),
        _ptr(tokens), _ptr(temperature), _ptr(uniforms), int(bool(no_draft)),
        _ptr(out["accept_len"]), _ptr(out["out_tokens"]), _ptr(out["p"]), _ptr(out["q"]),
        _ptr(out["alpha"]), _ptr(out["status"]), _ptr(out["boundary"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle verify_ragged: bad sizes")
    for k in ("p", "q", "alpha"):
        out[k] = out[k][:T]
    return out


def predict(draft, tokens, F: int, nthreads: int = 1, lib=None, fanout=None) -> dict:
    """Top-F outcome keys from draft logits [B, K+1, V]; tokens int32 [B, K].

    fanout (optional, K+1 ints in [0, F]): keep only the first fanout[k] keys
    at lookahead k (the rest are -1).
    """
    lib = lib or load()
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    B, K = tokens.shape
    V = draft.shape[-1]
    assert draft.shape[1] >= K + 1 and draft.strides[-1] == draft.itemsize
    keys = np.zeros((B, K + 1, F), np.int32)
    key_logits = np.zeros((B, K + 1, F), np.float32)
    status = np.zeros(B, np.int32)
    dbs, drs = _strides(draft)
    fan = None if fanout is None else np.ascontiguousarray(fanout, dtype=np.int32)
    assert fan is None or fan.shape == (K + 1,)
    rc = lib.specv_oracle_predict(B, K, V, F, _dtype_code(draft), _ptr(draft),
                                  dbs, drs, _ptr(tokens), None if fan is None else _ptr(fan),
                                  _ptr(keys), _ptr(key_logits), _ptr(status), int(nthreads))
    if rc != 0:
        raise ValueError("oracle predict: bad sizes")
    return dict(keys=keys, key_logits=key_logits, status=status)


def geometric_fanout(K: int, a: float, r: float, budget: int, max_f: int = 32,
                     lib=None) -> tuple:
    """[SSD] Theorem 12 fan-out: (integer F_k [K+1], real F_k [K+1])."""
    lib = lib or load()
    real = np.zeros(K + 1, np.float64)
    fk = np.zeros(K + 1, np.int32)
    rc = lib.specv_oracle_geometric_fanout(int(K), float(a), float(r), int(budget), int(max_f),
                                           _ptr(real), _ptr(fk))
    if rc != 0:
        raise ValueError("oracle geometric_fanout: bad arguments")
    return fk, real


def check_hit(keys, accept_len, out_tokens, lib=None) -> np.ndarray:
    lib = lib or load()
    keys = np.ascontiguousarray(keys, dtype=np.int32)
    accept_len = np.ascontiguousarray(accept_len, dtype=np.int32)
    out_tokens = np.ascontiguousarray(out_tokens, dtype=np.int32)
    B, K1, F = keys.shape
    hit = np.zeros(B, np.uint8)
    lib.specv_oracle_check_hit(B, K1 - 1, F, _ptr(keys), _ptr(accept_len),
                               _ptr(out_tokens), _ptr(hit))
    return hit


def row_probs(z, T: float, lib=None) -> np.ndarray:
    """The oracle's a1 distribution of one logit row (fp32 or bf16 bits)."""
    lib = lib or load()
    z = np.ascontiguousarray(z)
    p = np.zeros(z.shape[-1], np.float64)
    rc = lib.specv_oracle_row_probs(z.shape[-1], _dtype_code(z), _ptr(z),
                                    float(T), _ptr(p))
    if rc & ROW_ERRORS:
        raise ValueError(f"row status {rc}")
    return p


def mss(target, draft, cands, temperature, uniforms, num_cands=None, naive: bool = False,
        nthreads: int = 1, lib=None) -> dict:
    """[CS349D] §6.4 multi-step speculative sampling (naive=False) or naive
    sampling (naive=True) at B token-tree nodes.

    target, draft [B, V] (one row each per node; fp32 or int16 bf16 bits),
    cands int32 [B, M], num_cands int32 [B] or None (all M), temperature fp32
    [B], uniforms fp32 [B, M+1] (u_j for candidate j, column M for the draw).
    Returns accepted [B] (candidate index or -1), token [B], accept_prob
    [B, M], status [B], boundary [B].
    """
    lib = lib or load()
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    assert target.dtype == draft.dtype and target.ndim == 2 and draft.shape == target.shape
    B, V = target.shape
    cands = np.ascontiguousarray(cands, dtype=np.int32).reshape(B, -1)
    M = cands.shape[1]
    temperature = np.ascontiguousarray(temperature, dtype=np.float32)
    uniforms = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, M + 1)
    nc = None if num_cands is None else np.ascontiguousarray(num_cands, dtype=np.int32)
    out = dict(accepted=np.zeros(B, np.int32), token=np.zeros(B, np.int32),
               accept_prob=np.zeros((B, M), np.float64), status=np.zeros(B, np.int32),
               boundary=np.zeros(B, np.int32))
    rc = lib.specv_oracle_mss(B, M, V, _dtype_code(target), _ptr(target), V, _ptr(draft), V,
                              _ptr(cands), _ptr(nc) if nc is not None else None,
                              _ptr(temperature), _ptr(uniforms), int(bool(naive)),
                              _ptr(out["accepted"]), _ptr(out["token"]), _ptr(out["accept_prob"]),
                              _ptr(out["status"]), _ptr(out["boundary"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle mss: bad sizes")
    return out


def mss_law(p, q, cands, naive: bool = False, lib=None):
    """Exact law of the node's output token for one candidate tuple, given the
    distributions p, q (fp64 [V]); returns (law [V], P(some candidate
    accepted)).  Raises if a reachable residual has no mass."""
    lib = lib or load()
    p = np.ascontiguousarray(p, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    x = np.ascontiguousarray(cands, dtype=np.int32)
    law = np.zeros(p.shape[0], np.float64)
    pa = np.zeros(1, np.float64)
    rc = lib.specv_oracle_mss_law(p.shape[0], _ptr(p), _ptr(q), _ptr(x), x.shape[0],
                                  int(bool(naive)), _ptr(law), _ptr(pa))
    if rc != 0:
        raise ValueError("oracle mss_law: a reachable residual has no mass")
    return law, float(pa[0])
