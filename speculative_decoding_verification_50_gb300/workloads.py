"""Seeded synthetic inputs for speculative-sampling verification.

This module is the one piece shared by the CUDA path's tests and benchmark
and by the CPU oracle's tests.  It draws random numbers and rounds them to
the storage dtype; it holds none of the verification arithmetic (no softmax,
no acceptance test, no residual, no top-F).  Draft tokens are drawn with the
Gumbel-max trick (argmax of z/T plus Gumbel noise), which samples from the
draft distribution without forming it; greedy rows (T = 0) take the first
argmax of the draft logits.

Workloads follow the five synthetic configurations of the method's
benchmark plan (LLM vocabularies: Llama-3 V=128256, Qwen V=152064):

  cfg1   B=1,  K=4, V=4096,   fp32, z_t ~ N(0, 2^2), z_d = z_t + N(0, 1), T=1
  cfg2a  B=1,  K=5, V=128256, bf16, z_t ~ N(0, 3^2) with +6 on 8 random ids
         per row, z_d = z_t + N(0, 1.5^2), T=0 (greedy)
  cfg2b  as cfg2a with T=0.7
  cfg3   B=64, K=4, V=128256, bf16, z_t ~ N(0, 3^2), T_b from {0, 0.6, 1.0},
         z_d = z_t + N(0, sigma_b^2), sigma_b ~ U[0.5, 3]
  cfg4   B=32, K=4, V=128256, bf16, as cfg3 at T=1, draft logits at K+1
         positions (SSD layout), fan-out F=6
  cfg5   B=256, K=8, V=152064, fp32, z_t at sorted rank r is
         -1.1 ln r + N(0, 0.5^2), permuted per row, z_d = 0.8 z_t + N(0, 1), T=1

Every batch row b draws from its own PCG64 stream seeded by (seed, b), so the
bytes of a row do not depend on B, on which rows are generated, or on the
number of threads used to fill them.  Uniforms are fp32 in [0, 1).

bf16 logits are stored as int16 bit patterns (round-to-nearest-even from the
fp32 draw); numpy has no bf16 type.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BF16 = "bf16"
FP32 = "fp32"

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Spec:
    """Shape and distribution recipe of one synthetic workload."""

    name: str
    B: int
    K: int
    V: int
    dtype: str
    kind: str                 # "normal" | "boosted" | "zipf"
    sigma_t: float = 3.0      # target logit std ("normal", "boosted")
    sigma_d: tuple = (1.0, 1.0)  # draft noise std range (lo, hi), per batch row
    temps: tuple = (1.0,)     # temperatures drawn uniformly per batch row
    F: int = 0                # top-F fan-out (0: no outcome prediction)
    ssd: bool = False         # draft logits at K+1 positions instead of K
    boost_ids: int = 0
    boost: float = 0.0
    draft_scale: float = 1.0  # z_d = draft_scale * z_t + noise
    seed: int = 0

    @property
    def draft_rows(self) -> int:
        return self.K + 1 if self.ssd else self.K

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == BF16 else 4


SPECS = {
    "cfg1": Spec("cfg1", B=1, K=4, V=4096, dtype=FP32, kind="normal",
                 sigma_t=2.0, sigma_d=(1.0, 1.0), temps=(1.0,),
                 seed=SEED_BASE + 1000),
    "cfg2a": Spec("cfg2a", B=1, K=5, V=128256, dtype=BF16, kind="boosted",
                  sigma_t=3.0, sigma_d=(1.5, 1.5), temps=(0.0,),
                  boost_ids=8, boost=6.0, seed=SEED_BASE + 2000),
    "cfg2b": Spec("cfg2b", B=1, K=5, V=128256, dtype=BF16, kind="boosted",
                  sigma_t=3.0, sigma_d=(1.5, 1.5), temps=(0.7,),
                  boost_ids=8, boost=6.0, seed=SEED_BASE + 2001),
    "cfg3": Spec("cfg3", B=64, K=4, V=128256, dtype=BF16, kind="normal",
                 sigma_t=3.0, sigma_d=(0.5, 3.0), temps=(0.0, 0.6, 1.0),
                 seed=SEED_BASE + 3000),
    "cfg4": Spec("cfg4", B=32, K=4, V=128256, dtype=BF16, kind="normal",
                 sigma_t=3.0, sigma_d=(0.5, 3.0), temps=(1.0,), F=6, ssd=True,
                 seed=SEED_BASE + 4000),
    "cfg5": Spec("cfg5", B=256, K=8, V=152064, dtype=FP32, kind="zipf",
                 sigma_d=(1.0, 1.0), temps=(1.0,), draft_scale=0.8,
                 seed=SEED_BASE + 5000),
}


def custom(name: str = "custom", **kw) -> Spec:
    """A workload with explicit sizes (ragged V, K, B for edge cases)."""
    base = dict(B=2, K=3, V=1000, dtype=FP32, kind="normal", sigma_t=2.0,
                sigma_d=(1.0, 1.0), temps=(1.0,), seed=SEED_BASE + 9000)
    base.update(kw)
    return Spec(name, **base)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); return int16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return rounded.astype(np.uint16).view(np.int16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen int16 bf16 bit patterns to fp32 (exact)."""
    u = bits.view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == BF16 else x32.astype(np.float32)


def _stored_as_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f32(x) if dtype == BF16 else x


def _row_rng(spec: Spec, b: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([spec.seed, b])))


def _gumbel_argmax(rng: np.random.Generator, z: np.ndarray, T: float) -> int:
    """Index of max(z/T + g), g ~ Gumbel(0, 1): a draw from softmax(z/T)."""
    g = rng.gumbel(size=z.shape[-1])
    return int(np.argmax(z.astype(np.float64) / T + g))


def _fill_row(spec: Spec, b: int, out: dict, j: int) -> None:
    """Draw batch row b and store it at position j of the output arrays."""
    rng = _row_rng(spec, b)
    K, V = spec.K, spec.V
    T = float(spec.temps[rng.integers(len(spec.temps))]) if len(spec.temps) > 1 else float(spec.temps[0])
    lo, hi = spec.sigma_d
    sigma_d = float(rng.uniform(lo, hi)) if hi > lo else float(lo)

    if spec.kind == "zipf":
        base = -1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))
        zt = (base[None, :] + rng.normal(0.0, 0.5, size=(K + 1, V))).astype(np.float32)
        zt = rng.permuted(zt, axis=1)
    else:
        zt = rng.standard_normal(size=(K + 1, V), dtype=np.float32) * np.float32(spec.sigma_t)
        if spec.kind == "boosted":
            for i in range(K + 1):
                ids = rng.choice(V, size=spec.boost_ids, replace=False)
                zt[i, ids] += np.float32(spec.boost)
    zt_stored = _store(zt, spec.dtype)
    zt_exact = _stored_as_f32(zt_stored, spec.dtype)

    R = spec.draft_rows
    noise = rng.standard_normal(size=(R, V), dtype=np.float32) * np.float32(sigma_d)
    zd = np.float32(spec.draft_scale) * zt_exact[:R] + noise
    zd_stored = _store(zd, spec.dtype)
    zd_exact = _stored_as_f32(zd_stored, spec.dtype)

    tokens = np.empty(K, dtype=np.int32)
    for i in range(K):
        if T == 0.0:
            tokens[i] = int(np.argmax(zd_exact[i]))
        else:
            tokens[i] = _gumbel_argmax(rng, zd_exact[i], T)
    uniforms = rng.random(K + 1, dtype=np.float32)

    out["target"][j] = zt_stored
    out["draft"][j] = zd_stored
    out["tokens"][j] = tokens
    out["temperature"][j] = np.float32(T)
    out["uniforms"][j] = uniforms
    out["sigma_d"][j] = sigma_d


def generate(spec: Spec, rows=None, threads: int | None = None) -> dict:
    """Materialise a workload on the host.

    rows: optional list of batch-row indices to generate (default: all B).
      Row b's bytes are the same whichever subset is asked for.
    Returns a dict with numpy arrays:
      target      [b, K+1, V]   fp32, or int16 bf16 bits
      draft       [b, R, V]     R = K (verify layout) or K+1 (SSD layout)
      tokens      [b, K]        int32 draft tokens x_1..x_K
      temperature [b]           fp32 (0 = greedy)
      uniforms    [b, K+1]      fp32 in [0,1); columns 0..K-1 drive the
                                accept tests, column K the bonus draw
      sigma_d     [b]           draft noise std actually used (diagnostic)
    and the spec under "spec", the generated rows under "rows".
    """
    rows = list(range(spec.B)) if rows is None else [int(r) for r in rows]
    n = len(rows)
    st = np.int16 if spec.dtype == BF16 else np.float32
    out = {
        "target": np.empty((n, spec.K + 1, spec.V), dtype=st),
        "draft": np.empty((n, spec.draft_rows, spec.V), dtype=st),
        "tokens": np.empty((n, spec.K), dtype=np.int32),
        "temperature": np.empty(n, dtype=np.float32),
        "uniforms": np.empty((n, spec.K + 1), dtype=np.float32),
        "sigma_d": np.empty(n, dtype=np.float64),
    }

    def work(j_b):
        j, b = j_b
        _fill_row(spec, b, out, j)

    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    items = list(enumerate(rows))
    if threads <= 1 or n <= 1:
        for it in items:
            work(it)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, items))
    out["spec"] = spec
    out["rows"] = np.asarray(rows, dtype=np.int64)
    return out


# ---------------------------------------------------------------------------
# Token-tree nodes for multi-step speculative sampling

def _fill_node(spec: Spec, M: int, b: int, out: dict, j: int) -> None:
    """Node b: one target row and one draft row drawn by spec's recipe (its
    kind, temperature set and draft noise), M candidate children drawn
    independently from softmax(z_d/T) by the Gumbel-max trick (a greedy node
    proposes the draft argmax first, then draws at T = 1), and M+1 uniforms."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([spec.seed, b, 0x3155])))
    V = spec.V
    T = float(spec.temps[rng.integers(len(spec.temps))]) if len(spec.temps) > 1 else float(spec.temps[0])
    lo, hi = spec.sigma_d
    sigma_d = float(rng.uniform(lo, hi)) if hi > lo else float(lo)
    if spec.kind == "zipf":
        base = -1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))
        zt = rng.permuted((base + rng.normal(0.0, 0.5, size=V)).astype(np.float32))
    else:
        zt = rng.standard_normal(size=V, dtype=np.float32) * np.float32(spec.sigma_t)
        if spec.kind == "boosted":
            zt[rng.choice(V, size=spec.boost_ids, replace=False)] += np.float32(spec.boost)
    zt_stored = _store(zt, spec.dtype)
    zd = np.float32(spec.draft_scale) * _stored_as_f32(zt_stored, spec.dtype) + \
        rng.standard_normal(size=V, dtype=np.float32) * np.float32(sigma_d)
    zd_stored = _store(zd, spec.dtype)
    zd_exact = _stored_as_f32(zd_stored, spec.dtype)
    cands = np.empty(M, dtype=np.int32)
    for i in range(M):
        if T == 0.0:
            cands[i] = int(np.argmax(zd_exact)) if i == 0 else _gumbel_argmax(rng, zd_exact, 1.0)
        else:
            cands[i] = _gumbel_argmax(rng, zd_exact, T)
    out["target"][j] = zt_stored
    out["draft"][j] = zd_stored
    out["candidates"][j] = cands
    out["temperature"][j] = np.float32(T)
    out["uniforms"][j] = rng.random(M + 1, dtype=np.float32)


def generate_mss(spec: Spec, M: int, B: int | None = None, rows=None,
                 threads: int | None = None) -> dict:
    """Materialise B token-tree nodes (default spec.B) for multi-step
    speculative sampling with M candidates each.  Returns numpy arrays
      target [n, V], draft [n, V]   fp32, or int16 bf16 bits
      candidates [n, M]             int32, drawn i.i.d. from the draft softmax
      temperature [n]               fp32 (0 = greedy)
      uniforms [n, M+1]             fp32 in [0,1): u_j for candidate j, column
                                    M for the final draw
    Node b's bytes do not depend on which nodes are generated."""
    B = spec.B if B is None else B
    rows = list(range(B)) if rows is None else [int(r) for r in rows]
    n = len(rows)
    st = np.int16 if spec.dtype == BF16 else np.float32
    out = {
        "target": np.empty((n, spec.V), dtype=st),
        "draft": np.empty((n, spec.V), dtype=st),
        "candidates": np.empty((n, M), dtype=np.int32),
        "temperature": np.empty(n, dtype=np.float32),
        "uniforms": np.empty((n, M + 1), dtype=np.float32),
    }
    if threads is None:
        threads = min(16, os.cpu_count() or 1)
    items = list(enumerate(rows))
    if threads <= 1 or n <= 1:
        for j, b in items:
            _fill_node(spec, M, b, out, j)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda it: _fill_node(spec, M, it[1], out, it[0]), items))
    out["rows"] = np.asarray(rows, dtype=np.int64)
    return out
