"""The Saguaro sampler against the oracle on batches that exercise its
decision paths, run in a fresh process so that the library reads this
environment's SPECV_SAMPLE_WARP (one warp per row when 1, one CTA per row
when 0; the variable is read once per process).  Each case mixes greedy
rows, rows whose top keys hold most of the mass (the whole-row pass; two of them
share a CTA), a row
with a bad temperature and a row holding NaN, and ends on a partial CTA; one
case's rows are padded (16-byte aligned rows whose last vector is ragged).
Prints "sampler case ok <rows>" or raises.  Run by
tests/test_sampler_warp_gpu.py as `python -m tests._sampler_case`.
"""
import numpy as np
import torch

import oracle
import speculative_decoding_verification_50_gb300 as sv
from speculative_decoding_verification_50_gb300 import workloads as wl

PROB_TOL = 1e-5

# (rows, V, dtype, F, C): fp32 and bf16 rows of the benchmark vocabularies,
# a shorter aligned row, the widest key set at weight 0, and no keys at all
CASES = [
    (300, 152064, wl.FP32, 6, 0.3),
    (313, 128256, wl.BF16, 1, 0.25),
    (257, 50000, wl.FP32, 32, 0.0),
    (67, 152064, wl.FP32, 0, 1.0),
    (130, 50001, wl.FP32, 6, 0.3),  # rows padded to 50004: a ragged last vector
    (70, 4096, wl.FP32, 6, 0.3),    # short rows: one chunk, most pieces empty
    (70, 1000, wl.BF16, 3, 0.5),
]


def dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(torch.bfloat16) if bf16 else t).cuda()


def near_boundary(z, T, F, C, U, tok, olib):
    if T == 0:
        return False
    q = oracle.saguaro_probs(z, T, F, C, lib=olib)
    cs = np.cumsum(q)
    lo = cs[tok - 1] if tok > 0 else 0.0
    return abs(U - lo) < 1e-6 or abs(cs[tok] - U) < 1e-6


def run_case(rows, V, dtype, F, C, olib, seed):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 2.5, (rows, V)).astype(np.float32)
    heavy = (3, 16, 17, rows // 2, rows - 1)  # the keys hold most of the mass (16, 17: one CTA)
    for b in heavy:
        z[b, rng.choice(V, 6, replace=False)] += 16.0
    z[9, min(1234, V - 1)] = np.nan
    T = rng.choice([0.0, 0.7, 1.0, 1.3], rows).astype(np.float32)
    T[5] = -1.0
    T[list(heavy)] = 1.0
    U = rng.uniform(0, 1, rows).astype(np.float32)
    bf16 = dtype == wl.BF16
    zz = wl.f32_to_bf16_bits(z) if bf16 else z
    zdev = dev(zz, bf16)
    pad = (-V) % (8 if bf16 else 4)
    if pad:  # the same rows in a buffer whose rows start 16-byte aligned
        buf = torch.zeros((rows, V + pad), dtype=zdev.dtype, device=zdev.device)
        buf[:, :V] = zdev
        zdev = buf[:, :V]
    g = sv.specv_saguaro_sample(zdev, dev(T), F, C, dev(U))
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.saguaro_sample(zz, T, F, C, U, lib=olib)
    err = o["status"] & oracle.ROW_ERRORS
    assert err[5] and err[9], err[:12]
    assert np.array_equal(g["row_status"] & oracle.ROW_ERRORS, err), (g["row_status"], o["status"])
    ok = err == 0
    assert (g["tokens"][~ok] == -1).all()
    differ = 0
    for b in np.nonzero(ok)[0]:
        if g["tokens"][b] != o["tokens"][b]:
            assert near_boundary(zz[b], float(T[b]), F, C, float(U[b]), int(o["tokens"][b]), olib), \
                (rows, V, b, g["tokens"][b], o["tokens"][b], T[b])
            differ += 1
        else:
            assert abs(g["q"][b] - o["q"][b]) <= PROB_TOL, (rows, V, b, g["q"][b], o["q"][b])
    assert differ <= max(1, rows // 50), differ


def main():
    sv.load_library()
    olib = oracle.load(oracle.build())
    n = 0
    for i, case in enumerate(CASES):
        run_case(*case, olib=olib, seed=wl.SEED_BASE + 33000 + i)
        n += case[0]
    print(f"sampler case ok {n}")


if __name__ == "__main__":
    main()
