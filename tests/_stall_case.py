"""One verification call run in a fresh process with SPECV_TEST_STALL set (the
library reads it once per process): a bounded device wait is made to run out
and the call must still return, with the stalled batch row flagged
SPECV_ROW_DEVICE_TIMEOUT, its outputs those of an error row, every other row
equal to the oracle, and the CUDA context still usable.  Prints
"stall case ok <seconds>" or raises.  Run by tests/test_stall_gpu.py as
`python -m tests._stall_case <row>`.
"""
import sys
import time

import numpy as np
import torch

import oracle
import speculative_decoding_verification_50_gb300 as sv
from speculative_decoding_verification_50_gb300 import workloads as wl

# fp32 rows of 20000 logits (16-byte aligned: the staged paths), drafts far
# from the target so that most rows reject a draft (a residual pass).
SPEC = wl.custom("stall", B=6, K=3, V=20000, dtype=wl.FP32, temps=(0.7, 1.0),
                 sigma_d=(2.5, 3.0), seed=wl.SEED_BASE + 32000)


def main():
    row = int(sys.argv[1])
    sv.load_library()
    olib = oracle.load(oracle.build())
    d = wl.generate(SPEC)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    args = [dev(d[k]) for k in ("target", "draft", "tokens", "temperature", "uniforms")]
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    g = sv.specv_verify(*args)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    g = {k: v.cpu().numpy() for k, v in g.items()}
    st = g["row_status"]
    assert st[row] & sv.ROW_DEVICE_TIMEOUT, st
    assert (g["out_tokens"][row] == -1).all(), g["out_tokens"][row]
    assert dt > 0.3, dt  # a wait of about a second ran out
    o = oracle.verify(d["target"], d["draft"], d["tokens"], d["temperature"], d["uniforms"], lib=olib)
    rest = np.arange(SPEC.B) != row
    assert (st[rest] & sv.ROW_DEVICE_TIMEOUT == 0).all(), st
    ok = rest & (o["boundary"] == 0)
    assert np.array_equal(g["accept_len"][ok], o["accept_len"][ok]), (g["accept_len"], o["accept_len"])
    assert np.array_equal(g["out_tokens"][ok], o["out_tokens"][ok])
    assert np.abs(g["p_draft"][rest] - o["p"][rest]).max() <= 1e-5
    assert np.abs(g["q_draft"][rest] - o["q"][rest]).max() <= 1e-5
    # the context is still usable
    assert torch.arange(1000, device="cuda").sum().item() == 499500
    print(f"stall case ok {dt:.2f}")


if __name__ == "__main__":
    main()
