"""One parity case run in a fresh process, so that the library reads the
SPECV_* tuning variables of this environment (they are read once per
process): an SSD round (B=8, K=4, V=20000 bf16, F=6, mixed temperatures),
the Saguaro sampler and MSS, each against the oracle.  Prints "knob case ok"
or raises.  Run by tests/test_knobs_gpu.py as `python -m tests._knob_case`.
"""
import numpy as np
import torch

import oracle
import speculative_decoding_verification_50_gb300 as sv
from speculative_decoding_verification_50_gb300 import workloads as wl


def dev(a, bf16=False):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.view(torch.bfloat16) if bf16 else t).cuda()


def main():
    sv.load_library()
    olib = oracle.load(oracle.build())
    spec = wl.custom("knob", B=8, K=4, V=20000, dtype=wl.BF16, temps=(0.0, 0.7, 1.0),
                     sigma_d=(0.3, 2.0), F=6, ssd=True, seed=wl.SEED_BASE + 31000)
    d = wl.generate(spec)
    g = sv.specv_ssd_round(dev(d["target"], True), dev(d["draft"], True), dev(d["tokens"]),
                           dev(d["temperature"]), dev(d["uniforms"]), spec.F)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = oracle.verify(d["target"], d["draft"], d["tokens"], d["temperature"], d["uniforms"], lib=olib)
    op = oracle.predict(d["draft"], d["tokens"], spec.F, lib=olib)
    ok = o["boundary"] == 0
    assert np.array_equal(g["accept_len"][ok], o["accept_len"][ok]), (g["accept_len"], o["accept_len"])
    assert np.array_equal(g["out_tokens"][ok], o["out_tokens"][ok])
    assert np.abs(g["p_draft"] - o["p"]).max() <= 1e-5 and np.abs(g["q_draft"] - o["q"]).max() <= 1e-5
    assert np.array_equal(g["keys"], op["keys"])

    z = d["draft"].reshape(-1, spec.V)
    T = np.repeat(d["temperature"], spec.K + 1).astype(np.float32)
    U = np.random.default_rng(5).uniform(0, 1, z.shape[0]).astype(np.float32)
    s = sv.specv_saguaro_sample(dev(z, True), dev(T), 6, 0.3, dev(U))
    torch.cuda.synchronize()
    os_ = oracle.saguaro_sample(z, T, 6, 0.3, U, lib=olib)
    tok = s["tokens"].cpu().numpy()
    for b in np.nonzero(tok != os_["tokens"])[0]:  # only draws at a CDF boundary may differ
        q = oracle.saguaro_probs(z[b], float(T[b]), 6, 0.3, lib=olib)
        cs = np.cumsum(q)
        t = int(os_["tokens"][b])
        assert min(abs(U[b] - (cs[t - 1] if t else 0.0)), abs(cs[t] - U[b])) < 1e-6, b

    m = wl.generate_mss(spec, 3, B=16)
    r = sv.specv_mss_verify(dev(m["target"], True), dev(m["draft"], True), dev(m["candidates"]),
                            dev(m["temperature"]), dev(m["uniforms"]))
    torch.cuda.synchronize()
    om = oracle.mss(m["target"], m["draft"], m["candidates"], m["temperature"], m["uniforms"], lib=olib)
    okm = om["boundary"] == 0
    assert np.array_equal(r["out_token"].cpu().numpy()[okm], om["token"][okm])
    assert np.array_equal(r["accepted"].cpu().numpy()[okm], om["accepted"][okm])
    print("knob case ok")


if __name__ == "__main__":
    main()
