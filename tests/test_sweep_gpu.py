"""A seeded sweep of verification and SSD-round shapes against the oracle.

The hand-picked cases elsewhere pin the benchmark configurations and the
edge cases; this sweep draws 64 more shapes from a fixed seed, so that the
host's choices that depend on the sizes (chunk length and count, the
one-wave rule, the kernel-B cluster size and slice, the chunk-local draw,
ring or direct residual pass) meet combinations nobody picked: batch sizes
from 1 to 1216 across the cluster-size thresholds, K from 1 to 12, V from 1
to 152064, both dtypes, the three logit recipes, mixed temperatures and
F from 1 to 12.  Same bars as tests/test_parity_gpu.py: every row the oracle
does not flag is exact, and at most 2 % of the rows (at least one) differ.
The flagged rows themselves are only counted: a flat row of 152064 logits
has many tokens of probability below 2e-6, and a draw of such a token is
flagged whatever U is (both ends of its CDF step lie within 1e-6 of U).
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verification_50_gb300 import workloads as wl
from tests.test_parity_gpu import (compare_ssd, compare_verify, differing_rows, gpu_ssd, gpu_verify,
                                    oracle_ssd, oracle_verify)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

MAX_LOGITS = 60_000_000  # per case, so the oracle finishes each in a second or so


def _shapes(n=64, seed=20261202):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        B = int(rng.choice([1, 2, 3, 7, 8, 9, 17, 31, 64, 100, 150, 256, 300, 600, 1216]))
        K = int(rng.integers(1, 13))
        band = int(rng.integers(0, 5))
        V = int([rng.integers(1, 300), rng.integers(300, 5000), rng.integers(5000, 70000),
                 128256, 152064][band])
        ssd = bool(rng.integers(0, 2))
        if B * (2 * K + 2) * V > MAX_LOGITS:
            continue
        dtype = wl.FP32 if rng.integers(0, 2) else wl.BF16
        kind = str(rng.choice(["normal", "boosted", "zipf"]))
        temps = tuple(sorted(set(float(t) for t in rng.choice([0.0, 0.5, 0.8, 1.0, 1.5],
                                                              int(rng.integers(1, 4))))))
        F = int(rng.integers(1, 13)) if ssd else 0
        out.append(dict(B=B, K=K, V=V, dtype=dtype, kind=kind, temps=temps, ssd=ssd, F=F,
                        seed=wl.SEED_BASE + 12000 + len(out)))
    return out


SHAPES = _shapes()


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


def _id(s):
    mode = f"ssdF{s['F']}" if s["ssd"] else "verify"
    return f"{mode}-B{s['B']}-K{s['K']}-V{s['V']}-{s['dtype']}-{s['kind']}"


@pytest.mark.parametrize("shape", SHAPES, ids=_id)
def test_sweep_matches_oracle(sv, olib, shape):
    extra = dict(boost_ids=min(8, shape["V"]), boost=6.0) if shape["kind"] == "boosted" else {}
    if shape["kind"] == "zipf":
        extra = dict(draft_scale=0.8)
    spec = wl.custom(_id(shape), B=shape["B"], K=shape["K"], V=shape["V"], dtype=shape["dtype"],
                     kind=shape["kind"], temps=shape["temps"], sigma_d=(0.3, 2.5), ssd=shape["ssd"],
                     F=shape["F"], seed=shape["seed"], **extra)
    data = wl.generate(spec)
    if shape["ssd"]:
        g = gpu_ssd(sv, data, shape["F"])
        o, keys, kl = oracle_ssd(olib, data, shape["F"])
        compare_ssd(olib, g, o, keys, kl, data["temperature"], _id(shape))
    else:
        g = gpu_verify(sv, data)
        o = oracle_verify(olib, data)
        compare_verify(g, o, data["temperature"], _id(shape))
    nd = differing_rows(g, o)
    assert nd <= max(1, shape["B"] // 50), nd
