"""The seeded input generators against the configurations' recipes: the
logit distributions, the draft-token draws, the per-row streams and the bf16
rounding.  CPU only; the generators hold none of the method's arithmetic, so
these tests restate the recipes with plain numpy."""
import dataclasses

import numpy as np
import pytest

from speculative_decoding_verification_50_gb300 import workloads as wl


def f32(spec, x):
    return wl.bf16_bits_to_f32(x) if spec.dtype == wl.BF16 else x


def test_rows_do_not_depend_on_the_subset():
    spec = wl.custom("subset", B=9, K=3, V=300, dtype=wl.BF16, temps=(0.0, 0.8),
                     sigma_d=(0.5, 2.0), seed=wl.SEED_BASE + 77)
    full = wl.generate(spec)
    part = wl.generate(spec, rows=[7, 2, 5], threads=1)
    for k in ("target", "draft", "tokens", "temperature", "uniforms"):
        assert np.array_equal(part[k], full[k][[7, 2, 5]]), k


def test_cfg1_recipe():
    spec = wl.SPECS["cfg1"]
    d = wl.generate(spec)
    zt, zd = d["target"][0], d["draft"][0]
    assert zt.dtype == np.float32 and zt.shape == (5, 4096) and zd.shape == (4, 4096)
    assert abs(zt.std() - 2.0) < 0.05 and abs(zt.mean()) < 0.05
    e = zd - zt[:4]
    assert abs(e.std() - 1.0) < 0.03 and abs(e.mean()) < 0.03
    assert (d["temperature"] == 1.0).all()


def test_cfg3_recipe():
    spec = dataclasses.replace(wl.SPECS["cfg3"], V=20000)  # same recipe, shorter rows
    d = wl.generate(spec)
    zt, zd = f32(spec, d["target"]), f32(spec, d["draft"])
    assert abs(zt.std() - 3.0) < 0.02
    assert set(np.unique(d["temperature"]).tolist()) == {0.0, np.float32(0.6), 1.0}
    s = d["sigma_d"]
    assert (s >= 0.5).all() and (s <= 3.0).all() and s.max() - s.min() > 1.5
    for b in range(spec.B):
        e = zd[b] - zt[b, :spec.K]
        # the draft noise std is the row's sigma_b (bf16 rounding adds ~1e-2 relative)
        assert abs(e.std() / s[b] - 1.0) < 0.03, (b, e.std(), s[b])


def test_cfg5_recipe():
    spec = wl.SPECS["cfg5"]
    d = wl.generate(spec, rows=[0, 1])
    zt, zd = d["target"], d["draft"]
    V = spec.V
    base = -1.1 * np.log(np.arange(1, V + 1, dtype=np.float64))
    for b in range(2):
        for i in range(spec.K + 1):
            z = zt[b, i].astype(np.float64)
            # the values are the ranked base plus N(0, 0.5^2) noise, permuted:
            # mean and variance of the multiset
            assert abs(z.mean() - base.mean()) < 0.02
            assert abs(z.var() - (base.var() + 0.25)) < 0.03
        # permuted per row: the largest logit sits at a different index on each row
        assert len(set(np.argmax(zt[b], axis=1).tolist())) > 1
        for i in range(spec.K):
            x = zt[b, i].astype(np.float64)
            y = zd[b, i].astype(np.float64)
            slope = np.cov(x, y)[0, 1] / x.var()
            resid = y - 0.8 * x
            assert abs(slope - 0.8) < 0.01 and abs(resid.std() - 1.0) < 0.01 and abs(resid.mean()) < 0.01


def test_draft_tokens_follow_the_draft_distribution():
    """T > 0: tokens are draws from softmax(z_d/T) (expected counts per token
    over many rows); T = 0: the first argmax of the stored draft row."""
    spec = wl.custom("draws", B=20000, K=1, V=6, temps=(0.0, 0.5, 1.3), sigma_t=1.5,
                     sigma_d=(1.0, 1.0), seed=wl.SEED_BASE + 91)
    d = wl.generate(spec)
    z = d["draft"][:, 0].astype(np.float64)
    T = d["temperature"]
    x = d["tokens"][:, 0]
    g = T == 0
    assert g.any() and (x[g] == np.argmax(z[g], axis=1)).all()
    s = ~g
    zz = z[s] / T[s, None]
    q = np.exp(zz - zz.max(axis=1, keepdims=True))
    q /= q.sum(axis=1, keepdims=True)
    expect = q.sum(axis=0)
    var = (q * (1 - q)).sum(axis=0)
    count = np.bincount(x[s], minlength=6)
    assert (np.abs(count - expect) < 5 * np.sqrt(var)).all(), (count, expect)


def test_uniforms_and_layout():
    spec = wl.custom("layout", B=4, K=3, V=50, ssd=True, seed=wl.SEED_BASE + 92)
    d = wl.generate(spec)
    assert d["draft"].shape == (4, 4, 50) and d["target"].shape == (4, 4, 50)
    u = d["uniforms"]
    assert u.dtype == np.float32 and u.shape == (4, 4) and (u >= 0).all() and (u < 1).all()


@pytest.mark.parametrize("x,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),               # halfway: to the even mantissa
    (1.0 + 3 * 2.0 ** -8, 0x3F82),           # halfway: up to the even one
    (1.0 + 2.0 ** -8 + 2.0 ** -20, 0x3F81),  # past halfway: up
    (-2.0, 0xC000),
    (float("inf"), 0x7F80),
    (float("-inf"), 0xFF80),
])
def test_bf16_round_to_nearest_even(x, bits):
    got = wl.f32_to_bf16_bits(np.array([x], np.float32)).view(np.uint16)[0]
    assert got == bits, hex(got)


def test_bf16_round_trip_and_error_bound():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(100000) * 10).astype(np.float32)
    y = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(x))
    assert (np.abs(y - x) <= np.abs(x) * 2.0 ** -8).all()  # half an ulp of bf16
    assert np.array_equal(wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(y)), y)
    assert np.isnan(wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(np.array([np.nan], np.float32))))[0]


def test_mss_nodes():
    spec = wl.custom("nodes", B=1, K=1, V=40, temps=(0.0, 1.0), seed=wl.SEED_BASE + 93)
    m = wl.generate_mss(spec, 3, B=200)
    assert m["candidates"].shape == (200, 3) and m["uniforms"].shape == (200, 4)
    g = m["temperature"] == 0
    z = m["draft"].astype(np.float64)
    assert g.any() and (m["candidates"][g, 0] == np.argmax(z[g], axis=1)).all()
    assert ((m["candidates"] >= 0) & (m["candidates"] < 40)).all()
