"""The seeded generator: deterministic, correctly distributed, plants where stated."""
import math

import numpy as np

import synth


def test_deterministic_and_seed_dependent():
    a = synth.normal(10001, seed=7, stream=3, bf16=True)
    b = synth.normal(10001, seed=7, stream=3, bf16=True)
    c = synth.normal(10001, seed=8, stream=3, bf16=True)
    assert np.array_equal(a, b) and not np.array_equal(a, c)


def test_normal_moments():
    x = synth.to_f64(synth.normal(1 << 20, seed=1, stream=1, bf16=False))
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    # Box-Muller tails: P(|z| > 3) = 0.0027
    assert abs((np.abs(x) > 3).mean() - 0.0027) < 3e-4


def test_bf16_is_rne_of_float():
    xb = synth.normal(4096, seed=3, stream=9, bf16=True)
    xf = synth.normal(4096, seed=3, stream=9, bf16=False)
    # bf16 value is within half an ulp (2^-8 relative) of the float value
    err = np.abs(synth.bf16_to_f64(xb) - xf.astype(np.float64)) / np.maximum(np.abs(xf), 1e-30)
    assert err.max() <= 2.0 ** -8 + 1e-12


def test_needles_shift_keys_along_query_direction():
    wl = synth.WORKLOADS["c2"].replace(B=1, Hkv=2, Hq=8, L=4096)
    x = synth.make_inputs(wl)
    q = synth.to_f64(x.q)
    k = synth.to_f64(x.k)
    for g in range(wl.B * wl.Hkv):
        qs = q[0, :, g * wl.G:(g + 1) * wl.G].reshape(-1, wl.d).sum(0)
        qhat = qs / np.linalg.norm(qs)
        blocks = k[0, g].reshape(wl.nb, wl.Bk, wl.d).mean(1) @ qhat
        needles = np.nonzero(x.needle_mask[g])[0]
        assert len(needles) == wl.needles
        assert set(needles) <= set(range(1, wl.nb - 1))
        # needle block means sit alpha along qhat, the others near 0 (std 1/8)
        assert np.all(np.abs(blocks[needles] - wl.alpha) < 0.6)
        others = np.setdiff1d(np.arange(wl.nb), needles)
        assert np.abs(blocks[others]).max() < 0.7


def test_plant_is_rank_r():
    wl = synth.WORKLOADS["c4"].replace(L=1024, Hq=4, Hkv=1)
    x = synth.make_inputs(wl)
    k = synth.to_f64(x.k)[0, 0]
    # block means carry gamma * U e_b (+ noise of std 1/sqrt(Bk)): rank ~ r above the noise
    means = k.reshape(wl.nb, wl.Bk, wl.d).mean(1)
    sv = np.linalg.svd(means, compute_uv=False)
    noise = 1.0 / math.sqrt(wl.Bk) * (math.sqrt(wl.nb) + math.sqrt(wl.d))
    assert (sv > 2 * noise).sum() == wl.plant_rank
