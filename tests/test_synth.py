"""The seeded input generator: determinism, slicing, distributions and the
roundings it applies (checked against torch's casts)."""
import numpy as np
import torch

import synth
from synth import workloads as W


def test_slices_are_consistent(synth_mod):
    full = synth.normal_f32(7, 3, 10000)
    part = synth.normal_f32(7, 3, 1000, offset=4321)
    assert np.array_equal(full[4321:5321], part)
    assert not np.array_equal(full, synth.normal_f32(8, 3, 10000))
    assert not np.array_equal(full, synth.normal_f32(7, 4, 10000))


def test_normal_moments_and_bounds(synth_mod):
    x = synth.normal_f32(0, 1, 1 << 21).astype(np.float64)
    assert abs(x.mean()) < 3e-3 and abs(x.var() - 1.0) < 3e-3
    assert np.abs(x).max() <= 6.0
    # exact in fp32: every value is an integer multiple of 2^-16
    assert np.all(np.round(x * 65536) == x * 65536)


def test_uniform(synth_mod):
    u = synth.uniform_f32(0, 5, 1 << 20)
    assert u.min() >= 0.0 and u.max() <= 1.0 and abs(u.mean() - 0.5) < 2e-3


def test_bf16_and_e4m3_roundings_match_torch(synth_mod):
    x = synth.normal_f32(3, 9, 100000, scale=0.37)
    b = synth.normal_bf16(3, 9, 100000, scale=0.37)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(b, ref)
    e = synth.e4m3_normal(3, 9, 100000, scale=0.37)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e, ref)


def test_hot_keys(synth_mod):
    q, w = W.index_query(2, 0, 2)
    hv = W.hot_vectors(q, w, 3.0)
    assert np.allclose(np.linalg.norm(hv.astype(np.float64), axis=1), 3.0, rtol=1e-6)
    n = 50000
    k = W.index_latents(2, 0, 2, n, 1, 0, n, 0.02, hv[1])
    base = W.index_latents(2, 0, 2, n, 1, 0, n)
    hot = np.any(k != base, axis=1)
    assert 0.017 < hot.mean() < 0.023
    assert np.allclose(k[hot] - base[hot], hv[1][None, :], atol=1e-5)
