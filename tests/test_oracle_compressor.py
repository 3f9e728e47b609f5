"""Pins of the oracle's compressor (C = H W_KV, Z = H W_Z, per-channel softmax
pooling over non-overlapping groups of m tokens, K^I = Cbar W_IK) against
closed forms and exact integer arithmetic done in numpy."""
import numpy as np

import synth
from synth.workloads import cache_write_inputs


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """Exact bf16 bit patterns of values that are representable in bf16."""
    b = np.asarray(x, np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0)
    return (b >> 16).astype(np.uint16)


def test_pool_identity_m1(oracle_mod):
    rng = np.random.default_rng(0)
    C = rng.standard_normal((7, 5))
    Z = rng.standard_normal((7, 5))
    assert np.array_equal(oracle_mod.pool(C, Z, 1), C)


def test_pool_constant_scores_give_mean(oracle_mod):
    rng = np.random.default_rng(1)
    C = rng.standard_normal((12, 9))
    Z = np.full((12, 9), 0.37)
    got = oracle_mod.pool(C, Z, 4)
    assert np.allclose(got, C.reshape(3, 4, 9).mean(1), rtol=1e-15, atol=1e-15)


def test_pool_dominant_score_selects(oracle_mod):
    C = np.arange(8.0).reshape(4, 2)
    Z = np.zeros((4, 2))
    Z[1, 0] = 800.0
    Z[2, 1] = 800.0
    got = oracle_mod.pool(C, Z, 2)
    assert got[0, 0] == C[1, 0] and got[0, 1] == 0.5 * (C[0, 1] + C[1, 1])
    assert got[1, 1] == C[2, 1]


def test_pool_two_token_logistic_closed_form(oracle_mod):
    rng = np.random.default_rng(2)
    C = rng.standard_normal((64, 16))
    Z = rng.standard_normal((64, 16)) * 4
    got = oracle_mod.pool(C, Z, 2)
    z0, z1 = Z[0::2], Z[1::2]
    s0 = 1.0 / (1.0 + np.exp(z1 - z0))
    ref = s0 * C[0::2] + (1.0 - s0) * C[1::2]
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-14)


def test_cache_write_dyadic_exact(oracle_mod):
    """H in {-1,0,1}, W in {-1,0,1}/16, m = 1: every sum is an exact integer
    multiple of 1/16 (or 1/256 for K^I), so numpy integer matmuls give the exact
    pre-quantization values; the bytes must equal the quantizer applied to them."""
    rng = np.random.default_rng(3)
    T, d = 24, 256
    H = rng.integers(-1, 2, (T, d))
    Wkv = rng.integers(-1, 2, (d, 512))
    Wz = rng.integers(-1, 2, (d, 512))
    Wik = rng.integers(-1, 2, (512, 128))
    C = (H @ Wkv) / 16.0
    KI = (H @ Wkv @ Wik) / 256.0
    out = oracle_mod.cache_write(_bf16_bits(H), _bf16_bits(Wkv / 16.0), _bf16_bits(Wz / 16.0),
                                 _bf16_bits(Wik / 16.0), 1, return_prequant=True)
    kvc, kvs, ixc, ixs, cb, ki, att = out
    assert np.array_equal(att, cb)  # no RMSNorm / RoPE: the main quantizer sees the pooled latent
    assert np.array_equal(cb, C)
    assert np.array_equal(ki, KI)
    c2, s2 = oracle_mod.quantize_main(C.astype(np.float32))
    i2, j2 = oracle_mod.quantize_index(KI.astype(np.float32))
    assert np.array_equal(kvc, c2) and np.array_equal(kvs, s2)
    assert np.array_equal(ixc, i2) and np.array_equal(ixs, j2)


def test_cache_write_m2_matches_numpy_pipeline(oracle_mod):
    """Gaussian inputs at m = 2 against a numpy fp64 restatement (matmul + logistic
    pooling + matmul): pre-quantization values agree to fp64 rounding."""
    H, Wkv, Wz, Wik = cache_write_inputs(3, 16, 5120)
    f = synth.bf16_to_f32
    Hf, Wkvf, Wzf, Wikf = (f(a).astype(np.float64) for a in (H, Wkv, Wz, Wik))
    C = Hf @ Wkvf
    Z = Hf @ Wzf
    s0 = 1.0 / (1.0 + np.exp(Z[1::2] - Z[0::2]))
    Cb = s0 * C[0::2] + (1 - s0) * C[1::2]
    KI = Cb @ Wikf
    _, _, _, _, cb, ki, _ = oracle_mod.cache_write(H, Wkv, Wz, Wik, 2, return_prequant=True)
    assert np.allclose(cb, Cb, rtol=1e-12, atol=1e-12)
    assert np.allclose(ki, KI, rtol=1e-11, atol=1e-12)


def test_cache_write_rejects_ragged(oracle_mod):
    import pytest

    H = np.zeros((3, 8), np.uint16)
    W = np.zeros((8, 512), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.cache_write(H, W, W, np.zeros((512, 128), np.uint16), 2)
