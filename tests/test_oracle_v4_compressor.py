"""Pins of the oracle's V4 compressors ("DeepSeek-V4: Towards Highly Efficient
Million-Token Context Intelligence", CSA step 1 and HCA): the two-path
overlapping pool with position biases B^a, B^b (entry i draws from block i of
path a and block i-1 of path b, entry 0 from block 0 of path a alone) and the
single-path HCA pool with bias B, checked against closed forms (two-token
logistic, equal scores -> means, a dominant bias -> one row), reductions to the
separately pinned non-overlapping pool, exact integer arithmetic and brute-force
locality."""
import numpy as np
import pytest

import synth
from synth.workloads import hca_compressor_inputs, overlap_compressor_inputs


def _bits(x):
    b = np.asarray(x, np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0)
    return (b >> 16).astype(np.uint16)


def _rand(seed, *shape, s=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * s


def test_overlap_m1_two_token_logistic(oracle_mod):
    """m = 1: entry i > 0 mixes Ca[i] and Cb[i-1] with the logistic of the
    biased score difference; entry 0 is Ca[0]."""
    T, w = 9, 6
    Ca, Za, Cb, Zb = (_rand(k, T, w, s=3) for k in range(4))
    Ba, Bb = _rand(4, 1, w).astype(np.float32), _rand(5, 1, w).astype(np.float32)
    got = oracle_mod.pool_overlap(Ca, Za, Cb, Zb, Ba, Bb, 1)
    za = Za[1:] + Ba.astype(np.float64)
    zb = Zb[:-1] + Bb.astype(np.float64)
    s = 1.0 / (1.0 + np.exp(zb - za))
    ref = s * Ca[1:] + (1.0 - s) * Cb[:-1]
    assert np.array_equal(got[0], Ca[0])
    assert np.allclose(got[1:], ref, rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("m", [2, 4])
def test_overlap_equal_scores_give_means(oracle_mod, m):
    T, w = 5 * m, 7
    Ca, Cb = _rand(10, T, w), _rand(11, T, w)
    Z = np.full((T, w), -0.8)
    B0 = np.zeros((m, w), np.float32)
    got = oracle_mod.pool_overlap(Ca, Z, Cb, Z, B0, B0, m)
    a = Ca.reshape(T // m, m, w).sum(1)
    b = Cb.reshape(T // m, m, w).sum(1)
    assert np.allclose(got[0], a[0] / m, rtol=1e-14, atol=1e-15)
    assert np.allclose(got[1:], (a[1:] + b[:-1]) / (2 * m), rtol=1e-14, atol=1e-15)


def test_overlap_dominant_bias_selects_one_row(oracle_mod):
    """A bias of +700 on row r of one path picks that row of that path's block
    (block i for path a, block i - 1 for path b)."""
    m, T, w = 4, 24, 5
    Ca, Cb = _rand(20, T, w), _rand(21, T, w)
    Z = np.zeros((T, w))
    Ba = np.zeros((m, w), np.float32)
    Bb = np.zeros((m, w), np.float32)
    Ba[2, 0] = 700.0   # channel 0: row 2 of path a
    Bb[1, 3] = 700.0   # channel 3: row 1 of path b
    got = oracle_mod.pool_overlap(Ca, Z, Cb, Z, Ba, Bb, m)
    n = T // m
    for i in range(n):
        assert got[i, 0] == Ca[m * i + 2, 0]
        if i > 0:
            assert got[i, 3] == Cb[m * (i - 1) + 1, 3]
        else:   # no previous block: channel 3 is the plain mean of block 0 of path a
            assert np.isclose(got[0, 3], Ca[0:m, 3].mean(), rtol=1e-14, atol=1e-15)
    # an unbiased channel mixes all 2m rows equally
    assert np.isclose(got[2, 1], (Ca[8:12, 1].sum() + Cb[4:8, 1].sum()) / 8, rtol=1e-14)


def test_overlap_without_path_b_is_biased_pool(oracle_mod):
    """B^b = -1e30 removes path b everywhere: what remains is the non-overlapping
    pool of (Ca, Za + B^a)."""
    m, T, w = 4, 32, 9
    Ca, Za, Cb, Zb = (_rand(30 + k, T, w, s=2) for k in range(4))
    Ba = _rand(34, m, w).astype(np.float32)
    Bb = np.full((m, w), -1e30, np.float32)
    got = oracle_mod.pool_overlap(Ca, Za, Cb, Zb, Ba, Bb, m)
    ref = oracle_mod.pool(Ca, Za + np.tile(Ba.astype(np.float64), (T // m, 1)), m)
    assert np.allclose(got, ref, rtol=1e-15, atol=1e-15)


def test_overlap_locality(oracle_mod):
    """Changing the tokens of block j changes entries j and j + 1 only."""
    m, d = 4, 64
    T = 6 * m
    H, Wa, Wb, Za, Zb, Ba, Bb = overlap_compressor_inputs(5, T, d, m)
    base = oracle_mod.compress_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m)
    for j in (0, 2, 5):
        H2 = H.copy()
        H2[j * m:(j + 1) * m] = _bits(np.round(_rand(40 + j, m, d) * 4) / 4)
        got = oracle_mod.compress_overlap(H2, Wa, Wb, Za, Zb, Ba, Bb, m)
        changed = [i for i in range(T // m) if not np.array_equal(got[i], base[i])]
        assert changed == [i for i in (j, j + 1) if i < T // m]


def test_compress_overlap_dyadic_paths_exact(oracle_mod):
    """H in {-1,0,1}, W in {-1,0,1}/16, m = 1: the projections are exact.  With
    path b switched off every entry is Ca; with path a switched off entry 0 is
    Ca[0] (its only rows) and entry i > 0 is Cb[i - 1]."""
    rng = np.random.default_rng(7)
    T, d = 12, 128
    H = rng.integers(-1, 2, (T, d))
    Ws = [rng.integers(-1, 2, (d, 512)) for _ in range(4)]
    Ca, Cb = (H @ Ws[0]) / 16.0, (H @ Ws[1]) / 16.0
    bits = [_bits(W / 16.0) for W in Ws]
    zero = np.zeros((1, 512), np.float32)
    off = np.full((1, 512), -1e30, np.float32)
    got = oracle_mod.compress_overlap(_bits(H), *bits, zero, off, 1)
    assert np.array_equal(got, Ca)
    got = oracle_mod.compress_overlap(_bits(H), *bits, off, zero, 1)
    assert np.array_equal(got[0], Ca[0])
    assert np.array_equal(got[1:], Cb[:-1])


def test_project_dyadic_exact(oracle_mod):
    rng = np.random.default_rng(8)
    H = rng.integers(-1, 2, (33, 96))
    W = rng.integers(-3, 4, (96, 512))
    assert np.array_equal(oracle_mod.project(_bits(H), _bits(W / 32.0)), (H @ W) / 32.0)


def test_hca_zero_bias_is_pool(oracle_mod):
    m, T, w = 8, 40, 6
    C, Z = _rand(50, T, w), _rand(51, T, w, s=3)
    got = oracle_mod.pool_bias(C, Z, np.zeros((m, w), np.float32), m)
    assert np.array_equal(got, oracle_mod.pool(C, Z, m))


def test_hca_bias_shifts_scores(oracle_mod):
    m, T, w = 8, 40, 6
    C, Z = _rand(52, T, w), _rand(53, T, w, s=3)
    Bp = _rand(54, m, w, s=2).astype(np.float32)
    got = oracle_mod.pool_bias(C, Z, Bp, m)
    ref = oracle_mod.pool(C, Z + np.tile(Bp.astype(np.float64), (T // m, 1)), m)
    assert np.allclose(got, ref, rtol=1e-15, atol=1e-15)


def test_hca_row_constant_bias_invariant(oracle_mod):
    """A bias that is the same on every row of a channel cancels in the softmax."""
    m, T, w = 16, 64, 5
    C, Z = _rand(55, T, w), _rand(56, T, w, s=2)
    Bp = np.tile(_rand(57, 1, w, s=5).astype(np.float32), (m, 1))
    got = oracle_mod.pool_bias(C, Z, Bp, m)
    assert np.allclose(got, oracle_mod.pool(C, Z, m), rtol=1e-13, atol=1e-14)


def test_hca_dominant_bias_selects_one_row(oracle_mod):
    m, T, w = 128, 256, 3
    C = _rand(58, T, w)
    Z = _rand(59, T, w)
    Bp = np.zeros((m, w), np.float32)
    Bp[77, 1] = 900.0
    got = oracle_mod.pool_bias(C, Z, Bp, m)
    assert got[0, 1] == C[77, 1] and got[1, 1] == C[128 + 77, 1]


def test_compress_hca_m1_is_projection(oracle_mod):
    """m' = 1: each entry is its own token's C = H W_KV, exactly on dyadic data."""
    rng = np.random.default_rng(9)
    H = rng.integers(-1, 2, (10, 64))
    Wkv, Wz = rng.integers(-1, 2, (64, 512)), rng.integers(-1, 2, (64, 512))
    got = oracle_mod.compress_hca(_bits(H), _bits(Wkv / 16.0), _bits(Wz / 16.0),
                                  _rand(60, 1, 512).astype(np.float32), 1)
    assert np.array_equal(got, (H @ Wkv) / 16.0)


def test_compress_hca_matches_numpy_pipeline(oracle_mod):
    """m' = 128 on Gaussian inputs against numpy fp64 (matmul, biased softmax
    along the token axis of each block)."""
    m, T, d = 128, 256, 128
    H, Wkv, Wz, Bp = hca_compressor_inputs(3, T, d, m)
    f = lambda a: synth.bf16_to_f32(a).astype(np.float64)
    C = f(H) @ f(Wkv)
    Z = (f(H) @ f(Wz)).reshape(T // m, m, 512) + Bp.astype(np.float64)
    p = np.exp(Z - Z.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = (p * C.reshape(T // m, m, 512)).sum(1)
    got = oracle_mod.compress_hca(H, Wkv, Wz, Bp, m)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_compressors_reject_ragged(oracle_mod):
    H = np.zeros((6, 64), np.uint16)
    W = np.zeros((64, 512), np.uint16)
    B = np.zeros((4, 512), np.float32)
    with pytest.raises(ValueError):
        oracle_mod.compress_hca(H, W, W, B, 4)
    with pytest.raises(ValueError):
        oracle_mod.compress_overlap(H, W, W, W, W, B, B, 4)


def test_compressors_channels_independent_width_128(oracle_mod):
    """Every output channel pools only its own column: compressing with the first 128
    columns of the weights and biases (V4's indexer-key width c^I) gives the first 128
    channels of the 512-wide result, exactly."""
    m, d = 4, 64
    T = 6 * m
    H, Wa, Wb, Za, Zb, Ba, Bb = overlap_compressor_inputs(6, T, d, m)
    full = oracle_mod.compress_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m)
    cut = lambda a: np.ascontiguousarray(a[:, :128])
    narrow = oracle_mod.compress_overlap(H, cut(Wa), cut(Wb), cut(Za), cut(Zb), cut(Ba), cut(Bb), m)
    assert narrow.shape == (T // m, 128) and np.array_equal(narrow, full[:, :128])
    H2, Wkv, Wz, Bp = hca_compressor_inputs(6, 256, d, 128)
    full = oracle_mod.compress_hca(H2, Wkv, Wz, Bp, 128)
    narrow = oracle_mod.compress_hca(H2, cut(Wkv), cut(Wz), cut(Bp), 128)
    assert np.array_equal(narrow, full[:, :128])
