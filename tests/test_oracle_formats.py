"""Pins of the oracle's element formats (E2M1, E4M3, E8M0) against the format
tables, the round-to-nearest-even rule and an independent library (torch's
float8 dtypes).  None of these checks re-uses the oracle's own code path."""
import numpy as np
import pytest
import torch

from conftest import read_table


def test_e2m1_decode_table(oracle_mod):
    for code, val in read_table("e2m1_table.txt"):
        got = oracle_mod.e2m1_value(int(code))
        assert got == float(val)
        assert np.signbit(got) == np.signbit(float(val))


def test_e2m1_midpoint_decisions(oracle_mod):
    for x, code in read_table("e2m1_rounding.txt"):
        assert oracle_mod.e2m1_encode(float(x)) == int(code), x


def test_e2m1_neighbours_of_midpoints(oracle_mod):
    # just above / below each midpoint the nearest code is unambiguous
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c in range(7):
        mid = np.float32((mags[c] + mags[c + 1]) / 2)
        lo = np.nextafter(mid, np.float32(0))
        hi = np.nextafter(mid, np.float32(100))
        assert oracle_mod.e2m1_encode(float(lo)) == c
        assert oracle_mod.e2m1_encode(float(hi)) == c + 1
        assert oracle_mod.e2m1_encode(float(-lo)) == 8 | c
        assert oracle_mod.e2m1_encode(float(-hi)) == 8 | (c + 1)


def test_e2m1_encode_exhaustive_binades(oracle_mod):
    """Every fp32 in [2^-3, 2^4) (both signs): the code is a nearest magnitude and
    ties (only at the exact midpoints) go to the even code.  Checked with numpy."""
    bits = np.arange(0x3E000000, 0x41800000, dtype=np.uint32)  # [0.125, 16)
    x = bits.view(np.float32)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    codes = oracle_mod.e2m1_encode_array(x)
    assert np.all(codes < 8)
    err = np.abs(x.astype(np.float64) - mags[codes])
    best = np.min(np.abs(x.astype(np.float64)[:, None] - mags[None, :]), axis=1) \
        if x.size < 10 else None
    # nearest: compare with both neighbours of the chosen code
    up = np.minimum(codes + 1, 7)
    dn = np.maximum(codes.astype(np.int64) - 1, 0)
    assert np.all(err <= np.abs(x - mags[up]))
    assert np.all(err <= np.abs(x - mags[dn]))
    tie = (err == np.abs(x - mags[up])) & (up != codes)
    assert np.all(codes[tie] % 2 == 0)
    tie = (err == np.abs(x - mags[dn])) & (dn != codes)
    assert np.all(codes[tie] % 2 == 0)
    assert np.all(np.diff(codes.astype(np.int64)) >= 0)  # monotone
    neg = oracle_mod.e2m1_encode_array(-x)
    assert np.array_equal(neg, codes | 8)
    del best


def test_e2m1_small_and_large(oracle_mod):
    tiny = np.array([1e-30, 1e-8, 0.0, 0.2499], np.float32)
    assert np.all(oracle_mod.e2m1_encode_array(tiny) == 0)
    assert np.all(oracle_mod.e2m1_encode_array(-tiny) == 8)
    big = np.array([6.0, 7.0, 1e9, 3e38], np.float32)
    assert np.all(oracle_mod.e2m1_encode_array(big) == 7)


def test_e4m3_decode_matches_torch(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_value(b) for b in range(256)])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_rne(oracle_mod):
    """Against torch's fp32->float8_e4m3fn cast (round-to-nearest-even) on a dense
    strided sweep of fp32 in [2^-12, 448] and on every exact midpoint."""
    lo, hi = np.float32(2.0 ** -12).view(np.uint32), np.float32(448.0).view(np.uint32)
    x = np.arange(lo, hi + 1, 3, dtype=np.uint32).view(np.float32)
    vals = np.array([oracle_mod.e4m3_value(b) for b in range(127)])
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -x[:1000], np.array([0.0, -0.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle_mod.e4m3_encode_array(x)
    assert np.array_equal(ref, got)


def test_e4m3_saturates(oracle_mod):
    x = np.array([448.0, 460.0, 464.0, 480.0, 1e6, -1e6], np.float32)
    got = oracle_mod.e4m3_encode_array(x)
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]


def test_e8m0_matches_torch(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([oracle_mod.e8m0_value(b) for b in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(ref[:255], got[:255])


def test_fp4_range_pin(oracle_mod):
    # largest magnitude of E2M1 x E4M3 without a second-level scale: 448 * 6 = 2688
    from conftest import read_table as rt

    tab = {k: v for k, v in rt("bytes_per_token.txt")}
    assert oracle_mod.e4m3_value(0x7E) * oracle_mod.e2m1_value(7) == float(tab["fp4_max_magnitude"])
    assert abs(np.sqrt(512) - float(tab["latent_norm_bound"])) < 0.05


def _all_fp32_chunks(bits_per_chunk=17):
    n = 1 << bits_per_chunk
    for c in range(1 << (32 - bits_per_chunk)):
        yield (np.uint32(c) << np.uint32(bits_per_chunk)) | np.arange(n, dtype=np.uint32)


def test_e2m1_encode_all_fp32(oracle_mod):
    """Every fp32 bit pattern but the NaNs: the code's sign bit is the input's (a value
    that rounds to zero keeps its sign), its magnitude is the nearest E2M1 magnitude with
    ties to the even code, and everything beyond 6 (infinities too) saturates to 6."""
    from concurrent.futures import ThreadPoolExecutor

    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])

    def check(bits):
        x = bits.view(np.float32)
        x = x[~np.isnan(x)]
        codes = oracle_mod.e2m1_encode_array(x)
        if not np.array_equal(codes >> 3, np.signbit(x).astype(np.uint8)):
            return "sign"
        a = np.abs(x.astype(np.float64))
        c = (codes & 7).astype(np.int64)
        if not np.all(c[a >= 6.0] == 7):
            return "saturation"
        f = a < 6.0
        a, c = a[f], c[f]
        err = np.abs(a - mags[c])
        up, dn = np.minimum(c + 1, 7), np.maximum(c - 1, 0)
        eu, ed = np.abs(a - mags[up]), np.abs(a - mags[dn])
        if not (np.all(err <= eu) and np.all(err <= ed)):
            return "nearest"
        if not (np.all(c[(err == eu) & (up != c)] % 2 == 0) and np.all(c[(err == ed) & (dn != c)] % 2 == 0)):
            return "ties"
        return None

    with ThreadPoolExecutor(8) as ex:
        fails = [r for r in ex.map(check, _all_fp32_chunks()) if r]
    assert not fails, fails[:4]


def test_e4m3_encode_all_fp32(oracle_mod):
    """Every fp32 bit pattern but the NaNs: equal to torch's fp32 -> float8_e4m3fn cast
    (round to nearest even) wherever that cast is finite (|x| <= 464, where 464 rounds to
    448), and saturated to +-448 (bytes 0x7E / 0xFE) beyond it, infinities included."""
    from concurrent.futures import ThreadPoolExecutor

    def check(bits):
        x = bits.view(np.float32)
        x = x[~np.isnan(x)]
        got = oracle_mod.e4m3_encode_array(x)
        small = np.abs(x) <= 464.0
        ref = torch.from_numpy(x[small]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        if not np.array_equal(got[small], ref):
            return "rounding"
        big = ~small
        if not np.array_equal(got[big], np.where(np.signbit(x[big]), 0xFE, 0x7E).astype(np.uint8)):
            return "saturation"
        return None

    with ThreadPoolExecutor(8) as ex:
        fails = [r for r in ex.map(check, _all_fp32_chunks()) if r]
    assert not fails, fails[:4]
