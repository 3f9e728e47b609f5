"""Device codec == oracle codec, bit for bit, on identical fp32 inputs; device
generator == host generator."""
import numpy as np
import pytest

from gpu_common import csa2, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu

E2M1_MID = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _e4m3_vals():
    return torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()


def adversarial_main(rng, n):
    """Groups whose scale and elements sit exactly on rounding decision points."""
    x = rng.standard_normal((n, 512)).astype(np.float32)
    g = x.reshape(n, 32, 16)
    vals = _e4m3_vals()
    for r in range(n):
        for j in range(32):
            kind = (r * 32 + j) % 6
            if kind == 0:  # element ties at every E2M1 midpoint for a random scale
                s = vals[rng.integers(1, 127)]
                g[r, j, :7] = s * E2M1_MID * np.where(rng.random(7) < 0.5, -1, 1)
                g[r, j, 7] = 6 * s
                g[r, j, 8:] = s * rng.choice(E2M1_MID, 8)
            elif kind == 1:  # amax/6 exactly on an E4M3 midpoint
                c = rng.integers(0, 125)
                mid = np.float32((vals[c] + vals[c + 1]) / 2)
                g[r, j] *= 0.1
                g[r, j, rng.integers(16)] = 6 * mid
            elif kind == 2:
                g[r, j] = 0.0
            elif kind == 3:
                g[r, j] *= np.float32(1e-6)  # scales underflow to 0 / subnormal E4M3
                g[r, j, 0] = -1e-30
            elif kind == 4:
                g[r, j] *= np.float32(2000.0)  # saturating scales (amax/6 > 448)
    return x


def adversarial_index(rng, n):
    x = rng.standard_normal((n, 128)).astype(np.float32)
    g = x.reshape(n, 4, 32)
    for r in range(n):
        for j in range(4):
            kind = (r * 4 + j) % 6
            e = int(rng.integers(-20, 20))
            if kind == 0:  # amax exactly a power of two, elements on midpoints
                X = np.float32(2.0 ** (e - 2))
                g[r, j, :7] = X * E2M1_MID
                g[r, j, 7] = np.float32(2.0 ** e)
                g[r, j, 8:] = X * rng.choice(E2M1_MID, 24) * np.where(rng.random(24) < .5, -1, 1)
            elif kind == 1:
                g[r, j] = 0.0
            elif kind == 2:
                g[r, j] *= np.float32(1e-39)  # subnormal amax
            elif kind == 3:
                g[r, j] *= np.float32(1e37)
            elif kind == 4:
                g[r, j, 5] = -np.float32(7.9) * np.float32(2.0 ** e)  # clips to 6 X
    return x


def _run_codec(x_main, x_idx):
    n = max(x_main.shape[0], x_idx.shape[0])
    # both inputs must hold n rows: the entry point reads n rows of each
    x_main = np.concatenate([x_main, np.zeros((n - x_main.shape[0], 512), np.float32)])
    x_idx = np.concatenate([x_idx, np.zeros((n - x_idx.shape[0], 128), np.float32)])
    P = csa2.Planes.empty(1, n)
    csa2.quantize_entries(P, to_dev(x_main), to_dev(x_idx), n, 0)
    torch.cuda.synchronize()
    return (P.kv_codes.cpu().numpy(), P.kv_scales.cpu().numpy(), P.ix_codes.cpu().numpy(),
            P.ix_scales.cpu().numpy())


@pytest.mark.parametrize("kind", ["random", "adversarial"])
def test_codec_bit_exact(oracle_mod, kind):
    rng = np.random.default_rng(11)
    n = 4096
    if kind == "random":
        xm = (rng.standard_normal((n, 512)) * np.exp(rng.uniform(-8, 8, (n, 1)))).astype(np.float32)
        xi = (rng.standard_normal((n, 128)) * np.exp(rng.uniform(-8, 8, (n, 1)))).astype(np.float32)
    else:
        xm, xi = adversarial_main(rng, n), adversarial_index(rng, n)
    kvc, kvs, ixc, ixs = _run_codec(xm, xi)
    okvc, okvs = oracle_mod.quantize_main(xm)
    oixc, oixs = oracle_mod.quantize_index(xi)
    assert np.array_equal(kvs, okvs), np.argwhere(kvs != okvs)[:5]
    assert np.array_equal(kvc, okvc), np.argwhere(kvc != okvc)[:5]
    assert np.array_equal(ixs, oixs), np.argwhere(ixs != oixs)[:5]
    assert np.array_equal(ixc, oixc), np.argwhere(ixc != oixc)[:5]


def test_codec_all_e2m1_inputs(oracle_mod):
    """Every fp32 bit pattern in [2^-3, 2^4) of both signs through the main quantizer
    with scale 1 (a 6.0 in every group pins the scale byte to 0x38)."""
    bits = np.arange(0x3E000000, 0x41800000, 64, dtype=np.uint32)
    x = bits.view(np.float32)
    x = np.concatenate([x, -x])
    n_groups = -(-x.size // 15)
    pad = np.zeros(n_groups * 15, np.float32)
    pad[:x.size] = x
    g = np.concatenate([pad.reshape(n_groups, 15), np.full((n_groups, 1), 6.0, np.float32)], 1)
    n = -(-n_groups // 32)
    full = np.zeros((n * 32, 16), np.float32)
    full[:n_groups] = g
    xm = full.reshape(n, 512)
    kvc, kvs, _, _ = _run_codec(xm, np.zeros((1, 128), np.float32))
    okvc, okvs = oracle_mod.quantize_main(xm)
    assert np.array_equal(kvs[:n], okvs) and np.array_equal(kvc[:n], okvc)


def test_device_generator_matches_host():
    import synth

    n = 100003
    st = torch.cuda.current_stream().cuda_stream
    for fn_h, fn_d, dt in [(synth.normal_f32, synth.dev_normal_f32, torch.float32),
                           (synth.uniform_f32, synth.dev_uniform_f32, torch.float32)]:
        t = torch.empty(n, dtype=dt, device="cuda")
        fn_d(5, 17, n, t.data_ptr(), st, offset=12345)
        assert np.array_equal(t.cpu().numpy(), fn_h(5, 17, n, offset=12345))
    t = torch.empty(n, dtype=torch.int16, device="cuda")
    synth.dev_normal_bf16(5, 18, n, t.data_ptr(), st, scale=0.25)
    assert np.array_equal(t.cpu().numpy().view(np.uint16), synth.normal_bf16(5, 18, n, scale=0.25))
    t = torch.empty(n, dtype=torch.uint8, device="cuda")
    synth.dev_e4m3_normal(5, 19, n, t.data_ptr(), st)
    assert np.array_equal(t.cpu().numpy(), synth.e4m3_normal(5, 19, n))
    hv = np.linspace(-1, 1, 128).astype(np.float32)
    t = torch.empty(n * 128 // 128 * 128, dtype=torch.float32, device="cuda")
    hvd = to_dev(hv)
    synth.dev_keys_f32(5, 20, 21, t.numel(), 128, t.data_ptr(), st, offset=256, hot_prob=0.3,
                       hotvec_ptr=hvd.data_ptr())
    assert np.array_equal(t.cpu().numpy(),
                          synth.keys_f32(5, 20, 21, t.numel(), 128, offset=256, hot_prob=0.3,
                                         hotvec=hv))


def test_codec_division_exhaustive():
    """The main-KV codec divides each value by its group's E4M3 scale with an FMA-corrected
    reciprocal product; for every positive E4M3 scale and every fp32 significand of x with
    x / s in [2^-5, 2^7) it must equal the correctly rounded division bit for bit."""
    ws = csa2.workspace(512)
    bad, n = csa2.selftest_codec_division(ws)
    assert n == 126 * (1 << 23) * 12
    assert bad == 0, bad


def _oracle_sweep_sums(oracle_mod, nchunks=4096, bits_per_chunk=20):
    """The oracle's E2M1 codes and E4M3 bytes of every non-NaN fp32 bit pattern, summed per
    chunk of 2^20 patterns with weight 2 i + 1 (mod 2^64), i the pattern's index in its chunk."""
    from concurrent.futures import ThreadPoolExecutor

    n = 1 << bits_per_chunk
    wgt = 2 * np.arange(n, dtype=np.uint64) + np.uint64(1)

    def one(c):
        bits = (np.uint32(c) << np.uint32(bits_per_chunk)) | np.arange(n, dtype=np.uint32)
        x = bits.view(np.float32)
        ok = ~np.isnan(x)
        e2 = oracle_mod.e2m1_encode_array(np.where(ok, x, 0.0)).astype(np.uint64) * ok
        e4 = oracle_mod.e4m3_encode_array(np.where(ok, x, 0.0)).astype(np.uint64) * ok
        return c, (e2 * wgt).sum(dtype=np.uint64), (e4 * wgt).sum(dtype=np.uint64)

    out = np.zeros((nchunks, 2), np.uint64)
    with ThreadPoolExecutor(16) as ex:
        for c, s2, s4 in ex.map(one, range(nchunks)):
            out[c] = (s2, s4)
    return out


def test_element_encoders_all_fp32(oracle_mod):
    """The codec's fp32 -> E2M1 and fp32 -> E4M3 conversions equal the oracle's encoders on
    every one of the 2^32 fp32 bit patterns but the NaNs (both signs, zeros, subnormals,
    values beyond the saturation points, infinities): per chunk of 2^20 patterns, weighted
    sums of the codes agree, so a single differing code would show in its chunk."""
    ws = csa2.workspace(256 + 16 * 4096)
    gpu = csa2.selftest_encode_sweep(ws)
    ref = _oracle_sweep_sums(oracle_mod)
    bad = np.nonzero((gpu != ref).any(axis=1))[0]
    assert bad.size == 0, f"chunks {bad[:8]} differ (chunk c holds bit patterns c << 20 ..)"
