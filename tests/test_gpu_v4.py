"""The V4 compressors (csa2_compress_overlap, csa2_compress_hca) and the HCA
dense attention (csa2_dense_attn_decode) against the oracle.

Compressors.  Dyadic inputs make every projection exact, so with one path
switched off by a -1e30 bias (m = 1) the outputs must equal the oracle's bit
for bit.  On Gaussian inputs each output is checked against a bound built from
the arithmetic: C and Z are d-term sums of exact bf16 x bf16 products in fp32,
within KAPPA * u * sum_k |h_k w_k| of exact (u = 2^-24; KAPPA = 32 as for the
cache write); the pooled value sum_i p_i C_i then moves by at most
max_i eps_C,i + max_i eps_Z,i * sum_i p_i |C_i - Cbar| (first order in the
score errors: dp_i = p_i (dz_i - sum_j p_j dz_j)) plus the fp32 exp / sum /
divide, bounded by 16 u * sum_i p_i |C_i| + 16 u |Cbar| (2m terms of relative
error a few u each, 16 covering m up to 128 with the sums' depth).

Dense attention.  Same kernel as the sparse path reading entries 0 ..
n_entries[b] - 1 instead of an index list: bit-identical to csa2_sparse_attn_decode
given topk[b] = 0, 1, .., n_entries[b] - 1, and within the attention tolerance of
the oracle's attention over those entries."""
import numpy as np
import pytest

from gpu_common import SmallCache, csa2, require_gpu, to_dev, torch
from parity import check_attention
from synth import workloads as W

pytestmark = pytest.mark.gpu
U = 2.0 ** -24
KAPPA = 32.0
SCALE = 1.0 / np.sqrt(512.0)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _bits(x):
    b = np.asarray(x, np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0)
    return (b >> 16).astype(np.uint16)


def _f64(bf16):
    return (np.asarray(bf16).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _dev16(a):
    return to_dev(np.ascontiguousarray(a).view(np.int16))


def _gpu_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m):
    T, d = H.shape
    width = Wa.shape[1]
    out = torch.full((T // m, width), float("nan"), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.compress_workspace_size(T, d))
    csa2.compress_overlap(_dev16(H), T, d, _dev16(Wa), _dev16(Wb), _dev16(Za), _dev16(Zb),
                          to_dev(np.ascontiguousarray(Ba, np.float32)),
                          to_dev(np.ascontiguousarray(Bb, np.float32)), m, out, ws, width=width)
    assert csa2.check(ws)[0] == 0
    return out.cpu().numpy().astype(np.float64)


def _gpu_hca(H, Wkv, Wz, Bp, m):
    T, d = H.shape
    width = Wkv.shape[1]
    out = torch.full((T // m, width), float("nan"), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.compress_workspace_size(T, d))
    csa2.compress_hca(_dev16(H), T, d, _dev16(Wkv), _dev16(Wz), to_dev(np.ascontiguousarray(Bp, np.float32)),
                      m, out, ws, width=width)
    assert csa2.check(ws)[0] == 0
    return out.cpu().numpy().astype(np.float64)


def _pool_bound(parts, m):
    """parts: list of (C, Z + bias, eps_C, eps_Z) arrays [n_rows_of_entry][512] per entry,
    given as lists over entries.  Returns the per-entry, per-channel bound."""
    out = []
    for rows in parts:
        C, Z, eC, eZ = (np.concatenate([r[i] for r in rows]) for i in range(4))
        p = np.exp(Z - Z.max(0))
        p /= p.sum(0)
        cbar = (p * C).sum(0)
        out.append(eC.max(0) + eZ.max(0) * (p * np.abs(C - cbar)).sum(0)
                   + 16 * U * ((p * np.abs(C)).sum(0) + np.abs(cbar)))
    return np.stack(out)


def _proj_parts(oracle_mod, H, Wc, Wz):
    C = oracle_mod.project(H, Wc)
    Z = oracle_mod.project(H, Wz)
    aH = np.abs(_f64(H))
    eC = KAPPA * U * (aH @ np.abs(_f64(Wc)))
    eZ = KAPPA * U * (aH @ np.abs(_f64(Wz)))
    return C, Z, eC, eZ


@pytest.mark.parametrize("m", [1, 4])
def test_overlap_dyadic_paths_exact(oracle_mod, m):
    """H in {-1,0,1}, W in {-1,0,1}/16: exact projections.  One path switched off by a
    -1e30 bias leaves, at m = 1, one row per entry; at m = 4 (W_aZ = 0, path b off)
    the plain mean of m exact values, divided by 4 exactly: bit-equal outputs."""
    rng = np.random.default_rng(m)
    T, d = 8 * m + 128, 256
    H = _bits(rng.integers(-1, 2, (T, d)))
    Ws = [_bits(rng.integers(-1, 2, (d, 512)) / 16.0) for _ in range(4)]
    if m > 1:
        Ws[2] = np.zeros_like(Ws[2])
    zero = np.zeros((m, 512), np.float32)
    off = np.full((m, 512), -1e30, np.float32)
    cases = [(zero, off)] + ([(off, zero)] if m == 1 else [])
    for Ba, Bb in cases:
        got = _gpu_overlap(H, *Ws, Ba, Bb, m)
        ref = oracle_mod.compress_overlap(H, *Ws, Ba, Bb, m)
        assert np.array_equal(got, ref)


def test_hca_dyadic_m1_exact(oracle_mod):
    rng = np.random.default_rng(11)
    T, d = 200, 192
    H = _bits(rng.integers(-1, 2, (T, d)))
    Wkv, Wz = (_bits(rng.integers(-1, 2, (d, 512)) / 16.0) for _ in range(2))
    Bp = (rng.standard_normal((1, 512))).astype(np.float32)
    assert np.array_equal(_gpu_hca(H, Wkv, Wz, Bp, 1), oracle_mod.compress_hca(H, Wkv, Wz, Bp, 1))


def _overlap_bound(oracle_mod, H, Wa, Wb, Za, Zb, Ba, Bb, m):
    T = H.shape[0]
    Ca, ZA, eCa, eZa = _proj_parts(oracle_mod, H, Wa, Za)
    Cb, ZB, eCb, eZb = _proj_parts(oracle_mod, H, Wb, Zb)
    ba, bb = Ba.astype(np.float64), Bb.astype(np.float64)
    parts = []
    for i in range(T // m):
        a = slice(i * m, (i + 1) * m)
        rows = [(Ca[a], ZA[a] + ba, eCa[a], eZa[a])]
        if i > 0:
            b = slice((i - 1) * m, i * m)
            rows.append((Cb[b], ZB[b] + bb, eCb[b], eZb[b]))
        parts.append(rows)
    return _pool_bound(parts, m)


def _hca_bound(oracle_mod, H, Wkv, Wz, Bp, m):
    T = H.shape[0]
    C, Z, eC, eZ = _proj_parts(oracle_mod, H, Wkv, Wz)
    bp = Bp.astype(np.float64)
    parts = [[(C[i * m:(i + 1) * m], Z[i * m:(i + 1) * m] + bp, eC[i * m:(i + 1) * m], eZ[i * m:(i + 1) * m])]
             for i in range(T // m)]
    return _pool_bound(parts, m)


@pytest.mark.parametrize("T,d,m", [(512, 256, 4), (200, 512, 4), (264, 320, 2)])
def test_overlap_gaussian_within_bound(oracle_mod, T, d, m):
    """Several GEMM tiles, a ragged last tile (T = 200, 264) and an m = 2 variant."""
    H, Wa, Wb, Za, Zb, Ba, Bb = W.overlap_compressor_inputs(21, T, d, m)
    got = _gpu_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m)
    ref = oracle_mod.compress_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m)
    bound = _overlap_bound(oracle_mod, H, Wa, Wb, Za, Zb, Ba, Bb, m)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("T,d,m", [(384, 512, 128), (256, 256, 64), (96, 128, 8)])
def test_hca_gaussian_within_bound(oracle_mod, T, d, m):
    H, Wkv, Wz, Bp = W.hca_compressor_inputs(22, T, d, m)
    got = _gpu_hca(H, Wkv, Wz, Bp, m)
    ref = oracle_mod.compress_hca(H, Wkv, Wz, Bp, m)
    bound = _hca_bound(oracle_mod, H, Wkv, Wz, Bp, m)
    err = np.abs(got - ref)
    assert np.all(err <= bound), float((err / bound).max())


@pytest.mark.parametrize("width", [128, 256])
def test_narrow_widths_within_bound(oracle_mod, width):
    """V4's indexer keys go through the same compression at c^I = 128 channels (CSA step 2):
    the compressors at widths 128 and 256 against the oracle, within the same bound."""
    cut = lambda a: np.ascontiguousarray(a[:, :width])
    T, d, m = 200, 256, 4
    H, Wa, Wb, Za, Zb, Ba, Bb = W.overlap_compressor_inputs(23, T, d, m)
    Wa, Wb, Za, Zb, Ba, Bb = (cut(a) for a in (Wa, Wb, Za, Zb, Ba, Bb))
    got = _gpu_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m)
    ref = oracle_mod.compress_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m)
    assert got.shape == (T // m, width)
    assert np.all(np.abs(got - ref) <= _overlap_bound(oracle_mod, H, Wa, Wb, Za, Zb, Ba, Bb, m))
    T, m = 256, 128
    H, Wkv, Wz, Bp = W.hca_compressor_inputs(23, T, d, m)
    Wkv, Wz, Bp = cut(Wkv), cut(Wz), cut(Bp)
    got = _gpu_hca(H, Wkv, Wz, Bp, m)
    ref = oracle_mod.compress_hca(H, Wkv, Wz, Bp, m)
    assert np.all(np.abs(got - ref) <= _hca_bound(oracle_mod, H, Wkv, Wz, Bp, m))


def test_compressors_empty():
    H = torch.zeros((0, 64), dtype=torch.int16, device="cuda")
    Wt = torch.zeros((64, 512), dtype=torch.int16, device="cuda")
    B = torch.zeros((4, 512), dtype=torch.float32, device="cuda")
    out = torch.zeros((1, 512), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.compress_workspace_size(0, 64))
    csa2.compress_overlap(H, 0, 64, Wt, Wt, Wt, Wt, B, B, 4, out, ws)
    csa2.compress_hca(H, 0, 64, Wt, Wt, B, 4, out, ws)
    torch.cuda.synchronize()
    assert csa2.check(ws)[0] == 0 and torch.all(out == 0)


@pytest.mark.parametrize("width", [512, 128])
def test_overlap_full_size_sampled(oracle_mod, width):
    """The benchmarked prefill chunk (T = 65,536 tokens, d = 4096, m = 4): sampled
    entries against the oracle run on the two blocks each one reads; at the main-KV
    width and at V4's indexer-key width c^I = 128 (one channel block per token tile)."""
    T, d, m = 65536, 4096, 4
    H, Wa, Wb, Za, Zb, Ba, Bb = W.overlap_compressor_inputs(7, T, d, m)
    cut = lambda a: np.ascontiguousarray(a[:, :width])
    Wa, Wb, Za, Zb, Ba, Bb = (cut(a) for a in (Wa, Wb, Za, Zb, Ba, Bb))
    got = _gpu_overlap(H, Wa, Wb, Za, Zb, Ba, Bb, m)
    assert got.shape == (T // m, width)
    rng = np.random.default_rng(5)
    for i in [0, 1, T // m - 1] + [int(v) for v in rng.integers(2, T // m - 1, 13)]:
        Hs = H[max(0, (i - 1) * m):(i + 1) * m]  # the blocks entry i reads: it is the slice's last
        ref = oracle_mod.compress_overlap(Hs, Wa, Wb, Za, Zb, Ba, Bb, m)[-1]
        bound = _overlap_bound(oracle_mod, Hs, Wa, Wb, Za, Zb, Ba, Bb, m)[-1]
        assert np.all(np.abs(got[i] - ref) <= bound), i


def test_hca_full_size_sampled(oracle_mod):
    """HCA at m' = 128 on a 65,536-token chunk, d = 4096: sampled entries."""
    T, d, m = 65536, 4096, 128
    H, Wkv, Wz, Bp = W.hca_compressor_inputs(7, T, d, m)
    got = _gpu_hca(H, Wkv, Wz, Bp, m)
    for i in (0, 77, 311, T // m - 1):
        Hs = H[i * m:(i + 1) * m]
        ref = oracle_mod.compress_hca(Hs, Wkv, Wz, Bp, m)[0]
        bound = _hca_bound(oracle_mod, Hs, Wkv, Wz, Bp, m)[0]
        assert np.all(np.abs(got[i] - ref) <= bound), i


# ----------------------------------------------------------------------------- dense attention

def _dense(c, n_entries, n_max, swa, q, n_swa, **kw):
    B = len(n_entries)
    out = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.dense_attn_workspace_size(B, n_max, n_swa))
    swa_c = np.ascontiguousarray(swa[:, :n_swa])
    csa2.dense_attn_decode(c.planes, B, to_dev(np.asarray(n_entries, np.int32)), n_max,
                           to_dev(swa_c) if n_swa else None, n_swa, to_dev(q.view(np.int16)), SCALE, out, ws,
                           lse_out=lse, **kw)
    st, _ = csa2.check(ws)
    assert st == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def _sparse(c, topk, swa, q, n_swa, **kw):
    B, k = topk.shape
    out = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.sparse_attn_workspace_size(B, k, n_swa))
    swa_c = np.ascontiguousarray(swa[:, :n_swa])
    csa2.sparse_attn_decode(c.planes, B, to_dev(topk.astype(np.int32)), k, to_dev(swa_c) if n_swa else None,
                            n_swa, to_dev(q.view(np.int16)), SCALE, out, ws, lse_out=lse, **kw)
    assert csa2.check(ws)[0] == 0
    return out.cpu().numpy(), lse.cpu().numpy()


def _arange_topk(n_entries, n_max):
    t = np.full((len(n_entries), n_max), -1, np.int32)
    for b, n in enumerate(n_entries):
        t[b, :max(0, min(n, n_max))] = np.arange(max(0, min(n, n_max)))
    return t


def test_dense_attention_matches_oracle_and_sparse(oracle_mod):
    c = SmallCache(oracle_mod, 7, 3, 2048, stride=2112)
    n_entries, n_max = [2048, 777, 5], 2048  # the sparse path's top-k limit
    q = W.attn_query(7, 0, 3)
    swa = W.swa_rows(7, 0, 3, 128)
    out, lse = _dense(c, n_entries, n_max, swa, q, 128)
    topk = _arange_topk(n_entries, n_max)
    sout, slse = _sparse(c, topk, swa, q, 128)
    assert np.array_equal(out, sout) and np.array_equal(lse, slse)
    for b in range(3):
        kvc, kvs, _, _ = c.oracle_slot(b)
        ro, rl = oracle_mod.attention(kvc, kvs, topk[b], swa[b], q[b], SCALE)
        check_attention(out[b:b + 1], ro[None])
        assert np.allclose(lse[b], rl, rtol=1e-4, atol=1e-4)


def test_dense_attention_beyond_topk_limit(oracle_mod):
    """HCA at a 1M context sees 8,192 entries (more than the sparse path's top-k
    limit); n_entries above n_max count as n_max, negative as none."""
    c = SmallCache(oracle_mod, 8, 2, 8192)
    n_entries, n_max = [9000, -3], 8192
    q = W.attn_query(8, 0, 2)
    swa = W.swa_rows(8, 0, 2, 128)
    out, lse = _dense(c, n_entries, n_max, swa, q, 64)
    topk = _arange_topk(n_entries, n_max)
    for b in range(2):
        kvc, kvs, _, _ = c.oracle_slot(b)
        ro, rl = oracle_mod.attention(kvc, kvs, topk[b], swa[b][:64], q[b], SCALE)
        check_attention(out[b:b + 1], ro[None])
        assert np.allclose(lse[b], rl, rtol=1e-4, atol=1e-4)


def test_dense_attention_full_size_sampled(oracle_mod):
    """The benchmarked HCA launch: batch 32, every one of 8,192 entries + 128 window
    rows (4 CTAs per query and the merge); sampled queries against the oracle."""
    B, N = 32, 8192
    c = SmallCache(oracle_mod, 10, B, N)
    q = W.attn_query(10, 0, B)
    swa = W.swa_rows(10, 0, B, 128)
    out, lse = _dense(c, [N] * B, N, swa, q, 128)
    topk = _arange_topk([N], N)[0]
    for b in (0, 13, 31):
        kvc, kvs, _, _ = c.oracle_slot(b)
        ro, rl = oracle_mod.attention(kvc, kvs, topk, swa[b], q[b], SCALE)
        check_attention(out[b:b + 1], ro[None])
        assert np.allclose(lse[b], rl, rtol=1e-4, atol=1e-4)


def test_dense_attention_extras_and_empty(oracle_mod):
    c = SmallCache(oracle_mod, 9, 2, 600)
    q = W.attn_query(9, 0, 2)
    swa = W.swa_rows(9, 0, 2, 128)
    rng = np.random.default_rng(9)
    w = (1.0 + 0.3 * rng.standard_normal(512)).astype(np.float32)
    nr = csa2.norm_rope(to_dev(w), 1e-6, True, 10000.0)
    pos = to_dev(np.array([4097, 123456], np.int64))
    sink = to_dev((2.0 * rng.standard_normal(64)).astype(np.float32))
    kw = dict(q_nr=nr, q_pos=pos, sink=sink)
    out, lse = _dense(c, [600, 311], 600, swa, q, 100, **kw)
    sout, slse = _sparse(c, _arange_topk([600, 311], 600), swa, q, 100, **kw)
    assert np.array_equal(out, sout) and np.array_equal(lse, slse)
    out, lse = _dense(c, [0, 0], 0, swa, q, 0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))
