"""csa2_cache_write against the oracle: 100% identical bytes on dyadic inputs
(every sum exact), and banded identity on Gaussian inputs at m = 2."""
import numpy as np
import pytest

from gpu_common import csa2, require_gpu, to_dev, torch
from synth import workloads as W

pytestmark = pytest.mark.gpu
DELTA = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _bits(x):
    b = np.asarray(x, np.float32).view(np.uint32)
    assert np.all(b & 0xFFFF == 0)
    return (b >> 16).astype(np.uint16)


def _gpu_write(H, Wkv, Wz, Wik, m, seq=1, offset=5, stride=None):
    T, d = H.shape
    n = T // m
    stride = stride or (offset + n + 3)
    P = csa2.Planes.empty(seq + 1, stride)
    for t in (P.kv_codes, P.kv_scales, P.ix_codes, P.ix_scales):
        t.fill_(0xA5)
    ws = csa2.workspace(csa2.cache_write_workspace_size(T, m))
    csa2.cache_write(to_dev(H.view(np.int16)), T, d, to_dev(Wkv.view(np.int16)),
                     to_dev(Wz.view(np.int16)), to_dev(Wik.view(np.int16)), m, P, seq, offset, ws)
    assert csa2.check(ws)[0] == 0
    e0 = seq * stride + offset
    out = [t[e0:e0 + n].cpu().numpy() for t in (P.kv_codes, P.kv_scales, P.ix_codes, P.ix_scales)]
    # nothing outside the written range changed
    untouched = P.kv_scales.cpu().numpy()
    assert np.all(untouched[:e0] == 0xA5) and np.all(untouched[e0 + n:] == 0xA5)
    return out


@pytest.mark.parametrize("T,d", [(128, 256), (200, 512)])
def test_dyadic_bytes_exact(oracle_mod, T, d):
    rng = np.random.default_rng(T)
    H = _bits(rng.integers(-1, 2, (T, d)).astype(np.float32))
    Wkv = _bits(rng.integers(-1, 2, (d, 512)) / 16.0)
    Wz = _bits(rng.integers(-1, 2, (d, 512)) / 16.0)
    Wik = _bits(rng.integers(-1, 2, (512, 128)) / 16.0)
    got = _gpu_write(H, Wkv, Wz, Wik, 1)
    ref = oracle_mod.cache_write(H, Wkv, Wz, Wik, 1)
    for g, r, name in zip(got, ref, ("kv_codes", "kv_scales", "ix_codes", "ix_scales")):
        assert np.array_equal(g, r), name


def _group_bytes_ok(got_codes, got_scales, ref_codes, ref_scales, margins, group_bytes):
    """Groups far from a decision point must match exactly; returns (#exact-checked, #banded)."""
    n, ng = ref_scales.shape
    gc = got_codes.reshape(n, ng, group_bytes)
    rc = ref_codes.reshape(n, ng, group_bytes)
    far = margins.reshape(n, ng) > DELTA
    same = (gc == rc).all(-1) & (got_scales == ref_scales)
    bad = far & ~same
    assert not bad.any(), f"{bad.sum()} far-from-boundary groups differ, first {np.argwhere(bad)[:3]}"
    near = ~far
    # groups inside the band: the scale byte may move by at most one code
    ds = np.abs(got_scales.astype(int) - ref_scales.astype(int))
    assert np.all(ds[near] <= 1)
    return int(far.sum()), int(near.sum())


def test_gaussian_m2_banded(oracle_mod):
    T, d = 512, 5120
    H, Wkv, Wz, Wik = W.cache_write_inputs(3, T, d)
    got = _gpu_write(H, Wkv, Wz, Wik, 2)
    kvc, kvs, ixc, ixs, cb, ki = oracle_mod.cache_write(H, Wkv, Wz, Wik, 2, return_prequant=True)
    mm = oracle_mod.main_group_margins(cb.astype(np.float32).astype(np.float64))
    mi = oracle_mod.index_group_margins(ki.astype(np.float32).astype(np.float64))
    f1, b1 = _group_bytes_ok(got[0], got[1], kvc, kvs, mm, 8)
    f2, b2 = _group_bytes_ok(got[2], got[3], ixc, ixs, mi, 16)
    assert f1 > 0.99 * (f1 + b1) and f2 > 0.99 * (f2 + b2)
