"""csa2_index_topk_noalloc: the indexer entry point for callers that cannot
allocate device memory (plugins handed only their buffers, serving loops with
no allocator on the hot path).  It keeps its scratch in a fixed device array
inside the library; its results must equal those of csa2_index_topk, call after
call, even though every call reuses the same array.

This file is collected last so that, if it fails, a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import compressed_sparse_attention_nvfp4_gb300 as csa2
from synth import workloads as W


def test_rejects_requests_beyond_the_scratch_limit():
    """Host-side check: a request needing more than the fixed scratch returns
    CSA2_ERR_WORKSPACE before anything is launched (no GPU needed)."""
    L = csa2.lib()
    fake = csa2.KVPlanes(256, 256, 256, 256, 1 << 22)  # aligned, never dereferenced
    # FLAT over 4M entries for 8 queries needs 128 MiB of scores
    rc = L.csa2_index_topk_noalloc(ctypes.byref(fake), 8, 256, 1 << 22, 256, 256, 512, 0, 8, 0, None,
                                   256, None, None)
    assert rc == 3  # CSA2_ERR_WORKSPACE


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point(oracle_mod):
    from gpu_common import SmallCache, require_gpu, to_dev, torch

    require_gpu()
    B, n_max = 3, 4133
    q, w = W.index_query(5, 0, B)
    hv = W.hot_vectors(q, w, 3.0)
    c = SmallCache(oracle_mod, 5, B, n_max, hot_prob=0.02, hotvecs=hv, stride=4224)
    ne = to_dev(np.array([4133, 4000, 777], np.int32))
    qd, wd = to_dev(q.view(np.int16)), to_dev(w)

    def with_workspace(mode, k, keep, pool_in=None):
        topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
        pool = torch.full((B, max(keep, 1)), -7, dtype=torch.int32, device="cuda")
        ws = csa2.workspace(csa2.index_topk_workspace_size(B, n_max, k, 8, keep))
        csa2.index_topk(c.planes, B, ne, n_max, qd, wd, k, mode, topk, ws, 8, keep, pool_in=pool_in,
                        pool_out=pool if mode == csa2.TOPK_HIER_BUILD else None)
        assert csa2.check(ws)[0] == 0
        return topk.cpu().numpy(), pool.cpu().numpy()

    def without(mode, k, keep, pool_in=None):
        topk = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
        pool = torch.full((B, max(keep, 1)), -7, dtype=torch.int32, device="cuda")
        csa2.index_topk_noalloc(c.planes, B, ne, n_max, qd, wd, k, mode, topk, 8, keep, pool_in=pool_in,
                                pool_out=pool if mode == csa2.TOPK_HIER_BUILD else None)
        torch.cuda.synchronize()
        return topk.cpu().numpy(), pool.cpu().numpy()

    ref_flat = with_workspace(csa2.TOPK_FLAT, 512, 0)
    ref_hier = with_workspace(csa2.TOPK_HIER_BUILD, 64, 100)
    pool_in = to_dev(ref_hier[1][:, :100].copy())
    ref_pool = with_workspace(csa2.TOPK_POOL, 128, 100, pool_in)
    for _ in range(2):  # two calls in a row share (and reuse) the scratch array
        got = without(csa2.TOPK_FLAT, 512, 0)
        assert np.array_equal(got[0], ref_flat[0])
        got = without(csa2.TOPK_HIER_BUILD, 64, 100)
        assert np.array_equal(got[0], ref_hier[0]) and np.array_equal(got[1], ref_hier[1])
        got = without(csa2.TOPK_POOL, 128, 100, pool_in)
        assert np.array_equal(got[0], ref_pool[0])
        assert csa2.index_topk_noalloc_check() == (0, 0)

    # HIER_BUILD with no pool_out keeps the pool inside the scratch array
    topk = torch.full((B, 64), -7, dtype=torch.int32, device="cuda")
    csa2.index_topk_noalloc(c.planes, B, ne, n_max, qd, wd, 64, csa2.TOPK_HIER_BUILD, topk, 8, 100)
    assert csa2.index_topk_noalloc_check()[0] == 0
    assert np.array_equal(topk.cpu().numpy(), ref_hier[0])

    # an error found on the device: a visible count above n_max is clamped and reported
    # through the scratch array's error word, which the check reads and clears
    bad = to_dev(np.array([4133, 5000, 777], np.int32))
    topk = torch.full((B, 512), -7, dtype=torch.int32, device="cuda")
    csa2.index_topk_noalloc(c.planes, B, bad, n_max, qd, wd, 512, csa2.TOPK_FLAT, topk)
    assert csa2.index_topk_noalloc_check() == (6, 5000)  # CSA2_ERR_INDEX_RANGE, the offending count
    assert csa2.index_topk_noalloc_check() == (0, 0)     # cleared
    got = without(csa2.TOPK_FLAT, 512, 0)                 # the next call starts clean
    assert np.array_equal(got[0], ref_flat[0])
    assert csa2.index_topk_noalloc_check()[0] == 0
