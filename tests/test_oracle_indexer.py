"""Pins of the oracle's lightning-indexer score and its selectors against numpy
restatements, brute-force rank counting and the hierarchy invariant."""
import numpy as np
import pytest

import synth
from synth.workloads import index_query, index_latents


def _planes(seed, n, hot=0.0, hotvec=None):
    import oracle

    lat = index_latents(seed, 0, 1, n, 0, 0, n, hot, hotvec)
    return oracle.quantize_index(lat)


def test_score_matches_numpy(oracle_mod):
    ic, isc = _planes(0, 300)
    q, w = index_query(0, 0, 1)
    got = oracle_mod.index_scores(ic, isc, q[0], w[0])
    K = oracle_mod.dequant_index(ic, isc)
    Q = synth.bf16_to_f32(q[0]).astype(np.float64)
    ref = np.maximum(K @ Q.T, 0.0) @ w[0].astype(np.float64)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13)
    at = oracle_mod.index_scores_at(ic, isc, np.array([5, -1, 299]), q[0], w[0])
    assert at[0] == got[5] and at[2] == got[299] and at[1] == -np.inf


def test_score_relu_and_sign(oracle_mod):
    """A key orthogonal to every head scores 0; a negative head weight flips sign."""
    ic = np.zeros((2, 64), np.uint8)
    isc = np.full((2, 4), 127, np.uint8)
    ic[1, 0] = 2  # element 0 = 1.0
    q = np.zeros((32, 128), np.uint16)
    q[:, 0] = 0x3F80  # 1.0
    q[3, 0] = 0xBF80  # -1.0 -> ReLU(-1) = 0
    w = np.ones(32, np.float32)
    w[0] = -2.0
    s = oracle_mod.index_scores(ic, isc, q, w)
    assert s[0] == 0.0
    # heads 1,2,4..31 give +1 each (30), head 0 gives -2, head 3 is clipped to 0
    assert s[1] == 30.0 - 2.0


def _brute_topk(scores, k):
    n = len(scores)
    chosen = []
    for j in range(n):
        better = sum(1 for i in range(n) if scores[i] > scores[j] or (scores[i] == scores[j] and i < j))
        if better < k:
            chosen.append(j)
    return chosen


@pytest.mark.parametrize("n,k", [(1, 4), (7, 4), (8, 8), (9, 8), (200, 17), (511, 512), (513, 512)])
def test_topk_brute_force(oracle_mod, n, k):
    rng = np.random.default_rng(n * 31 + k)
    scores = rng.integers(0, max(2, n // 4), n).astype(np.float64)  # many ties
    got = oracle_mod.topk(scores, k)
    ref = _brute_topk(list(scores), k)
    assert list(got[:len(ref)]) == ref
    assert np.all(got[len(ref):] == -1)


def test_topk_equal_scores_take_lowest_indices(oracle_mod):
    got = oracle_mod.topk(np.full(1000, 3.5), 512)
    assert np.array_equal(got, np.arange(512))


def test_block_max_and_pool(oracle_mod):
    rng = np.random.default_rng(5)
    n = 8 * 300 + 5  # ragged last block
    s = rng.standard_normal(n)
    bm = oracle_mod.block_max(s, 8)
    pad = np.concatenate([s, np.full(3, -np.inf)])
    assert np.array_equal(bm, pad.reshape(-1, 8).max(1))
    pool = oracle_mod.hier_pool(bm, 40)
    ref = _brute_topk(list(bm), 40)
    assert list(pool) == ref


def test_hierarchy_invariant_flat_in_pool(oracle_mod):
    """With n_blocks_keep >= k the flat top-k is contained in the pool, so the
    top-k inside the pool equals the flat top-k (the best entry of any block that
    holds a top-k entry ranks its block above every block without one)."""
    rng = np.random.default_rng(6)
    for trial in range(20):
        n = int(rng.integers(100, 3000))
        k = int(rng.integers(1, 60))
        keep = int(rng.integers(k, k + 40))
        s = rng.integers(0, 50, n).astype(np.float64) if trial % 2 else rng.standard_normal(n)
        flat = oracle_mod.topk(s, k)
        pool = oracle_mod.hier_pool(oracle_mod.block_max(s, 8), keep)
        hier = oracle_mod.pool_topk(s, pool, 8, k)
        assert np.array_equal(flat, hier)


def test_flat_topk_through_a_pool_of_k_blocks(oracle_mod):
    """The smallest pool that keeps the invariant: k blocks.  The flat top-k equals the
    top-k of the k best blocks' entries exactly, with heavy ties (a few distinct values,
    all-equal scores), partial last blocks and fewer blocks than k -- the identity the
    library's FLAT selection over long contexts relies on."""
    rng = np.random.default_rng(16)
    for trial in range(40):
        n = int(rng.integers(1, 5000))
        k = int(rng.integers(1, 700))
        kind = trial % 4
        if kind == 0:
            s = rng.standard_normal(n)
        elif kind == 1:
            s = rng.integers(0, 4, n).astype(np.float64)
        elif kind == 2:
            s = np.full(n, 2.5)
        else:
            s = np.repeat(rng.standard_normal((n + 7) // 8), 8)[:n]  # every block constant
        flat = oracle_mod.topk(s, k)
        pool = oracle_mod.hier_pool(oracle_mod.block_max(s, 8), k)
        assert np.array_equal(flat, oracle_mod.pool_topk(s, pool, 8, k)), (trial, n, k)


def test_hierarchy_sizes():
    """2048 blocks of 8 positions give at most 16,384 candidates; 1M entries make
    131,072 blocks (the hierarchical indexer's sizes)."""
    from synth.workloads import BLOCK, N_BLOCKS_KEEP

    assert BLOCK * N_BLOCKS_KEEP == 16384
    assert (1 << 20) // BLOCK == 131072


def test_pool_topk_restricts_to_pool(oracle_mod):
    s = np.arange(64, dtype=np.float64)  # best entries are the last ones
    pool = np.array([0, 2, -1], np.int32)  # blocks 0 and 2 only
    got = oracle_mod.pool_topk(s, pool, 8, 4)
    assert list(got) == [20, 21, 22, 23]
    got = oracle_mod.pool_topk(s, pool, 8, 20, n=19)  # entries >= n are invisible
    assert list(got[:11]) == list(range(0, 8)) + [16, 17, 18]
    assert np.all(got[11:] == -1)
