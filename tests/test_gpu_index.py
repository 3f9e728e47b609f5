"""csa2_index_topk against the oracle: scores, FLAT / HIER_BUILD / POOL
selection on ragged sizes spanning several tiles, and the degenerate cases."""
import numpy as np
import pytest

from gpu_common import SmallCache, csa2, require_gpu, to_dev, torch
from parity import check_topk
from synth import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(scope="module")
def cache(oracle_mod):
    q, w = W.index_query(0, 0, 3)
    hv = W.hot_vectors(q, w, 3.0)
    return SmallCache(oracle_mod, 0, 3, 4133, hot_prob=0.02, hotvecs=hv, stride=4224), q, w


def _run(c, q, w, n_entries, k, mode, keep=0, pool_in=None, n_max=None):
    B = len(n_entries)
    n_max = n_max or c.n_max
    ne = to_dev(np.array(n_entries, np.int32))
    qd, wd = to_dev(q.view(np.int16)), to_dev(w)
    topk = torch.empty((B, k), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, max(keep, 1)), dtype=torch.int32, device="cuda")
    ncols = keep * 8 if mode == csa2.TOPK_POOL else n_max
    scores = torch.empty((B, ncols), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_workspace_size(B, n_max, k, 8, keep))
    csa2.index_topk(c.planes, B, ne, n_max, qd, wd, k, mode, topk, ws, 8, keep,
                    pool_in=None if pool_in is None else to_dev(pool_in.astype(np.int32)),
                    pool_out=pool if mode == csa2.TOPK_HIER_BUILD else None, scores_out=scores)
    st, _ = csa2.check(ws)
    assert st == 0
    return topk.cpu().numpy(), pool.cpu().numpy(), scores.cpu().numpy()


def test_planes_identical(cache, oracle_mod):
    c, _, _ = cache
    for b in range(c.B):
        for g, o in zip(c.gpu_slot(b), c.oracle_slot(b)):
            assert np.array_equal(g, o)


def test_scores_match_oracle(cache, oracle_mod):
    c, q, w = cache
    n_entries = [4133, 4096, 700]
    topk, _, scores = _run(c, q, w, n_entries, 512, csa2.TOPK_FLAT)
    for b, n in enumerate(n_entries):
        _, _, ixc, ixs = c.oracle_slot(b)
        ref = oracle_mod.index_scores(ixc, ixs, q[b], w[b], n=n)
        assert np.allclose(scores[b, :n], ref, rtol=2e-5, atol=2e-5 * np.abs(ref).max())
        check_topk(topk[b], ref, 512, what=f"flat[{b}]")


@pytest.mark.parametrize("k,keep", [(64, 100), (512, 2048), (128, 16)])
def test_hier_build(cache, oracle_mod, k, keep):
    c, q, w = cache
    n_entries = [4133, 1000, 9]
    topk, pool, _ = _run(c, q, w, n_entries, k, csa2.TOPK_HIER_BUILD, keep=keep)
    for b, n in enumerate(n_entries):
        _, _, ixc, ixs = c.oracle_slot(b)
        s = oracle_mod.index_scores(ixc, ixs, q[b], w[b], n=n)
        bm = oracle_mod.block_max(s, 8)
        check_topk(pool[b], bm, keep, what=f"pool[{b}]")
        # token top-k inside the GPU's pool (the oracle scores decide)
        valid = np.zeros(n, bool)
        for u in pool[b][pool[b] >= 0]:
            valid[8 * u:min(8 * u + 8, n)] = True
        check_topk(topk[b], s, k, valid=valid, what=f"hier[{b}]")
        if keep >= k:  # the hierarchy invariant: same as the flat top-k (up to near-ties)
            check_topk(topk[b], s, k, what=f"hier-vs-flat[{b}]")


def test_pool_mode(cache, oracle_mod):
    c, q, w = cache
    n_entries = [4133, 4096, 700]
    keep = 300
    # the pool comes from the oracle with another query (a Reindex layer's pool)
    q2, w2 = W.index_query(0, 1, 3)
    pools = []
    for b, n in enumerate(n_entries):
        _, _, ixc, ixs = c.oracle_slot(b)
        pools.append(oracle_mod.hier_pool(oracle_mod.block_max(
            oracle_mod.index_scores(ixc, ixs, q2[b], w2[b], n=n), 8), keep))
    pools = np.stack(pools)
    topk, _, scores = _run(c, q, w, n_entries, 512, csa2.TOPK_POOL, keep=keep, pool_in=pools)
    for b, n in enumerate(n_entries):
        _, _, ixc, ixs = c.oracle_slot(b)
        s = oracle_mod.index_scores(ixc, ixs, q[b], w[b], n=n)
        valid = np.zeros(n, bool)
        for u in pools[b][pools[b] >= 0]:
            valid[8 * u:min(8 * u + 8, n)] = True
        check_topk(topk[b], s, 512, valid=valid, what=f"pool-mode[{b}]")
        ref = oracle_mod.pool_topk(s, pools[b], 8, 512)
        agree = np.intersect1d(topk[b][topk[b] >= 0], ref[ref >= 0]).size
        assert agree >= min(512, valid.sum()) - 2


def test_staged_pool_equals_pool_mode(cache, oracle_mod):
    """The pool's keys staged once (csa2_pool_stage) and re-scored by two Reindex queries
    (csa2_index_topk_staged) give exactly POOL mode's top-k and candidate scores; padded
    pool slots and blocks beyond n_entries stay masked although their staged bytes are
    left as garbage."""
    c, q, w = cache
    n_entries = [4133, 4096, 700]
    keep, k, B = 600, 512, 3
    q2, w2 = W.index_query(0, 1, 3)
    q3, w3 = W.index_query(0, 2, 3)
    pools = []
    for b, n in enumerate(n_entries):
        _, _, ixc, ixs = c.oracle_slot(b)
        pools.append(oracle_mod.hier_pool(oracle_mod.block_max(
            oracle_mod.index_scores(ixc, ixs, q2[b], w2[b], n=n), 8), keep))
    pools = np.stack(pools)
    assert (pools[2] < 0).any() and (pools[0] < 0).any()  # padding present
    pool_d = to_dev(pools.astype(np.int32))
    ne = to_dev(np.array(n_entries, np.int32))
    stage = csa2.PoolStage.empty(B, keep)
    stage.codes.fill_(0xFF)
    stage.scales.fill_(0xFF)
    csa2.pool_stage(c.planes, B, ne, c.n_max, pool_d, stage, 8, keep)
    ws = csa2.workspace(csa2.index_topk_workspace_size(B, c.n_max, k, 8, keep))
    for qq, ww in ((q, w), (q3, w3)):
        topk = torch.empty((B, k), dtype=torch.int32, device="cuda")
        scores = torch.empty((B, keep * 8), dtype=torch.float32, device="cuda")
        csa2.index_topk_staged(stage, B, ne, c.n_max, to_dev(qq.view(np.int16)), to_dev(ww), k, pool_d, topk,
                               ws, 8, keep, scores_out=scores)
        assert csa2.check(ws)[0] == 0
        ref_topk, _, ref_scores = _run(c, qq, ww, n_entries, k, csa2.TOPK_POOL, keep=keep, pool_in=pools)
        topk, scores = topk.cpu().numpy(), scores.cpu().numpy()
        assert np.array_equal(topk, ref_topk)
        for b, n in enumerate(n_entries):
            cand = np.full(keep * 8, False)
            for u_i, u in enumerate(pools[b]):
                if u >= 0:
                    cand[u_i * 8:u_i * 8 + min(8, n - 8 * u)] = True
            assert np.array_equal(scores[b][cand], ref_scores[b][cand])
            _, _, ixc, ixs = c.oracle_slot(b)
            s = oracle_mod.index_scores(ixc, ixs, qq[b], ww[b], n=n)
            valid = np.zeros(n, bool)
            for u in pools[b][pools[b] >= 0]:
                valid[8 * u:min(8 * u + 8, n)] = True
            check_topk(topk[b], s, k, valid=valid, what=f"staged[{b}]")


def test_degenerate_sizes(cache, oracle_mod):
    c, q, w = cache
    for n_entries in ([1, 511, 513], [0, 8, 7]):
        topk, _, _ = _run(c, q, w, n_entries, 512, csa2.TOPK_FLAT)
        for b, n in enumerate(n_entries):
            _, _, ixc, ixs = c.oracle_slot(b)
            s = oracle_mod.index_scores(ixc, ixs, q[b], w[b], n=n)
            check_topk(topk[b], s, 512, what=f"n={n}")
    topk, pool, _ = _run(c, q, w, [0, 3, 17], 4, csa2.TOPK_HIER_BUILD, keep=2)
    assert np.all(topk[0] == -1) and np.all(pool[0] == -1)
    assert list(topk[1][:3]) == [0, 1, 2] and topk[1][3] == -1


def test_equal_scores_take_lowest_indices(cache):
    """A zero query scores every entry exactly 0: the k lowest indices win."""
    c, q, w = cache
    qz = np.zeros_like(q)
    topk, _, _ = _run(c, qz, w, [4133, 4096, 700], 512, csa2.TOPK_FLAT)
    for b in range(3):
        assert np.array_equal(topk[b], np.arange(512))
    topk, pool, _ = _run(c, qz, w, [4133, 4096, 700], 64, csa2.TOPK_HIER_BUILD, keep=100)
    assert np.array_equal(pool[0], np.arange(100)) and np.array_equal(topk[0], np.arange(64))


def test_negative_weights_general_sign(cache, oracle_mod):
    c, q, w = cache
    wn = (w - 0.5).astype(np.float32)
    topk, _, scores = _run(c, q, wn, [4133, 4096, 700], 256, csa2.TOPK_FLAT)
    for b, n in enumerate([4133, 4096, 700]):
        _, _, ixc, ixs = c.oracle_slot(b)
        s = oracle_mod.index_scores(ixc, ixs, q[b], wn[b], n=n)
        check_topk(topk[b], s, 256, what=f"signed[{b}]")


def test_mxfp4_query(cache, oracle_mod):
    """The MXFP4 indexer query: bytes identical to the oracle's quantize-then-decode of q (the
    key rule on groups of 32), tiny and all-zero groups included; the index over the quantized
    query matches the oracle's scores of the same quantized query."""
    import synth

    c, q, w = cache
    q = q.copy()
    q[0, 0, :32] = 0                                      # an all-zero group
    q[1, 3, 32:64] = (q[1, 3, 32:64].astype(np.uint32) & 0x807F).astype(np.uint16)  # subnormal-range group
    n_rows = q.shape[0] * q.shape[1]
    qd = to_dev(q.view(np.int16))
    out = torch.empty_like(qd)
    csa2.quantize_index_query(qd, n_rows, out)
    got = out.cpu().numpy().view(np.uint16).reshape(q.shape)
    codes, scales = oracle_mod.quantize_index(synth.bf16_to_f32(q).reshape(n_rows, 128))
    vals = oracle_mod.dequant_index(codes, scales).astype(np.float32)
    ref = (vals.view(np.uint32) >> 16).astype(np.uint16).reshape(q.shape)
    assert np.array_equal(vals.view(np.uint32) & 0xFFFF, np.zeros_like(vals.view(np.uint32)))  # exact in bf16
    assert np.array_equal(got, ref)
    # in place, and through the index
    csa2.quantize_index_query(qd, n_rows, qd)
    assert np.array_equal(qd.cpu().numpy().view(np.uint16).reshape(q.shape), ref)
    n_entries = [4133, 4096, 700]
    topk, _, scores = _run(c, got, w, n_entries, 512, csa2.TOPK_FLAT)
    for b, n in enumerate(n_entries):
        _, _, ixc, ixs = c.oracle_slot(b)
        s = oracle_mod.index_scores(ixc, ixs, got[b], w[b], n=n)
        assert np.allclose(scores[b, :n], s, rtol=2e-5, atol=2e-5 * np.abs(s).max())
        check_topk(topk[b], s, 512, what=f"mxfp4-q[{b}]")


def _prefill(planes, seq, q, w, n_vis, n_max, k=512):
    Q = q.shape[0]
    topk = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_prefill_workspace_size(Q, n_max, k))
    csa2.index_topk_prefill(planes, seq, Q, to_dev(n_vis), n_max, to_dev(q.view(np.int16)), to_dev(w), k, topk, ws)
    assert csa2.check(ws)[0] == 0
    return topk.cpu().numpy()


@pytest.mark.parametrize("Q", [40, 43, 100, 160])
def test_prefill_indexer_shared_slot(cache, oracle_mod, Q):
    """Q queries of one slot, each with its own causal bound: every query's top-512 is the
    oracle's top-512 of that query over entries [0, n_visible).  Every count fits one
    select CTA, so the selects run in the one-CTA band; 43 queries leave the scan a last
    group of three (it scans four queries per key tile)."""
    c, _, _ = cache
    seq = 1
    q, w = W.index_query(4, 0, Q)
    rng = np.random.default_rng(2)
    n_vis = np.concatenate([[0, 1, 7, 513, 4133], rng.integers(0, 4134, Q - 5)]).astype(np.int32)
    topk = _prefill(c.planes, seq, q, w, n_vis, c.n_max)
    _, _, ixc, ixs = c.oracle_slot(seq)
    for i in range(Q):
        s = oracle_mod.index_scores(ixc, ixs, q[i], w[i], n=int(n_vis[i])) if n_vis[i] else np.zeros(0)
        check_topk(topk[i], s, 512, what=f"prefill[{i}]")


def test_prefill_indexer_batches(cache, oracle_mod):
    """A 2^24-entry bound makes the scores, block maxima and pools of only 17 queries fit
    the workspace's 1.25 GiB, so 40 queries run in three launches, each selecting through
    a pool of 512 blocks whose maxima go through the streaming select (the visible entries
    are the cache's first 4,133)."""
    c, _, _ = cache
    Q, stride = 40, 1 << 24
    big = csa2.Planes.empty(1, stride)
    src = c.gpu_slot(0)
    for t, a in zip((big.kv_codes, big.kv_scales, big.ix_codes, big.ix_scales), src):
        t[:a.shape[0]] = torch.from_numpy(a).to(t.device)
    q, w = W.index_query(5, 0, Q)
    n_vis = np.random.default_rng(3).integers(1, 4134, Q).astype(np.int32)
    assert csa2.index_topk_prefill_workspace_size(Q, stride, 512) < 2 * (1 << 30)
    topk = _prefill(big, 0, q, w, n_vis, stride)
    _, _, ixc, ixs = c.oracle_slot(0)
    for i in range(Q):
        s = oracle_mod.index_scores(ixc, ixs, q[i], w[i], n=int(n_vis[i]))
        check_topk(topk[i], s, 512, what=f"prefill-batched[{i}]")


def test_prefill_indexer_mxfp4_queries(cache, oracle_mod):
    """Half of the queries are MXFP4 (the oracle's quantize-then-decode of their bf16 rows),
    half plain bf16, in one launch: the scan takes the hi-only path (N = 32) for the former
    and the hi/lo path for the latter; every query's top-512 matches the oracle's scores of
    the query it was given."""
    import synth

    c, _, _ = cache
    seq, Q = 1, 48
    q, w = W.index_query(6, 0, Q)
    codes, scales = oracle_mod.quantize_index(synth.bf16_to_f32(q[:Q // 2]).reshape(-1, 128))
    vals = oracle_mod.dequant_index(codes, scales).astype(np.float32)
    assert np.array_equal(vals.view(np.uint32) & 0xFFFF, np.zeros_like(vals.view(np.uint32)))  # exact in bf16
    q = q.copy()
    q[:Q // 2] = (vals.view(np.uint32) >> 16).astype(np.uint16).reshape(Q // 2, 32, 128)
    n_vis = np.random.default_rng(4).integers(1, 4134, Q).astype(np.int32)
    topk = _prefill(c.planes, seq, q, w, n_vis, c.n_max)
    _, _, ixc, ixs = c.oracle_slot(seq)
    for i in range(Q):
        s = oracle_mod.index_scores(ixc, ixs, q[i], w[i], n=int(n_vis[i]))
        check_topk(topk[i], s, 512, what=f"prefill-mxfp4[{i}]")


def test_prefill_indexer_mixed_groups(cache, oracle_mod):
    """MXFP4 and bf16 queries alternate, so every four-query group of the scan mixes them
    (the group takes the hi/lo path, exact for both), and 42 queries end in a group of two;
    the visible counts differ inside each group.  Every top-512 matches the oracle's."""
    import synth

    c, _, _ = cache
    seq, Q = 1, 42
    q, w = W.index_query(7, 0, Q)
    codes, scales = oracle_mod.quantize_index(synth.bf16_to_f32(q[::2]).reshape(-1, 128))
    vals = oracle_mod.dequant_index(codes, scales).astype(np.float32)
    q = q.copy()
    q[::2] = (vals.view(np.uint32) >> 16).astype(np.uint16).reshape(-1, 32, 128)
    n_vis = np.random.default_rng(5).integers(1, 4134, Q).astype(np.int32)
    topk = _prefill(c.planes, seq, q, w, n_vis, c.n_max)
    _, _, ixc, ixs = c.oracle_slot(seq)
    for i in range(Q):
        s = oracle_mod.index_scores(ixc, ixs, q[i], w[i], n=int(n_vis[i]))
        check_topk(topk[i], s, 512, what=f"prefill-mixed[{i}]")
