"""Parity on the decode workloads, in the launch configuration the benchmark
uses: the single-query 4K workload in full, the batch-64 encoder workload (one
index pass shared by six attention passes) and the batch-32 1M-context
hierarchical workload at full size, checked on sampled queries whose whole
caches the oracle regenerates from the same seeded generator."""
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from gpu_common import csa2, require_gpu, to_dev, torch
from parity import check_attention, check_topk
from synth import workloads as W

pytestmark = pytest.mark.gpu
SCALE = 1.0 / math.sqrt(512)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def oracle_planes(oracle, seed, f, B, N, b, hot_prob=0.0, hotvec=None, chunk=1 << 16):
    """The oracle's encoding of sequence b's cache (generated on the host)."""
    kvc = np.empty((N, 256), np.uint8)
    kvs = np.empty((N, 32), np.uint8)
    ixc = np.empty((N, 64), np.uint8)
    ixs = np.empty((N, 4), np.uint8)

    def enc(j0):
        cnt = min(chunk, N - j0)
        a = oracle.quantize_main(W.main_latents(seed, f, B, N, b, j0, cnt))
        c = oracle.quantize_index(W.index_latents(seed, f, B, N, b, j0, cnt, hot_prob, hotvec))
        return j0, cnt, a, c

    with ThreadPoolExecutor(16) as ex:
        for j0, cnt, (c1, s1), (c2, s2) in ex.map(enc, range(0, N, chunk)):
            kvc[j0:j0 + cnt], kvs[j0:j0 + cnt] = c1, s1
            ixc[j0:j0 + cnt], ixs[j0:j0 + cnt] = c2, s2
    return kvc, kvs, ixc, ixs


def gpu_decode(wl, planes, layers_q, layers_swa, qd, wd, hier=False, keep=2048):
    B, N, k = wl.B, wl.N, wl.k
    ne = torch.full((B,), N, dtype=torch.int32, device="cuda")
    topk = torch.empty((B, k), dtype=torch.int32, device="cuda")
    pool = torch.empty((B, keep), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_workspace_size(B, N, k, 8, keep if hier else 0))
    if hier:
        csa2.index_topk(planes, B, ne, N, qd, wd, k, csa2.TOPK_HIER_BUILD, topk, ws, 8, keep, pool_out=pool)
    else:
        csa2.index_topk(planes, B, ne, N, qd, wd, k, csa2.TOPK_FLAT, topk, ws)
    assert csa2.check(ws)[0] == 0
    outs = []
    wsa = csa2.workspace(csa2.sparse_attn_workspace_size(B, k, wl.n_swa))
    for qa, swa in zip(layers_q, layers_swa):
        out = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
        csa2.sparse_attn_decode(planes, B, topk, k, swa, wl.n_swa, qa, SCALE, out, wsa)
        assert csa2.check(wsa)[0] == 0
        outs.append(out.cpu().numpy())
    return topk.cpu().numpy(), pool.cpu().numpy(), outs


def test_single_query_4k(oracle_mod):
    """B=1, N=4096, FLAT top-512 + 64x512 attention over 512 + 128 rows: every output."""
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    wl = W.SINGLE_4K
    planes = csa2.Planes.empty(wl.B, wl.N)
    WL.fill_planes(planes, wl.seed, 0, wl.B, wl.N)
    qd, wd, q, w = WL.index_query_dev(wl.seed, 0, wl.B)
    qa_d, qa = WL.attn_query_dev(wl.seed, 0, wl.B)
    swa_d = WL.swa_dev(wl.seed, 0, wl.B)
    topk, _, outs = gpu_decode(wl, planes, [qa_d], [swa_d], qd, wd)
    kvc, kvs, ixc, ixs = oracle_planes(oracle_mod, wl.seed, 0, wl.B, wl.N, 0)
    s = oracle_mod.index_scores(ixc, ixs, q[0], w[0])
    check_topk(topk[0], s, wl.k, what="4k topk")
    sel = oracle_mod.topk(s, wl.k)
    ref, _ = oracle_mod.attention(kvc, kvs, sel, W.swa_rows(wl.seed, 0, 1)[0], qa[0], SCALE)
    check_attention(outs[0], ref[None])


def test_encoder_batch64_six_attention_passes(oracle_mod):
    """B=64, N=32,768 (65,536 tokens at m=2): one FLAT index pass, six attention
    passes (Full + 5 Reuse) each with its own q and window; queries 0 and 63 checked."""
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    wl = W.ENCODER_B64
    planes = csa2.Planes.empty(wl.B, wl.N)
    WL.fill_planes(planes, wl.seed, 0, wl.B, wl.N)
    qd, wd, q, w = WL.index_query_dev(wl.seed, 0, wl.B)
    qs = [WL.attn_query_dev(wl.seed, l, wl.B) for l in range(wl.n_attn)]
    swas = [WL.swa_dev(wl.seed, l, wl.B) for l in range(wl.n_attn)]
    topk, _, outs = gpu_decode(wl, planes, [a for a, _ in qs], swas, qd, wd)
    for b in (0, 63):
        kvc, kvs, ixc, ixs = oracle_planes(oracle_mod, wl.seed, 0, wl.B, wl.N, b)
        s = oracle_mod.index_scores(ixc, ixs, q[b], w[b])
        check_topk(topk[b], s, wl.k, what=f"encoder topk[{b}]")
        sel = oracle_mod.topk(s, wl.k)
        for l in range(wl.n_attn):
            sw = W.swa_rows(wl.seed, l, wl.B)[b]
            ref, _ = oracle_mod.attention(kvc, kvs, sel, sw, qs[l][1][b], SCALE)
            check_attention(outs[l][b:b + 1], ref[None], what=f"encoder attn[{b}, layer {l}]")


def test_decoder_1m_hierarchical_full_size(oracle_mod):
    """B=32 at 1,048,576 entries, HIER_BUILD (131,072 blocks -> 2,048 -> top-512) +
    attention: the benchmark's configuration; queries 0 and 31 checked against the
    oracle over their whole caches (pool, top-k and attention)."""
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    wl = W.DECODER_1M
    planes = csa2.Planes.empty(wl.B, wl.N)
    qd, wd, q, w = WL.index_query_dev(wl.seed, 0, wl.B)
    hv = W.hot_vectors(q, w, wl.hot_gain)
    WL.fill_planes(planes, wl.seed, 0, wl.B, wl.N, hot_prob=wl.hot_prob, hotvecs=hv)
    qa_d, qa = WL.attn_query_dev(wl.seed, 0, wl.B)
    swa_d = WL.swa_dev(wl.seed, 0, wl.B)
    topk, pool, outs = gpu_decode(wl, planes, [qa_d], [swa_d], qd, wd, hier=True)
    del planes
    torch.cuda.empty_cache()
    for b in (0, 31):
        kvc, kvs, ixc, ixs = oracle_planes(oracle_mod, wl.seed, 0, wl.B, wl.N, b, wl.hot_prob, hv[b])
        s = oracle_mod.index_scores(ixc, ixs, q[b], w[b])
        bm = oracle_mod.block_max(s, 8)
        check_topk(pool[b], bm, 2048, what=f"1M pool[{b}]")
        check_topk(topk[b], s, wl.k, what=f"1M topk[{b}]")
        sel = oracle_mod.pool_topk(s, oracle_mod.hier_pool(bm, 2048), 8, wl.k)
        ref, _ = oracle_mod.attention(kvc, kvs, sel, W.swa_rows(wl.seed, 0, wl.B)[b], qa[b], SCALE)
        check_attention(outs[0][b:b + 1], ref[None], what=f"1M attn[{b}]")


def forty_layer_step(oracle_mod, seed, B, T, keep, check_queries, k=512):
    """Runs the 40-layer decode step (SWA-only, Full, Reuse, Reindex layers) at batch B over a
    T-token context through schedule.run_step, then checks the queries in `check_queries`
    against the oracle over their whole caches: every index layer's top-k (and the decoder
    Full layer's pool) under the 1e-3 band, and all 40 attention outputs within 1e-2 RMS.
    The oracle follows the same schedule with its own selections; where an entry inside
    the band differs, the attention reference takes the GPU's (band-checked) selection."""
    from compressed_sparse_attention_nvfp4_gb300 import schedule as SCH
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL
    from synth import e4m3_normal

    t = csa2.v41_layer_table()
    full = [l for l in range(40) if t["mode"][l] == csa2.LAYER_FULL]
    n_of = {f: T // t["m"][f] for f in full}
    kv, ne, nm = {}, {}, {}
    for f in full:
        kv[f] = csa2.Planes.empty(B, n_of[f])
        WL.fill_planes(kv[f], seed, f, B, n_of[f])
        ne[f] = torch.full((B,), n_of[f], dtype=torch.int32, device="cuda")
        nm[f] = n_of[f]
    qidx, w, q, swa, out, qh, wh, qah = {}, {}, {}, {}, {}, {}, {}, {}
    for l in range(40):
        if t["mode"][l] in (csa2.LAYER_FULL, csa2.LAYER_REINDEX):
            qidx[l], w[l], qh[l], wh[l] = WL.index_query_dev(seed, l, B)
        q[l], qah[l] = WL.attn_query_dev(seed, l, B)
        swa[l] = WL.swa_dev(seed, l, B)
        out[l] = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
    buf = SCH.StepBuffers(B=B, kv=kv, n_entries=ne, n_max=nm, qidx=qidx, w=w, q=q, swa=swa, out=out,
                          k=k, n_blocks_keep=keep)
    SCH.allocate_scratch(buf)
    calls = SCH.run_step(buf)
    torch.cuda.synchronize()
    assert calls == 40 + 8 + 1  # 40 attention calls, 8 indexer calls, one gather of the shared pool
    assert csa2.check(buf.ws_index)[0] == 0 and csa2.check(buf.ws_attn)[0] == 0
    gtopk = {l: buf.topk[l].cpu().numpy() for l in buf.topk}
    dec_full = [f for f in full if t["m"][f] == 1][0]
    gpool = buf.pool[dec_full].cpu().numpy()
    gout = {l: out[l][list(check_queries)].cpu().numpy() for l in range(40)}
    del buf, kv, q, swa, out
    torch.cuda.empty_cache()

    def ref_selection(oracle_sel, gpu_sel):
        g = gpu_sel[gpu_sel >= 0]
        o = np.sort(oracle_sel[oracle_sel >= 0])
        return oracle_sel if np.array_equal(o, g) else g.astype(np.int32)

    for qi, b in enumerate(check_queries):
        planes = {f: oracle_planes(oracle_mod, seed, f, B, n_of[f], b) for f in full}
        sel = {}
        opool = None
        for l in range(40):
            mode = t["mode"][l]
            if mode == csa2.LAYER_SWA:
                sel_l = np.zeros(0, np.int32)
                kv_o = planes[full[0]][:2]
            else:
                f = t["kv_src"][l]
                kvc, kvs, ixc, ixs = planes[f]
                if mode in (csa2.LAYER_FULL, csa2.LAYER_REINDEX):
                    s = oracle_mod.index_scores(ixc, ixs, qh[l][b], wh[l][b])
                    if mode == csa2.LAYER_FULL and t["m"][l] == 2:
                        check_topk(gtopk[l][b], s, k, what=f"L{l} flat[{b}]")
                        sel[l] = ref_selection(oracle_mod.topk(s, k), gtopk[l][b])
                    else:
                        if mode == csa2.LAYER_FULL:
                            bm = oracle_mod.block_max(s, 8)
                            check_topk(gpool[b], bm, keep, what=f"L{l} pool[{b}]")
                            opool = oracle_mod.hier_pool(bm, keep)
                        valid = np.zeros(n_of[f], bool)
                        for u in gpool[b][gpool[b] >= 0]:
                            valid[8 * u:8 * u + 8] = True
                        check_topk(gtopk[l][b], s, k, valid=valid, what=f"L{l} in-pool[{b}]")
                        sel[l] = ref_selection(oracle_mod.pool_topk(s, opool, 8, k), gtopk[l][b])
                sel_l = sel[t["topk_src"][l]]
                kv_o = (kvc, kvs)
            n_sw = W.N_SWA * W.D_MAIN
            sw = e4m3_normal(seed, W.tid_swa(l), n_sw, offset=b * n_sw).reshape(W.N_SWA, W.D_MAIN)
            ref, _ = oracle_mod.attention(kv_o[0], kv_o[1], sel_l, sw, qah[l][b], SCALE)
            check_attention(gout[l][qi:qi + 1], ref[None], what=f"L{l} attn[{b}]")


def test_v41_forty_layer_step_reduced(oracle_mod):
    """The 40-layer decode step at batch 2 and a 16,384-token context (8,192 encoder
    entries at m=2, 16,384 decoder entries at m=1, a 256-block pool): every index layer
    and all 40 outputs of both queries vs the oracle."""
    forty_layer_step(oracle_mod, seed=4, B=2, T=16384, keep=256, check_queries=(0, 1))


def test_v41_forty_layer_step_full_size(oracle_mod):
    """The 40-layer decode step at the benchmark's shape: batch 128 at a 262,144-token
    context (131,072 encoder entries at m=2, 262,144 decoder entries at m=1, a 2,048-block
    pool), the launch configuration bench.py times (the select's cluster halving at batch
    128, the pool gather over 128 x 2,048 blocks, one attention CTA per query).  Queries 0
    and 127 are checked against the oracle over their whole caches in every layer
    ("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression", 4.2 and 4.3)."""
    forty_layer_step(oracle_mod, seed=4, B=128, T=262144, keep=2048, check_queries=(0, 127))


def test_prefill_indexer_full_size_sampled(oracle_mod):
    """The prefill indexer at the benchmark's shape: 2,048 queries over one 131,072-entry
    slot, query i seeing its first 64 (i + 1) entries (the causal bound of token 128 (i + 1)
    at m = 2), in one call as bench.py times it: the scan writes the scores and the 8-entry
    block maxima, and each query's top-512 is selected through a pool of its 512 best blocks.
    Queries from the shortest to the longest (on both sides of 16,384, 32,768 and 65,536
    visible entries) are checked against the oracle's scores of their visible prefix
    ("DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence", CSA step 2)."""
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    N, Q, seed, k = 131072, 2048, 6, 512
    n_vis = (np.arange(Q, dtype=np.int64) + 1) * 64
    planes = csa2.Planes.empty(1, N)
    WL.fill_planes(planes, seed, 0, 1, N)
    qd, wd, q, w = WL.index_query_dev(seed, 0, Q)
    topk = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_prefill_workspace_size(Q, N, k))
    csa2.index_topk_prefill(planes, 0, Q, to_dev(n_vis.astype(np.int32)), N, qd, wd, k, topk, ws)
    assert csa2.check(ws)[0] == 0
    topk = topk.cpu().numpy()
    del planes, ws
    torch.cuda.empty_cache()

    ixc = np.empty((N, 64), np.uint8)
    ixs = np.empty((N, 4), np.uint8)

    def enc(j0, cnt=1 << 16):
        return j0, oracle_mod.quantize_index(W.index_latents(seed, 0, 1, N, 0, j0, cnt, 0.0, None))

    with ThreadPoolExecutor(4) as ex:
        for j0, (c2, s2) in ex.map(enc, range(0, N, 1 << 16)):
            ixc[j0:j0 + (1 << 16)], ixs[j0:j0 + (1 << 16)] = c2, s2
    for i in (0, 7, 255, 256, 511, 512, 1023, 1024, 2047):
        s = oracle_mod.index_scores(ixc, ixs, q[i], w[i], n=int(n_vis[i]))
        check_topk(topk[i], s, k, what=f"prefill-full[{i}]")


def test_select_bands_and_streaming_select(oracle_mod):
    """Selections past 8 x 16,384 candidates, which no benchmarked shape reaches: a FLAT
    decode over 150,016 entries, selected through a pool of k blocks by csa2_index_topk and
    directly by the streaming select (`k_select`, whose slices exceed a CTA's shared memory)
    in the allocation-free entry point -- the two must give the same ids exactly -- and a
    prefill whose visible counts sit on both sides of every size-band edge (16,384, 32,768,
    65,536, 131,072), the last band again streaming.  Every top-512 against the oracle's
    scores ("DeepSeek-V4: Towards Highly Efficient Million-Token Context Intelligence",
    CSA step 2)."""
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    N, B, seed, k = 150016, 2, 11, 512
    planes = csa2.Planes.empty(B, N)
    WL.fill_planes(planes, seed, 0, B, N)
    ixc = np.empty((B, N, 64), np.uint8)
    ixs = np.empty((B, N, 4), np.uint8)
    for b in range(B):
        for j0 in range(0, N, 1 << 16):
            cnt = min(1 << 16, N - j0)
            c2, s2 = oracle_mod.quantize_index(W.index_latents(seed, 0, B, N, b, j0, cnt, 0.0, None))
            ixc[b, j0:j0 + cnt], ixs[b, j0:j0 + cnt] = c2, s2

    # FLAT decode, both queries streaming
    n_entries = [N, 140000]
    qd, wd, q, w = WL.index_query_dev(seed, 0, B)
    topk = torch.empty((B, k), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_workspace_size(B, N, k))
    ne = to_dev(np.array(n_entries, np.int32))
    csa2.index_topk(planes, B, ne, N, qd, wd, k, csa2.TOPK_FLAT, topk, ws)
    assert csa2.check(ws)[0] == 0
    direct = torch.full((B, k), -7, dtype=torch.int32, device="cuda")
    csa2.index_topk_noalloc(planes, B, ne, N, qd, wd, k, csa2.TOPK_FLAT, direct)
    assert csa2.index_topk_noalloc_check()[0] == 0
    topk = topk.cpu().numpy()
    assert np.array_equal(topk, direct.cpu().numpy())  # the pool of k blocks loses nothing
    for b, n in enumerate(n_entries):
        s = oracle_mod.index_scores(ixc[b], ixs[b], q[b], w[b], n=n)
        check_topk(topk[b], s, k, what=f"flat-streaming[{b}]")

    # prefill over slot 1 with visible counts around every band edge
    n_vis = np.array([N, 131073, 131072, 65537, 65536, 32769, 32768, 16385, 16384, 7, 0], np.int32)
    Q = n_vis.shape[0]
    qd, wd, q, w = WL.index_query_dev(seed, 1, Q)
    topk = torch.empty((Q, k), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_prefill_workspace_size(Q, N, k))
    csa2.index_topk_prefill(planes, 1, Q, to_dev(n_vis), N, qd, wd, k, topk, ws)
    assert csa2.check(ws)[0] == 0
    topk = topk.cpu().numpy()
    for i in range(Q):
        n = int(n_vis[i])
        s = oracle_mod.index_scores(ixc[1], ixs[1], q[i], w[i], n=n) if n else np.zeros(0)
        check_topk(topk[i], s, k, what=f"prefill-band[{i}] n={n}")
