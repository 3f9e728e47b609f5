"""The C-ABI library: it loads without a GPU, exports every entry point that
include/csa2.h declares, validates arguments on the host, and carries the
V4.1-Flash layer table whose byte arithmetic the pages print."""
import ctypes
import os
import re

import pytest

import compressed_sparse_attention_nvfp4_gb300 as csa2
from conftest import ROOT, read_table


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(csa2.LIB_PATH):
        from compressed_sparse_attention_nvfp4_gb300 import build

        build.build()
    return csa2.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(csa2_\w+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_header_entry_sizes():
    text = open(os.path.join(ROOT, "include", "csa2.h")).read()
    tab = {k: v for k, v in read_table("bytes_per_token.txt")}
    get = lambda name: int(re.search(rf"#define {name} (\d+)", text).group(1))
    assert get("CSA2_MAIN_CODE_BYTES") + get("CSA2_MAIN_SCALE_BYTES") == int(tab["main_entry_bytes"])
    assert get("CSA2_IDX_CODE_BYTES") + get("CSA2_IDX_SCALE_BYTES") == int(tab["index_entry_bytes"])
    assert get("CSA2_ENTRY_BYTES") == int(tab["entry_bytes"])


def test_status_strings(L):
    for s in range(7):
        assert csa2.status_string(s)


def test_layer_table_matches_pages(L):
    t = csa2.v41_layer_table()
    names = {csa2.LAYER_SWA: "SWA", csa2.LAYER_FULL: "FULL", csa2.LAYER_REINDEX: "REINDEX",
             csa2.LAYER_REUSE: "REUSE"}
    rows = read_table("v41_schedule.txt")
    assert len(rows) == 40
    for l, (li, mode, m) in enumerate(rows):
        assert int(li) == l
        assert names[t["mode"][l]] == mode, l
        assert t["m"][l] == int(m), l
    full = [l for l in range(40) if t["mode"][l] == csa2.LAYER_FULL]
    tab = {k: v for k, v in read_table("bytes_per_token.txt")}
    assert full == [int(x) for x in tab["full_layers"].split(",")]
    reindex = [l for l in range(40) if t["mode"][l] == csa2.LAYER_REINDEX]
    assert reindex == [24, 28, 32, 36]
    reuse = [l for l in range(40) if t["mode"][l] == csa2.LAYER_REUSE]
    assert len(full) == 4 and len(reindex) == 4 and len(reuse) == 30  # 38 CSA2 layers, 8 indexers
    # sources: p(l) nearest Full at or before l, p'(l) nearest Full/Reindex
    for l in range(2, 40):
        assert t["kv_src"][l] == max(f for f in full if f <= l)
        assert t["topk_src"][l] == max(f for f in full + reindex if f <= l)
        assert t["pool_src"][l] == (20 if l in reindex else -1)


def test_global_bytes_per_token_890(L):
    """B_global = sum over KV-owning layers of entry_bytes / m_l = 3*356/2 + 356 = 890."""
    t = csa2.v41_layer_table()
    tab = {k: v for k, v in read_table("bytes_per_token.txt")}
    total = sum(csa2.ENTRY_BYTES / t["m"][l] for l in range(40) if t["mode"][l] == csa2.LAYER_FULL)
    assert total == int(tab["global_bytes_per_token"])
    assert 2 ** 20 * total / 2 ** 20 == 890  # 890 MiB at a 2^20-token context
    # the other models of the same table, by the same formula
    assert 95 * 2 * 8 * 128 * 2 == int(tab["v1_bytes_per_token"])
    assert 61 * ((512 + 16 + 128) + (128 + 4)) == int(tab["v32_bytes_per_token"])


def test_indexer_mac_model(L):
    """Decode indexer MACs: 4096 * (3N/2 + N) + 4 * 4096 * 16384 = 10240 N + 0.27 G
    ("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression", 4.4),
    counted from the layer table: Full layers scan N/m entries, Reindex layers the pool."""
    t = csa2.v41_layer_table()
    N = 1 << 20
    macs = 0
    for l in range(40):
        if t["mode"][l] == csa2.LAYER_FULL:
            macs += csa2.H_IDX * csa2.D_IDX * (N // t["m"][l])
        elif t["mode"][l] == csa2.LAYER_REINDEX:
            macs += csa2.H_IDX * csa2.D_IDX * 2048 * 8
    assert macs == 10240 * N + 4 * 4096 * 16384
    assert abs(macs - 10.2e9 - 0.27e9) / macs < 0.08  # "about 10.2 G" plus the constant term


def test_host_validation_without_gpu(L):
    P = csa2.KVPlanes(None, None, None, None, 0)
    rc = L.csa2_index_topk(ctypes.byref(P), 1, None, 0, None, None, 512, 0, 8, 0, None, None, None,
                           None, None, 0, None)
    assert rc == 1
    rc = L.csa2_sparse_attn_decode(ctypes.byref(P), 1, None, 512, None, 0, None, 1.0, None, None,
                                   None, None, None, None, None, 0, None)
    assert rc == 1
    assert L.csa2_quantize_index_query(None, -1, None, None) == 1
    assert L.csa2_quantize_index_query(16, 4, None, None) == 1      # no output
    assert L.csa2_quantize_index_query(8, 4, 16, None) == 1         # misaligned input
    assert L.csa2_quantize_index_query(None, 0, None, None) == 0    # nothing to do
    rc = L.csa2_cache_write(None, 64, 5120, None, None, None, 2, ctypes.byref(P), 0, 0, None, 0, None, 0,
                            None)
    assert rc == 1
    fake = csa2.KVPlanes(16, 16, 16, 16, 100)  # aligned non-null pointers, never dereferenced
    # k out of range, bad mode, workspace missing
    assert L.csa2_index_topk(ctypes.byref(fake), 1, 16, 10, 16, 16, 0, 0, 8, 0, None, 16, None, None,
                             None, 0, None) == 1
    assert L.csa2_index_topk(ctypes.byref(fake), 1, 16, 10, 16, 16, 8, 7, 8, 0, None, 16, None, None,
                             None, 0, None) == 1
    assert L.csa2_index_topk(ctypes.byref(fake), 1, 16, 10, 16, 16, 8, 0, 8, 0, None, 16, None, None,
                             None, 0, None) == 3
    assert L.csa2_index_topk(ctypes.byref(fake), 1, 16, 10, 16, 16, 8, 2, 8, 16, None, 16, None, None,
                             256, 1 << 20, None) == 1  # POOL without pool_in
    assert L.csa2_index_topk(ctypes.byref(fake), 1, 16, 10, 16, 16, 8, 1, 4, 16, None, 16, None, None,
                             256, 1 << 20, None) == 2  # block != 8
    assert L.csa2_cache_write(16, 64, 5120, 16, 16, 16, 3, ctypes.byref(fake), 0, 0, None, 0, 256,
                              1 << 30, None) == 2  # m = 3
    assert L.csa2_sparse_attn_decode(ctypes.byref(fake), 1, 16, 512, 16, 129, 16, 1.0, None, None, None, None,
                                     16, None, 256, 1 << 30, None) == 1  # n_swa > 128
    for bad_scale in (0.0, -0.04, float("inf"), float("nan")):  # the softmax scale must be positive, finite
        assert L.csa2_sparse_attn_decode(ctypes.byref(fake), 1, 16, 512, 16, 128, 16, bad_scale, None, None,
                                         None, None, 16, None, 256, 1 << 30, None) == 1
    # RoPE of the query needs the positions; a base <= 1 and a negative eps are rejected
    nr = csa2.NormRope(None, 1e-6, 1, 10000.0)
    assert L.csa2_sparse_attn_decode(ctypes.byref(fake), 1, 16, 512, 16, 128, 16, 0.04, ctypes.byref(nr),
                                     None, None, None, 16, None, 256, 1 << 30, None) == 1
    for bad in (csa2.NormRope(None, 1e-6, 1, 1.0), csa2.NormRope(None, -1.0, 0, 10000.0),
                csa2.NormRope(4, 1e-6, 0, 10000.0)):  # misaligned weight
        assert L.csa2_sparse_attn_decode(ctypes.byref(fake), 1, 16, 512, 16, 128, 16, 0.04, ctypes.byref(bad),
                                         16, None, None, 16, None, 256, 1 << 30, None) == 1
        assert L.csa2_cache_write(16, 64, 5120, 16, 16, 16, 2, ctypes.byref(fake), 0, 0, ctypes.byref(bad), 0,
                                  256, 1 << 30, None) == 1


def test_pool_stage_validation_without_gpu(L):
    fake = csa2.KVPlanes(16, 16, 32, 16, 100)  # aligned non-null pointers, never dereferenced
    vp = ctypes.c_void_p
    # csa2_pool_stage: missing pool, block != 8, pool larger than 16,384 entries, misaligned codes
    assert L.csa2_pool_stage(ctypes.byref(fake), 1, 16, 100, 8, 4, None, vp(64), vp(64), None) == 1
    assert L.csa2_pool_stage(ctypes.byref(fake), 1, 16, 100, 4, 4, vp(16), vp(64), vp(64), None) == 2
    assert L.csa2_pool_stage(ctypes.byref(fake), 1, 16, 100, 8, 2049, vp(16), vp(64), vp(64), None) == 1
    assert L.csa2_pool_stage(ctypes.byref(fake), 1, 16, 100, 8, 4, vp(16), vp(48), vp(64), None) == 1
    assert L.csa2_pool_stage(ctypes.byref(fake), 1, 16, 101, 8, 4, vp(16), vp(64), vp(64), None) == 1  # n_max > stride
    # csa2_index_topk_staged: k = 0, no pool, block != 8, no workspace, a workspace too small
    args = lambda k=8, pool=16, block=8, ws=None, nb=0: (vp(64), vp(64), 1, vp(16), 100, vp(16), vp(16), k, block,
                                                         4, vp(pool) if pool else None, vp(16), None,
                                                         vp(ws) if ws else None, nb, None)
    assert L.csa2_index_topk_staged(*args(k=0)) == 1
    assert L.csa2_index_topk_staged(*args(pool=0)) == 1
    assert L.csa2_index_topk_staged(*args(block=4)) == 2
    assert L.csa2_index_topk_staged(*args()) == 3
    assert L.csa2_index_topk_staged(*args(ws=256, nb=512)) == 3
    # a workspace sized for csa2_index_topk is enough (more than the staged call needs)
    full = L.csa2_index_topk_workspace_size(1, 100, 8, 8, 4)
    assert full > 0


def test_v4_compressor_and_dense_validation_without_gpu(L):
    fake = csa2.KVPlanes(16, 16, 16, 16, 100)
    args = (16, 16, 16, 16, 16, 16)  # Wa_kv, Wb_kv, Wa_z, Wb_z, Ba, Bb
    ws = csa2.compress_workspace_size(8, 64)
    assert L.csa2_compress_overlap(16, 10, 64, *args, 4, 512, 16, 256, ws, None) == 2      # T % m != 0
    assert L.csa2_compress_overlap(16, 8, 96, *args, 4, 512, 16, 256, ws, None) == 2       # d % 64 != 0
    assert L.csa2_compress_overlap(16, 8, 64, *args, 0, 512, 16, 256, ws, None) == 1       # m < 1
    assert L.csa2_compress_overlap(16, 8, 64, *args, 4, 512, None, 256, ws, None) == 1     # no output
    assert L.csa2_compress_overlap(16, 8, 64, 16, 16, 16, 16, None, 16, 4, 512, 16, 256, ws, None) == 1
    assert L.csa2_compress_overlap(16, 8, 64, *args, 4, 512, 16, 256, ws - 1, None) == 3   # workspace short
    assert L.csa2_compress_overlap(16, 8, 64, *args, 4, 512, 16, 128, ws, None) == 3       # misaligned ws
    assert L.csa2_compress_hca(16, 256, 64, 16, 16, 16, 128, 512, 16, 256, ws, None) == 3
    assert L.csa2_compress_hca(16, 200, 64, 16, 16, 16, 128, 512, 16, 256, 1 << 30, None) == 2
    assert L.csa2_compress_hca(16, 256, 64, 8, 16, 16, 128, 512, 16, 256, 1 << 30, None) == 1  # misaligned W
    assert csa2.compress_workspace_size(65536, 4096) >= 4 * 65536 * 512 * 4
    for bad_width in (0, 64, 640, 200):  # a multiple of 128, at most 512
        assert L.csa2_compress_hca(16, 256, 64, 16, 16, 16, 128, bad_width, 16, 256, 1 << 30, None) == 2
    # dense attention: n_max beyond the slot or the limit, no counts, bad scale
    assert L.csa2_dense_attn_decode(ctypes.byref(fake), 1, 16, 101, None, 0, 16, 0.04, None, None, None, None, 16,
                                    None, 256, 1 << 30, None) == 1
    big = csa2.KVPlanes(16, 16, 16, 16, 1 << 20)
    assert L.csa2_dense_attn_decode(ctypes.byref(big), 1, 16, 65537, None, 0, 16, 0.04, None, None, None, None, 16,
                                    None, 256, 1 << 30, None) == 1
    assert L.csa2_dense_attn_decode(ctypes.byref(fake), 1, None, 50, None, 0, 16, 0.04, None, None, None, None, 16,
                                    None, 256, 1 << 30, None) == 1
    assert L.csa2_dense_attn_decode(ctypes.byref(fake), 1, 16, 50, None, 0, 16, -1.0, None, None, None, None, 16,
                                    None, 256, 1 << 30, None) == 1
    assert L.csa2_dense_attn_decode(ctypes.byref(fake), 1, 16, 50, None, 0, 16, 0.04, None, None, None, None, 16,
                                    None, 256, 16, None) == 3
    assert csa2.dense_attn_workspace_size(1, 8192, 128) > csa2.dense_attn_workspace_size(1, 0, 128) > 0
    # window bounds need both arrays, 8-byte aligned
    for bad_win in (csa2.Window(None, 16), csa2.Window(16, None), csa2.Window(12, 16)):
        assert L.csa2_sparse_attn_decode(ctypes.byref(fake), 1, 16, 512, 16, 128, 16, 0.04, None, None, None,
                                         ctypes.byref(bad_win), 16, None, 256, 1 << 30, None) == 1


def test_workspace_queries(L):
    assert csa2.index_topk_workspace_size(32, 1 << 20, 512, 8, 2048) >= 32 * (1 << 20) * 4
    assert csa2.sparse_attn_workspace_size(32, 512, 128) > 0
    assert csa2.cache_write_workspace_size(131072, 5120, 2) >= 65536 * 640 * 4


def test_flat_workspace_holds_the_pool_from_65536_entries():
    """FLAT over 65,536 entries or more selects through a pool of k blocks, so its
    workspace (the same query as every mode's) holds B x k pool ids from there on."""
    B, k = 128, 512
    below = csa2.index_topk_workspace_size(B, 65535, k)
    at = csa2.index_topk_workspace_size(B, 65536, k)
    assert at - below >= B * k * 4
    # a HIER_BUILD workspace with a larger pool already covers it
    assert csa2.index_topk_workspace_size(B, 65536, k, 8, 2048) >= at


def test_prefill_workspace_budget():
    """The prefill indexer's batches hold the scores, the block maxima and the pools of as
    many queries as fit about 1.25 GiB: 2,048 queries over 131,072 entries in one batch,
    and at least one query whatever the slot."""
    one = csa2.index_topk_prefill_workspace_size(2048, 131072, 512)
    per_query = (131072 + 131072 // 8 + 512) * 4
    assert one >= 2048 * per_query
    assert one <= (5 << 28) + 64 * 1024
    # a 2^24-entry slot: batches of 17 queries
    big = csa2.index_topk_prefill_workspace_size(40, 1 << 24, 512)
    assert 17 * ((1 << 24) + (1 << 21) + 512) * 4 <= big <= (5 << 28) + 64 * 1024
    # shorter slots keep no maxima or pools
    assert csa2.index_topk_prefill_workspace_size(100, 4224, 512) < 100 * 4288 * 4 + 64 * 1024


def test_kernel_timing_switch_without_gpu(L):
    """Switching timing on and off and reading totals touch no device when
    nothing was launched: no totals, status ok."""
    csa2.timing_enable(True)
    assert csa2.kernel_times() == {}
    csa2.timing_enable(False)
    assert csa2.kernel_times() == {}
