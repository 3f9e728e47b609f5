"""One decode step over the V4.1-Flash 40-layer schedule, dispatched through the C ABI.

The layer table comes from the library (``csa2_v41_layer_table``): layers 0-1
attend only to their sliding window; Full layers {2, 8, 14, 20} own a global KV
and run the indexer (the encoder's at m=2 with a flat top-k, the decoder's at
m=1 with the hierarchical pool); Reindex layers {24, 28, 32, 36} re-score the
decoder Full layer's pool with their own query (the pool's indexer keys are
gathered once, right after the pool is built, and every Reindex layer scans
that staged copy); Reuse layers take the top-k of
the nearest Full/Reindex layer.  Every layer runs its own 64-head attention over
its top-k entries of the KV it shares plus its own window
("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression", sections 2,
4.2 and 4.3; "DeepSeek-V4.1-Flash course, 02 Architecture", 2.3.1 and 2.3.2).

This module only decides which call each layer makes; the work runs in the
library's kernels on the caller's stream, so a step can be captured in a CUDA
graph.
"""
from __future__ import annotations

from dataclasses import dataclass, field

from . import (LAYER_FULL, LAYER_REINDEX, LAYER_REUSE, LAYER_SWA, TOPK_FLAT, TOPK_HIER_BUILD,
               Planes, PoolStage, index_topk, index_topk_staged, index_topk_workspace_size, pool_stage,
               sparse_attn_decode, sparse_attn_workspace_size, v41_layer_table, workspace)


@dataclass
class StepBuffers:
    """Device tensors of one decode step.

    kv[f]       Planes of Full layer f (f in the table's Full layers)
    n_entries[f] int32 [B] visible entries of that KV; n_max[f] its host bound
    qidx[l], w[l] indexer query / head weights of Full and Reindex layers
    q[l], swa[l]  attention query and window rows of every layer
    out[l]        fp32 [B, 64, 512] output of every layer
    """
    B: int
    kv: dict
    n_entries: dict
    n_max: dict
    qidx: dict
    w: dict
    q: dict
    swa: dict
    out: dict
    n_swa: int = 128
    k: int = 512
    block: int = 8
    n_blocks_keep: int = 2048
    softmax_scale: float = 512 ** -0.5
    topk: dict = field(default_factory=dict)
    pool: dict = field(default_factory=dict)
    stage: dict = field(default_factory=dict)
    ws_index: object = None
    ws_attn: object = None


def allocate_scratch(buf: StepBuffers, device="cuda") -> None:
    """Top-k / pool outputs and workspaces of a step (allocated once, reused)."""
    import torch

    t = v41_layer_table()
    n_max_all = max(buf.n_max.values())
    for l in range(40):
        if t["mode"][l] in (LAYER_FULL, LAYER_REINDEX):
            buf.topk[l] = torch.empty((buf.B, buf.k), dtype=torch.int32, device=device)
        if t["mode"][l] == LAYER_FULL and t["m"][l] == 1:
            buf.pool[l] = torch.empty((buf.B, buf.n_blocks_keep), dtype=torch.int32, device=device)
            if any(t["pool_src"][r] == l for r in range(40) if t["mode"][r] == LAYER_REINDEX):
                buf.stage[l] = PoolStage.empty(buf.B, buf.n_blocks_keep, buf.block, device)
    buf.ws_index = workspace(index_topk_workspace_size(buf.B, n_max_all, buf.k, buf.block,
                                                       buf.n_blocks_keep), device)
    buf.ws_attn = workspace(sparse_attn_workspace_size(buf.B, buf.k, buf.n_swa), device)


def run_step(buf: StepBuffers, stream=None) -> int:
    """Issues the 40 layers' calls in order; returns the number of library calls."""
    t = v41_layer_table()
    calls = 0
    for l in range(40):
        mode = t["mode"][l]
        if mode == LAYER_SWA:
            # no global branch: attention over the window alone (k = 0)
            any_kv = next(iter(buf.kv.values()))
            sparse_attn_decode(any_kv, buf.B, None, 0, buf.swa[l], buf.n_swa, buf.q[l], buf.softmax_scale,
                               buf.out[l], buf.ws_attn, stream=stream)
            calls += 1
            continue
        f = t["kv_src"][l]
        kv, ne, nm = buf.kv[f], buf.n_entries[f], buf.n_max[f]
        if mode == LAYER_FULL:
            if t["m"][l] == 1:  # the decoder's first Full layer builds the candidate pool
                index_topk(kv, buf.B, ne, nm, buf.qidx[l], buf.w[l], buf.k, TOPK_HIER_BUILD, buf.topk[l],
                           buf.ws_index, buf.block, buf.n_blocks_keep, pool_out=buf.pool[l],
                           stream=stream)
                if l in buf.stage:  # one gather of the pool's keys serves every Reindex layer
                    pool_stage(kv, buf.B, ne, nm, buf.pool[l], buf.stage[l], buf.block, buf.n_blocks_keep,
                               stream=stream)
                    calls += 1
            else:
                index_topk(kv, buf.B, ne, nm, buf.qidx[l], buf.w[l], buf.k, TOPK_FLAT, buf.topk[l],
                           buf.ws_index, stream=stream)
            calls += 1
        elif mode == LAYER_REINDEX:
            p = t["pool_src"][l]
            index_topk_staged(buf.stage[p], buf.B, ne, nm, buf.qidx[l], buf.w[l], buf.k, buf.pool[p],
                              buf.topk[l], buf.ws_index, buf.block, buf.n_blocks_keep, stream=stream)
            calls += 1
        topk = buf.topk[t["topk_src"][l]]
        sparse_attn_decode(kv, buf.B, topk, buf.k, buf.swa[l], buf.n_swa, buf.q[l], buf.softmax_scale,
                           buf.out[l], buf.ws_attn, stream=stream)
        calls += 1
    return calls


def capture_step(buf: StepBuffers, stream):
    """A CUDA graph of one run_step on `stream` (a torch stream): replaying it issues the
    step's kernels with no host work per call.  The buffers stay bound to the graph."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        run_step(buf, stream=stream)  # warm: attributes set and maps built outside the capture
        torch.cuda.current_stream().synchronize()
        with torch.cuda.graph(g, stream=stream):
            run_step(buf, stream=stream)
    return g
