"""Device-resident inputs of the decode and cache-write workloads.

Latents are drawn by the seeded generator (``synth``) directly in device
memory and encoded into the cache planes by the library's own codec
(``csa2_quantize_entries``), chunk by chunk, so multi-gigabyte caches are built
without host traffic.  Small per-query tensors (q^I, w, q) are drawn on the host
and uploaded; sliding-window rows are drawn on the device.
"""
from __future__ import annotations

import numpy as np
import torch

import synth
from synth import workloads as W

from . import Planes, quantize_entries


def fill_planes(planes: Planes, seed: int, f: int, B: int, N: int, hot_prob: float = 0.0,
                hotvecs: np.ndarray | None = None, chunk: int = 1 << 18, stream=None) -> None:
    """Entries 0..N-1 of slots 0..B-1 of `planes` from the latents of Full layer f."""
    dev = planes.kv_codes.device
    st = (stream or torch.cuda.current_stream()).cuda_stream
    cnt_max = min(chunk, N)
    cbar = torch.empty((cnt_max, W.D_MAIN), dtype=torch.float32, device=dev)
    ki = torch.empty((cnt_max, W.D_IDX), dtype=torch.float32, device=dev)
    hv = None
    if hotvecs is not None:
        hv = torch.from_numpy(np.ascontiguousarray(hotvecs, np.float32)).to(dev)
    for b in range(B):
        for j0 in range(0, N, chunk):
            cnt = min(chunk, N - j0)
            synth.dev_normal_f32(seed, W.tid_main(f), cnt * W.D_MAIN, cbar.data_ptr(), st,
                                 offset=(b * N + j0) * W.D_MAIN)
            synth.dev_keys_f32(seed, W.tid_index(f), W.tid_hot(f), cnt * W.D_IDX, W.D_IDX,
                               ki.data_ptr(), st, offset=(b * N + j0) * W.D_IDX,
                               hot_prob=hot_prob if hv is not None else 0.0,
                               hotvec_ptr=None if hv is None else hv[b].data_ptr())
            quantize_entries(planes, cbar, ki, cnt, e0=b * planes.seq_stride + j0, stream=st)


def upload(a: np.ndarray, device="cuda", dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device)


def index_query_dev(seed: int, layer: int, B: int, device="cuda"):
    q, w = W.index_query(seed, layer, B)
    return upload(q.view(np.int16), device), upload(w, device), q, w


def attn_query_dev(seed: int, layer: int, B: int, device="cuda"):
    q = W.attn_query(seed, layer, B)
    return upload(q.view(np.int16), device), q


def swa_dev(seed: int, layer: int, B: int, n_swa: int = W.N_SWA, device="cuda", stream=None):
    t = torch.empty((B, n_swa, W.D_MAIN), dtype=torch.uint8, device=device)
    st = (stream or torch.cuda.current_stream()).cuda_stream
    synth.dev_e4m3_normal(seed, W.tid_swa(layer), B * n_swa * W.D_MAIN, t.data_ptr(), st)
    return t
