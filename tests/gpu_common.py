"""Shared setup of the GPU parity tests: same seeded latents on both sides, each
side encoding them with its own codec."""
from __future__ import annotations

import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import compressed_sparse_attention_nvfp4_gb300 as csa2  # noqa: E402
from synth import workloads as W  # noqa: E402


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(csa2.LIB_PATH):
        from compressed_sparse_attention_nvfp4_gb300 import build

        build.build()
    import synth

    if not os.path.exists(synth.DEV_LIB):
        from synth import build as sb

        sb.build_dev()


def to_dev(a: np.ndarray, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


class SmallCache:
    """B slots of n_max entries: fp32 latents on the host, the oracle's planes,
    and the GPU planes encoded on the device from the same latents."""

    def __init__(self, oracle, seed, B, n_max, f=0, hot_prob=0.0, hotvecs=None, stride=None):
        self.B, self.n_max = B, n_max
        stride = stride or n_max
        self.main = np.concatenate([W.main_latents(seed, f, B, n_max, b, 0, n_max) for b in range(B)])
        self.idx = np.concatenate([
            W.index_latents(seed, f, B, n_max, b, 0, n_max, hot_prob,
                            None if hotvecs is None else hotvecs[b]) for b in range(B)])
        self.o_kvc, self.o_kvs = oracle.quantize_main(self.main)
        self.o_ixc, self.o_ixs = oracle.quantize_index(self.idx)
        self.planes = csa2.Planes.empty(B, stride)
        cb = torch.zeros((B * stride, 512), dtype=torch.float32, device="cuda")
        ki = torch.zeros((B * stride, 128), dtype=torch.float32, device="cuda")
        for b in range(B):
            cb[b * stride:b * stride + n_max] = to_dev(self.main[b * n_max:(b + 1) * n_max])
            ki[b * stride:b * stride + n_max] = to_dev(self.idx[b * n_max:(b + 1) * n_max])
        csa2.quantize_entries(self.planes, cb, ki, B * stride, 0)
        torch.cuda.synchronize()
        self.stride = stride

    def oracle_slot(self, b):
        s = slice(b * self.n_max, (b + 1) * self.n_max)
        return self.o_kvc[s], self.o_kvs[s], self.o_ixc[s], self.o_ixs[s]

    def gpu_slot(self, b):
        s = slice(b * self.stride, b * self.stride + self.n_max)
        p = self.planes
        return (p.kv_codes[s].cpu().numpy(), p.kv_scales[s].cpu().numpy(),
                p.ix_codes[s].cpu().numpy(), p.ix_scales[s].cpu().numpy())
