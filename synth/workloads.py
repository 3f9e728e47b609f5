"""Workload recipes: shapes, seeds, tensor ids and value distributions.

Each workload mirrors one decode or prefill configuration of the CSA2 design
(DeepSeek-V4.1-Flash: pushing the limits of KV cache compression, setup list and
section 4): 512-channel main-KV latents, 128-d indexer keys, 32 indexer heads,
64 attention heads of dimension 512, top-512 selection, a 128-row sliding
window.  Only random draws and their shapes live here.

Tensor ids (the generator's stream id per role):
    main latents of the KV owned by Full layer f ..... 1 + 64*f
    indexer-key latents of Full layer f .............. 2 + 64*f
    hot-entry draw of Full layer f ................... 3 + 64*f
    indexer query q^I of indexing layer l ............ 4 + 64*l
    indexer head weights w of indexing layer l ....... 5 + 64*l
    attention query q of layer l ..................... 6 + 64*l
    sliding-window rows of layer l ................... 7 + 64*l
    cache-write H, W_KV, W_Z, W_IK ................... 8, 9, 10, 11
    V4 two-path compressor W_aKV, W_bKV, W_aZ, W_bZ .. 12, 13, 14, 15
    V4 position biases B^a, B^b, HCA B ............... 16, 17, 18
Seeds: workload c uses seed c.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from . import bf16_to_f32, e4m3_normal, keys_f32, normal_bf16, normal_f32, uniform_f32

D_MAIN = 512      # main-KV latent channels
D_IDX = 128       # indexer head dimension
H_IDX = 32        # indexer heads
H_ATT = 64        # attention query heads
TOPK = 512
N_SWA = 128
BLOCK = 8
N_BLOCKS_KEEP = 2048


def tid_main(f): return 1 + 64 * f
def tid_index(f): return 2 + 64 * f
def tid_hot(f): return 3 + 64 * f
def tid_qidx(l): return 4 + 64 * l
def tid_w(l): return 5 + 64 * l
def tid_q(l): return 6 + 64 * l
def tid_swa(l): return 7 + 64 * l


TID_H, TID_WKV, TID_WZ, TID_WIK = 8, 9, 10, 11


@dataclass
class DecodeWorkload:
    name: str
    seed: int
    B: int
    N: int                      # entries per sequence (context / m)
    mode: str                   # "flat" or "hier"
    n_attn: int = 1             # attention passes sharing one index pass (Full + Reuse)
    hot_prob: float = 0.0
    hot_gain: float = 3.0
    k: int = TOPK
    n_swa: int = N_SWA
    softmax_scale: float = 1.0 / math.sqrt(D_MAIN)
    extra: dict = field(default_factory=dict)


# the decode workloads (cache write and the 40-layer step are described separately)
SINGLE_4K = DecodeWorkload("single query, one Full layer, 4,096 entries", 0, 1, 4096, "flat")
ENCODER_B64 = DecodeWorkload("batch 64, encoder Full at m=2, 32,768 entries, 1 index + 6 attention",
                             1, 64, 32768, "flat", n_attn=6)
DECODER_1M = DecodeWorkload("batch 32, decoder Full at m=1, 1,048,576 entries, hierarchical",
                            2, 32, 1 << 20, "hier", hot_prob=0.02)


@dataclass
class CacheWriteWorkload:
    name: str
    seed: int
    T: int
    d_model: int
    m: int


PREFILL_128K = CacheWriteWorkload("prefill cache write, 131,072 tokens, d=5120, m=2", 3, 131072,
                                  5120, 2)


@dataclass
class ScheduleWorkload:
    name: str
    seed: int
    B: int
    context: int


STEP_256K = ScheduleWorkload("40-layer decode step, batch 128, 262,144-token context", 4, 128,
                             262144)


# ----------------------------------------------------------------------------- small host draws

def index_query(seed: int, layer: int, B: int):
    """q^I bf16 bits [B,32,128] ~ N(0,1) and head weights w fp32 [B,32] ~ U(0,1)."""
    q = normal_bf16(seed, tid_qidx(layer), B * H_IDX * D_IDX).reshape(B, H_IDX, D_IDX)
    w = uniform_f32(seed, tid_w(layer), B * H_IDX).reshape(B, H_IDX)
    return q, w


def attn_query(seed: int, layer: int, B: int) -> np.ndarray:
    """Attention query bf16 bits [B,64,512] ~ N(0,1) (unscaled)."""
    return normal_bf16(seed, tid_q(layer), B * H_ATT * D_MAIN).reshape(B, H_ATT, D_MAIN)


def swa_rows(seed: int, layer: int, B: int, n_swa: int = N_SWA) -> np.ndarray:
    """Sliding-window rows as FP8 E4M3 bytes [B,n_swa,512] of N(0,1)."""
    return e4m3_normal(seed, tid_swa(layer), B * n_swa * D_MAIN).reshape(B, n_swa, D_MAIN)


def hot_vectors(q_bits: np.ndarray, w: np.ndarray, gain: float) -> np.ndarray:
    """Per-sequence hot direction: gain * normalize(sum_h w_h q_h), fp64 then fp32.

    Summation runs sequentially over heads and dimensions so that every machine
    produces the same bits.  Shape [B,128] fp32.
    """
    q = bf16_to_f32(q_bits).astype(np.float64)
    B = q.shape[0]
    out = np.empty((B, q.shape[2]), np.float32)
    for b in range(B):
        acc = np.zeros(q.shape[2], np.float64)
        for h in range(q.shape[1]):
            acc = acc + float(w[b, h]) * q[b, h]
        ss = 0.0
        for v in acc.tolist():
            ss += v * v
        nrm = math.sqrt(ss)
        out[b] = (acc * (gain / nrm)).astype(np.float32)
    return out


def main_latents(seed: int, f: int, B: int, N: int, b: int, j0: int, count: int) -> np.ndarray:
    """Main-KV latents fp32 [count,512] ~ N(0,1) of entries j0.. of sequence b."""
    off = (b * N + j0) * D_MAIN
    return normal_f32(seed, tid_main(f), count * D_MAIN, offset=off).reshape(count, D_MAIN)


def index_latents(seed: int, f: int, B: int, N: int, b: int, j0: int, count: int,
                  hot_prob: float = 0.0, hotvec: np.ndarray | None = None) -> np.ndarray:
    """Indexer-key latents fp32 [count,128] of entries j0.. of sequence b (hot mixture)."""
    off = (b * N + j0) * D_IDX
    return keys_f32(seed, tid_index(f), tid_hot(f), count * D_IDX, D_IDX, offset=off,
                    hot_prob=hot_prob, hotvec=hotvec).reshape(count, D_IDX)


def cache_write_inputs(seed: int, T: int, d_model: int, t0: int = 0):
    """H bf16 [T,d] ~ N(0,1); W_KV, W_Z bf16 [d,512] ~ N(0,1/d); W_IK bf16 [512,128] ~ N(0,1/512)."""
    H = normal_bf16(seed, TID_H, T * d_model, offset=t0 * d_model).reshape(T, d_model)
    sd = np.float32(1.0 / math.sqrt(d_model))
    Wkv = normal_bf16(seed, TID_WKV, d_model * D_MAIN, scale=float(sd)).reshape(d_model, D_MAIN)
    Wz = normal_bf16(seed, TID_WZ, d_model * D_MAIN, scale=float(sd)).reshape(d_model, D_MAIN)
    sk = np.float32(1.0 / math.sqrt(D_MAIN))
    Wik = normal_bf16(seed, TID_WIK, D_MAIN * D_IDX, scale=float(sk)).reshape(D_MAIN, D_IDX)
    return H, Wkv, Wz, Wik


TID_WA_KV, TID_WB_KV, TID_WA_Z, TID_WB_Z = 12, 13, 14, 15
TID_BA, TID_BB, TID_BHCA = 16, 17, 18
BIAS_SD = 0.5     # position-bias draw N(0, 0.5^2)


def overlap_compressor_inputs(seed: int, T: int, d_model: int, m: int, t0: int = 0):
    """H bf16 [T,d] ~ N(0,1); W_aKV, W_bKV, W_aZ, W_bZ bf16 [d,512] ~ N(0,1/d);
    B^a, B^b fp32 [m,512] ~ N(0, 0.5^2)."""
    H = normal_bf16(seed, TID_H, T * d_model, offset=t0 * d_model).reshape(T, d_model)
    sd = float(np.float32(1.0 / math.sqrt(d_model)))
    Ws = [normal_bf16(seed, t, d_model * D_MAIN, scale=sd).reshape(d_model, D_MAIN)
          for t in (TID_WA_KV, TID_WB_KV, TID_WA_Z, TID_WB_Z)]
    Ba = normal_f32(seed, TID_BA, m * D_MAIN, scale=BIAS_SD).reshape(m, D_MAIN)
    Bb = normal_f32(seed, TID_BB, m * D_MAIN, scale=BIAS_SD).reshape(m, D_MAIN)
    return (H, *Ws, Ba, Bb)


def hca_compressor_inputs(seed: int, T: int, d_model: int, m: int, t0: int = 0):
    """H bf16 [T,d] ~ N(0,1); W_KV, W_Z bf16 [d,512] ~ N(0,1/d); B fp32 [m,512] ~ N(0, 0.5^2)."""
    H, Wkv, Wz, _ = cache_write_inputs(seed, T, d_model, t0)
    Bp = normal_f32(seed, TID_BHCA, m * D_MAIN, scale=BIAS_SD).reshape(m, D_MAIN)
    return H, Wkv, Wz, Bp
