"""CSA2 oracle -- TEST INFRASTRUCTURE ONLY.

ctypes wrapper over ``csa2_oracle.c``, the plain CPU restatement of the CSA2
decode path and cache writer (fp64 except where the cache format fixes fp32).
Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library.

Parity status of each function (what pins it independently of itself) is in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(_HERE, "libcsa2oracle.so")
_lib = None

D_MAIN, D_IDX, H_IDX, H_ATT = 512, 128, 32, 64


def _load():
    global _lib
    if _lib is None:
        src = os.path.join(os.path.dirname(LIB), "csa2_oracle.c")
        if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(src):
            from . import build as _b

            _b.build()
        lib = ctypes.CDLL(LIB)
        vp, i64, i32, f32, f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                  ctypes.c_double)
        lib.o_e2m1_value.argtypes = [ctypes.c_int]
        lib.o_e2m1_value.restype = f64
        lib.o_e2m1_encode.argtypes = [f32]
        lib.o_e2m1_encode.restype = ctypes.c_int
        lib.o_e4m3_value.argtypes = [ctypes.c_int]
        lib.o_e4m3_value.restype = f64
        lib.o_e4m3_encode.argtypes = [f32]
        lib.o_e4m3_encode.restype = ctypes.c_int
        lib.o_e8m0_value.argtypes = [ctypes.c_int]
        lib.o_e8m0_value.restype = f64
        for f in ("o_quantize_main", "o_quantize_index", "o_dequant_main", "o_dequant_index"):
            getattr(lib, f).argtypes = [vp, i64, vp, vp] if "quantize" in f and "de" not in f \
                else [vp, vp, i64, vp]
            getattr(lib, f).restype = None
        lib.o_main_group_margin.argtypes = [vp]
        lib.o_main_group_margin.restype = f64
        lib.o_index_group_margin.argtypes = [vp]
        lib.o_index_group_margin.restype = f64
        lib.o_cache_write.argtypes = [vp, i64, ctypes.c_int, vp, vp, vp, ctypes.c_int, vp, vp, vp,
                                      vp, vp, vp, ctypes.c_int, vp, f64, ctypes.c_int, f64, f64, f64, vp]
        lib.o_cache_write.restype = ctypes.c_int
        lib.o_pool.argtypes = [vp, vp, i64, ctypes.c_int, ctypes.c_int, vp]
        lib.o_pool.restype = None
        lib.o_index_scores.argtypes = [vp, vp, i64, vp, vp, vp, ctypes.c_int]
        lib.o_index_scores.restype = None
        lib.o_index_scores_at.argtypes = [vp, vp, vp, i64, vp, vp, vp]
        lib.o_index_scores_at.restype = None
        lib.o_topk.argtypes = [vp, i64, ctypes.c_int, vp]
        lib.o_topk.restype = ctypes.c_int
        lib.o_block_max.argtypes = [vp, i64, ctypes.c_int, vp]
        lib.o_block_max.restype = None
        lib.o_hier_pool.argtypes = [vp, i64, ctypes.c_int, vp]
        lib.o_hier_pool.restype = ctypes.c_int
        lib.o_pool_topk.argtypes = [vp, i64, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
        lib.o_pool_topk.restype = ctypes.c_int
        lib.o_attention.argtypes = [vp, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, f64, vp, vp]
        lib.o_attention.restype = None
        lib.o_attention_ex.argtypes = [vp, vp, vp, ctypes.c_int, vp, ctypes.c_int, vp, f64, vp, f64,
                                       ctypes.c_int, f64, f64, vp, vp, vp]
        lib.o_attention_ex.restype = None
        lib.o_attention_rows.argtypes = [vp, ctypes.c_int, vp, f64, vp, f64, ctypes.c_int, f64, f64,
                                         vp, vp, vp]
        lib.o_attention_rows.restype = None
        lib.o_rmsnorm.argtypes = [vp, ctypes.c_int, vp, f64, vp]
        lib.o_rmsnorm.restype = None
        lib.o_rope.argtypes = [vp, f64, f64]
        lib.o_rope.restype = None
        lib.o_swa_row.argtypes = [vp, vp, f64, ctypes.c_int, f64, f64, vp, vp]
        lib.o_swa_row.restype = None
        lib.o_project.argtypes = [vp, i64, ctypes.c_int, ctypes.c_int, vp, vp, ctypes.c_int]
        lib.o_project.restype = None
        lib.o_pool_overlap.argtypes = [vp, vp, vp, vp, vp, vp, i64, ctypes.c_int, ctypes.c_int, vp]
        lib.o_pool_overlap.restype = None
        lib.o_pool_bias.argtypes = [vp, vp, vp, i64, ctypes.c_int, ctypes.c_int, vp]
        lib.o_pool_bias.restype = None
        lib.o_compress_overlap.argtypes = [vp, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                           ctypes.c_int, vp, ctypes.c_int]
        lib.o_compress_overlap.restype = ctypes.c_int
        lib.o_compress_hca.argtypes = [vp, i64, ctypes.c_int, ctypes.c_int, vp, vp, vp, ctypes.c_int, vp,
                                       ctypes.c_int]
        lib.o_compress_hca.restype = ctypes.c_int
        lib.o_e2m1_encode_array.argtypes = [vp, i64, vp]
        lib.o_e2m1_encode_array.restype = None
        lib.o_e4m3_encode_array.argtypes = [vp, i64, vp]
        lib.o_e4m3_encode_array.restype = None
        _lib = lib
    return _lib


def _p(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _threads() -> int:
    return max(1, min(128, os.cpu_count() or 1))


# ----------------------------------------------------------------------------- formats

def e2m1_value(code: int) -> float:
    return _load().o_e2m1_value(code)


def e2m1_encode(x: float) -> int:
    return _load().o_e2m1_encode(x)


def e2m1_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32).ravel()
    out = np.empty(x.shape[0], np.uint8)
    _load().o_e2m1_encode_array(_p(x), x.shape[0], _p(out))
    return out


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32).ravel()
    out = np.empty(x.shape[0], np.uint8)
    _load().o_e4m3_encode_array(_p(x), x.shape[0], _p(out))
    return out


def e4m3_value(b: int) -> float:
    return _load().o_e4m3_value(b)


def e4m3_encode(x: float) -> int:
    return _load().o_e4m3_encode(x)


def e8m0_value(b: int) -> float:
    return _load().o_e8m0_value(b)


# ----------------------------------------------------------------------------- quantizers

def quantize_main(x: np.ndarray):
    """fp32 [n,512] -> (codes u8 [n,256], scales u8 [n,32])."""
    x = np.ascontiguousarray(x, np.float32)
    n = x.shape[0]
    codes = np.zeros((n, 256), np.uint8)
    scales = np.zeros((n, 32), np.uint8)
    _load().o_quantize_main(_p(x), n, _p(codes), _p(scales))
    return codes, scales


def quantize_index(x: np.ndarray):
    """fp32 [n,128] -> (codes u8 [n,64], scales u8 [n,4])."""
    x = np.ascontiguousarray(x, np.float32)
    n = x.shape[0]
    codes = np.zeros((n, 64), np.uint8)
    scales = np.zeros((n, 4), np.uint8)
    _load().o_quantize_index(_p(x), n, _p(codes), _p(scales))
    return codes, scales


def dequant_main(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    n = codes.shape[0]
    out = np.empty((n, D_MAIN), np.float64)
    _load().o_dequant_main(_p(codes), _p(scales), n, _p(out))
    return out


def dequant_index(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.uint8)
    n = codes.shape[0]
    out = np.empty((n, D_IDX), np.float64)
    _load().o_dequant_index(_p(codes), _p(scales), n, _p(out))
    return out


def main_group_margins(x: np.ndarray) -> np.ndarray:
    """Relative distance of each 16-channel group to its nearest rounding decision point."""
    x = np.ascontiguousarray(np.asarray(x, np.float64).reshape(-1, 16))
    lib = _load()
    return np.array([lib.o_main_group_margin(_p(np.ascontiguousarray(r))) for r in x])


def index_group_margins(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, np.float64).reshape(-1, 32))
    lib = _load()
    return np.array([lib.o_index_group_margin(_p(np.ascontiguousarray(r))) for r in x])


# ----------------------------------------------------------------------------- cache write

def cache_write(H: np.ndarray, Wkv: np.ndarray, Wz: np.ndarray, Wik: np.ndarray, m: int,
                return_prequant: bool = False, norm_weight=None, eps: float = 1e-6,
                rope: bool = False, rope_base: float = 10000.0, pos_first: float = 0.0,
                pos_step: float | None = None):
    """H bf16 bits [T,d]; W_KV, W_Z bf16 bits [d,512]; W_IK bf16 bits [512,128].

    Returns (kv_codes, kv_scales, ix_codes, ix_scales) for T/m entries and, if
    asked, the fp64 pooled latents Cbar [T/m,512] and indexer keys K^I [T/m,128],
    and the values the main quantizer saw [T/m,512].  norm_weight (fp32 [512] or
    None) and rope: RMSNorm / RoPE of the main-KV copy, entry j at position
    pos_first + j * pos_step (pos_step defaults to m).
    """
    H = np.ascontiguousarray(H, np.uint16)
    T, d = H.shape
    n = T // m
    kvc = np.zeros((n, 256), np.uint8)
    kvs = np.zeros((n, 32), np.uint8)
    ixc = np.zeros((n, 64), np.uint8)
    ixs = np.zeros((n, 4), np.uint8)
    cb = np.zeros((n, D_MAIN), np.float64) if return_prequant else None
    ki = np.zeros((n, D_IDX), np.float64) if return_prequant else None
    att = np.zeros((n, D_MAIN), np.float64) if return_prequant else None
    nw = None if norm_weight is None else np.ascontiguousarray(norm_weight, np.float32)
    rc = _load().o_cache_write(_p(H), T, d, _p(np.ascontiguousarray(Wkv, np.uint16)),
                               _p(np.ascontiguousarray(Wz, np.uint16)),
                               _p(np.ascontiguousarray(Wik, np.uint16)), m, _p(kvc), _p(kvs),
                               _p(ixc), _p(ixs), _p(cb), _p(ki), _threads(), _p(nw), float(eps),
                               int(bool(rope)), float(rope_base), float(pos_first),
                               float(m if pos_step is None else pos_step), _p(att))
    if rc != 0:
        raise ValueError("oracle cache_write: bad arguments")
    if return_prequant:
        return kvc, kvs, ixc, ixs, cb, ki, att
    return kvc, kvs, ixc, ixs


def pool(C: np.ndarray, Z: np.ndarray, m: int) -> np.ndarray:
    C = np.ascontiguousarray(C, np.float64)
    Z = np.ascontiguousarray(Z, np.float64)
    T, width = C.shape
    out = np.empty((T // m, width), np.float64)
    _load().o_pool(_p(C), _p(Z), T, width, m, _p(out))
    return out


# ----------------------------------------------------------------------------- V4 compressors

def _u16(a):
    return np.ascontiguousarray(a, np.uint16)


def _f32(a):
    return np.ascontiguousarray(a, np.float32)


def project(H: np.ndarray, W: np.ndarray) -> np.ndarray:
    """H bf16 bits [T,d] times W bf16 bits [d,width], fp64 sums: [T,width]."""
    H, W = _u16(H), _u16(W)
    T, d = H.shape
    out = np.empty((T, W.shape[1]), np.float64)
    _load().o_project(_p(H), T, d, W.shape[1], _p(W), _p(out), _threads())
    return out


def pool_overlap(Ca, Za, Cb, Zb, Ba, Bb, m: int) -> np.ndarray:
    """Two-path overlapping pool ("DeepSeek-V4 ...", CSA step 1): entry i takes
    rows [m i, m i + m) of (Ca, Za + Ba) and rows [m (i-1), m i) of (Cb, Zb + Bb),
    one per-channel softmax over the 2m scores; entry 0 only the first part.
    C*, Z* fp64 [T,width]; B* fp32 [m,width]."""
    Ca, Za, Cb, Zb = (np.ascontiguousarray(a, np.float64) for a in (Ca, Za, Cb, Zb))
    T, width = Ca.shape
    Ba, Bb = _f32(Ba), _f32(Bb)
    assert Ba.shape == (m, width) and Bb.shape == (m, width) and T % m == 0
    out = np.empty((T // m, width), np.float64)
    _load().o_pool_overlap(_p(Ca), _p(Za), _p(Cb), _p(Zb), _p(Ba), _p(Bb), T, width, m, _p(out))
    return out


def pool_bias(C, Z, Bp, m: int) -> np.ndarray:
    """HCA pool: entry i = per-channel softmax over rows [m i, m i + m) of Z + B."""
    C, Z = (np.ascontiguousarray(a, np.float64) for a in (C, Z))
    T, width = C.shape
    Bp = _f32(Bp)
    assert Bp.shape == (m, width) and T % m == 0
    out = np.empty((T // m, width), np.float64)
    _load().o_pool_bias(_p(C), _p(Z), _p(Bp), T, width, m, _p(out))
    return out


def compress_overlap(H, Wa_kv, Wb_kv, Wa_z, Wb_z, Ba, Bb, m: int) -> np.ndarray:
    """CSA step 1 end to end: [T/m, width] fp64 compressed entries of H (W_* [d, width])."""
    H = _u16(H)
    T, d = H.shape
    width = np.asarray(Wa_kv).shape[1]
    out = np.empty((T // m if m > 0 else 0, width), np.float64)
    rc = _load().o_compress_overlap(_p(H), T, d, width, _p(_u16(Wa_kv)), _p(_u16(Wb_kv)), _p(_u16(Wa_z)),
                                    _p(_u16(Wb_z)), _p(_f32(Ba)), _p(_f32(Bb)), m, _p(out), _threads())
    if rc != 0:
        raise ValueError("oracle compress_overlap: bad arguments")
    return out


def compress_hca(H, Wkv, Wz, Bp, m: int) -> np.ndarray:
    """HCA compressor end to end: [T/m, width] fp64 compressed entries of H (W [d, width])."""
    H = _u16(H)
    T, d = H.shape
    width = np.asarray(Wkv).shape[1]
    out = np.empty((T // m if m > 0 else 0, width), np.float64)
    rc = _load().o_compress_hca(_p(H), T, d, width, _p(_u16(Wkv)), _p(_u16(Wz)), _p(_f32(Bp)), m, _p(out),
                                _threads())
    if rc != 0:
        raise ValueError("oracle compress_hca: bad arguments")
    return out


# ----------------------------------------------------------------------------- indexer

def index_scores(ix_codes, ix_scales, q_bits, w, n=None, nthreads=None) -> np.ndarray:
    """Scores of entries 0..n-1.  q_bits bf16 [32,128]; w fp32 [32]."""
    ix_codes = np.ascontiguousarray(ix_codes, np.uint8)
    ix_scales = np.ascontiguousarray(ix_scales, np.uint8)
    n = ix_codes.shape[0] if n is None else n
    out = np.empty(n, np.float64)
    _load().o_index_scores(_p(ix_codes), _p(ix_scales), n,
                           _p(np.ascontiguousarray(q_bits, np.uint16)),
                           _p(np.ascontiguousarray(w, np.float32)), _p(out),
                           _threads() if nthreads is None else nthreads)
    return out


def index_scores_at(ix_codes, ix_scales, idx, q_bits, w) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.shape[0], np.float64)
    _load().o_index_scores_at(_p(np.ascontiguousarray(ix_codes, np.uint8)),
                              _p(np.ascontiguousarray(ix_scales, np.uint8)), _p(idx),
                              idx.shape[0], _p(np.ascontiguousarray(q_bits, np.uint16)),
                              _p(np.ascontiguousarray(w, np.float32)), _p(out))
    return out


def topk(scores: np.ndarray, k: int, n: int | None = None) -> np.ndarray:
    scores = np.ascontiguousarray(scores, np.float64)
    n = scores.shape[0] if n is None else n
    out = np.empty(k, np.int32)
    _load().o_topk(_p(scores), n, k, _p(out))
    return out


def block_max(scores: np.ndarray, blk: int, n: int | None = None) -> np.ndarray:
    scores = np.ascontiguousarray(scores, np.float64)
    n = scores.shape[0] if n is None else n
    out = np.empty((n + blk - 1) // blk, np.float64)
    _load().o_block_max(_p(scores), n, blk, _p(out))
    return out


def hier_pool(bmax: np.ndarray, keep: int) -> np.ndarray:
    bmax = np.ascontiguousarray(bmax, np.float64)
    out = np.empty(keep, np.int32)
    _load().o_hier_pool(_p(bmax), bmax.shape[0], keep, _p(out))
    return out


def pool_topk(scores: np.ndarray, pool_blocks: np.ndarray, blk: int, k: int,
              n: int | None = None) -> np.ndarray:
    scores = np.ascontiguousarray(scores, np.float64)
    n = scores.shape[0] if n is None else n
    pool_blocks = np.ascontiguousarray(pool_blocks, np.int32)
    out = np.empty(k, np.int32)
    _load().o_pool_topk(_p(scores), n, _p(pool_blocks), pool_blocks.shape[0], blk, k, _p(out))
    return out


# ----------------------------------------------------------------------------- attention

def attention(kv_codes, kv_scales, topk_idx, swa, q_bits, scale, q_norm_weight=None,
              eps: float = 1e-6, qpos=None, rope_base: float = 10000.0, sink=None):
    """One query: returns (out fp64 [64,512], lse fp64 [64]).

    q_norm_weight (fp32 [512]): RMSNorm of each query head; qpos: RoPE of the
    query at qpos and of the output at -qpos; sink (fp32 [64]): per-head sink
    logits in the softmax denominator.  Each is off when None.
    """
    topk_idx = np.ascontiguousarray(topk_idx, np.int32)
    swa = np.ascontiguousarray(swa, np.uint8).reshape(-1, D_MAIN)
    out = np.empty((H_ATT, D_MAIN), np.float64)
    lse = np.empty(H_ATT, np.float64)
    nw = None if q_norm_weight is None else np.ascontiguousarray(q_norm_weight, np.float32)
    sk = None if sink is None else np.ascontiguousarray(sink, np.float32)
    _load().o_attention_ex(_p(np.ascontiguousarray(kv_codes, np.uint8)),
                           _p(np.ascontiguousarray(kv_scales, np.uint8)), _p(topk_idx),
                           topk_idx.shape[0], _p(swa) if swa.size else None, swa.shape[0],
                           _p(np.ascontiguousarray(q_bits, np.uint16)), float(scale), _p(nw),
                           float(eps), int(qpos is not None), float(rope_base),
                           float(0.0 if qpos is None else qpos), _p(sk), _p(out), _p(lse))
    return out, lse


def attention_rows(X, q_bits, scale, q_norm_weight=None, eps: float = 1e-6, qpos=None,
                   rope_base: float = 10000.0, sink=None):
    """attention() over given fp64 rows X [rows,512] instead of cache entries."""
    X = np.ascontiguousarray(X, np.float64).reshape(-1, D_MAIN)
    out = np.empty((H_ATT, D_MAIN), np.float64)
    lse = np.empty(H_ATT, np.float64)
    nw = None if q_norm_weight is None else np.ascontiguousarray(q_norm_weight, np.float32)
    sk = None if sink is None else np.ascontiguousarray(sink, np.float32)
    _load().o_attention_rows(_p(X) if X.size else None, X.shape[0],
                             _p(np.ascontiguousarray(q_bits, np.uint16)), float(scale), _p(nw),
                             float(eps), int(qpos is not None), float(rope_base),
                             float(0.0 if qpos is None else qpos), _p(sk), _p(out), _p(lse))
    return out, lse


def rmsnorm(x, weight=None, eps: float = 1e-6) -> np.ndarray:
    """RMSNorm of each row of x (fp64) over its channels."""
    x = np.ascontiguousarray(x, np.float64)
    rows = x.reshape(-1, x.shape[-1])
    out = np.empty_like(rows)
    w = None if weight is None else np.ascontiguousarray(weight, np.float32)
    for i in range(rows.shape[0]):
        _load().o_rmsnorm(_p(np.ascontiguousarray(rows[i])), rows.shape[1], _p(w), float(eps),
                          _p(out[i:i + 1]))
    return out.reshape(x.shape)


def rope(x, pos: float, base: float = 10000.0) -> np.ndarray:
    """RoPE of the last 64 channels of each 512-channel row of x at position pos."""
    out = np.array(x, np.float64, copy=True).reshape(-1, D_MAIN)
    for i in range(out.shape[0]):
        row = np.ascontiguousarray(out[i])
        _load().o_rope(_p(row), float(pos), float(base))
        out[i] = row
    return out.reshape(np.shape(x))


def swa_row(x, norm_weight=None, eps: float = 1e-6, pos=None, rope_base: float = 10000.0):
    """One window row: (E4M3 bytes [512], the fp64 values before the encoding)."""
    x = np.ascontiguousarray(x, np.float64).reshape(D_MAIN)
    out = np.empty(D_MAIN, np.uint8)
    pre = np.empty(D_MAIN, np.float64)
    w = None if norm_weight is None else np.ascontiguousarray(norm_weight, np.float32)
    _load().o_swa_row(_p(x), _p(w), float(eps), int(pos is not None), float(rope_base),
                      float(0.0 if pos is None else pos), _p(out), _p(pre))
    return out, pre
