"""CSA2 decode over the FP4 global KV cache, GB300 (sm_103a).

Thin ctypes binding of ``libcsa2.so`` (declared in ``include/csa2.h``): the
functions below only marshal arguments -- every step of the path runs in the
library's CUDA kernels.  PyTorch, when used by a caller, only provides device
memory and streams: tensors are accepted wherever a device pointer is expected.

There is no CPU fallback: importing works without a GPU (for the ABI checks),
but any call needs the built library and a CUDA device.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsa2.so")

D_MAIN, D_IDX, H_IDX, H_ATT = 512, 128, 32, 64
ENTRY_BYTES = 356
TOPK_FLAT, TOPK_HIER_BUILD, TOPK_POOL = 0, 1, 2
LAYER_SWA, LAYER_FULL, LAYER_REINDEX, LAYER_REUSE = 0, 1, 2, 3

STATUS = {0: "CSA2_OK", 1: "CSA2_ERR_INVALID_ARG", 2: "CSA2_ERR_UNSUPPORTED",
          3: "CSA2_ERR_WORKSPACE", 4: "CSA2_ERR_CUDA", 5: "CSA2_ERR_DEVICE_TIMEOUT",
          6: "CSA2_ERR_INDEX_RANGE"}


class Csa2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class KVPlanes(ctypes.Structure):
    """csa2_kv_planes: device pointers of the four planes and the slot stride."""
    _fields_ = [("kv_codes", ctypes.c_void_p), ("kv_scales", ctypes.c_void_p),
                ("ix_codes", ctypes.c_void_p), ("ix_scales", ctypes.c_void_p),
                ("seq_stride", ctypes.c_int64)]


class NormRope(ctypes.Structure):
    """csa2_norm_rope: RMSNorm weight (device fp32 [512] or None), eps, RoPE on/off, base."""
    _fields_ = [("norm_weight", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
                ("rope", ctypes.c_int32), ("rope_base", ctypes.c_float)]


def norm_rope(norm_weight=None, eps: float = 1e-6, rope: bool = False, rope_base: float = 10000.0):
    """A csa2_norm_rope for the cache write (main-KV copy) or the attention (query heads).
    The struct keeps a reference to norm_weight, so the device array lives as long as it."""
    nr = NormRope(_ptr(norm_weight), float(eps), int(bool(rope)), float(rope_base))
    nr._weight = norm_weight
    return nr


class Window(ctypes.Structure):
    """csa2_window: per-row positions [B][n_swa] and per-query lowest visible position [B] (int64, device)."""
    _fields_ = [("row_pos", ctypes.c_void_p), ("lo", ctypes.c_void_p)]


def window(row_pos, lo) -> Window:
    """A csa2_window over device int64 arrays; keeps references to both."""
    win = Window(_ptr(row_pos), _ptr(lo))
    win._refs = (row_pos, lo)
    return win


class KernelTime(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C-ABI library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CSA2 CUDA library not built ({LIB_PATH}); "
                               "run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        pl = ctypes.POINTER(KVPlanes)
        nr = ctypes.POINTER(NormRope)
        wn = ctypes.POINTER(Window)
        sig = {
            "csa2_quantize_entries": ([vp, vp, i64, pl, i64, vp], ctypes.c_int),
            "csa2_cache_write": ([vp, i64, i32, vp, vp, vp, i32, pl, i32, i64, nr, i64, vp, sz, vp],
                                 ctypes.c_int),
            "csa2_cache_write_workspace_size": ([i64, i32, i32], sz),
            "csa2_quantize_index_query": ([vp, i64, vp, vp], ctypes.c_int),
            "csa2_cache_append": ([vp, i32, i32, vp, vp, vp, i32, pl, i32, vp, vp, nr, vp, vp, sz, vp],
                                  ctypes.c_int),
            "csa2_cache_append_workspace_size": ([i32, i32, i32], sz),
            "csa2_swa_append": ([vp, i32, vp, vp, i32, nr, vp, vp, i32, vp], ctypes.c_int),
            "csa2_index_topk": ([pl, i32, vp, i64, vp, vp, i32, ctypes.c_int, i32, i32, vp, vp, vp,
                                 vp, vp, sz, vp], ctypes.c_int),
            "csa2_index_topk_workspace_size": ([i32, i64, i32, i32, i32], sz),
            "csa2_pool_stage": ([pl, i32, vp, i64, i32, i32, vp, vp, vp, vp], ctypes.c_int),
            "csa2_index_topk_staged": ([vp, vp, i32, vp, i64, vp, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp],
                                       ctypes.c_int),
            "csa2_index_topk_prefill": ([pl, i32, i32, vp, i64, vp, vp, i32, vp, vp, sz, vp], ctypes.c_int),
            "csa2_index_topk_prefill_workspace_size": ([i32, i64, i32], sz),
            "csa2_index_topk_noalloc": ([pl, i32, vp, i64, vp, vp, i32, ctypes.c_int, i32, i32, vp,
                                         vp, vp, vp], ctypes.c_int),
            "csa2_sparse_attn_decode": ([pl, i32, vp, i32, vp, i32, vp, f32, nr, vp, vp, wn, vp, vp, vp, sz,
                                         vp], ctypes.c_int),
            "csa2_sparse_attn_workspace_size": ([i32, i32, i32], sz),
            "csa2_dense_attn_decode": ([pl, i32, vp, i64, vp, i32, vp, f32, nr, vp, vp, wn, vp, vp, vp, sz, vp],
                                       ctypes.c_int),
            "csa2_dense_attn_workspace_size": ([i32, i64, i32], sz),
            "csa2_compress_overlap": ([vp, i64, i32, vp, vp, vp, vp, vp, vp, i32, i32, vp, vp, sz, vp], ctypes.c_int),
            "csa2_compress_hca": ([vp, i64, i32, vp, vp, vp, i32, i32, vp, vp, sz, vp], ctypes.c_int),
            "csa2_compress_workspace_size": ([i64, i32], sz),
            "csa2_v41_layer_table": ([i32, vp, vp, vp, vp, vp], ctypes.c_int),
            "csa2_check": ([vp, vp, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
            "csa2_index_topk_noalloc_check": ([vp, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
            "csa2_selftest_wait_timeout": ([ctypes.c_longlong, vp, sz, vp], ctypes.c_int),
            "csa2_selftest_codec_division": ([vp, sz, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int64),
                                              vp], ctypes.c_int),
            "csa2_selftest_encode_sweep": ([ctypes.c_uint32, ctypes.c_uint32, vp, sz, vp, vp], ctypes.c_int),
            "csa2_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "csa2_timing_enable": ([i32], ctypes.c_int),
            "csa2_kernel_times": ([ctypes.POINTER(KernelTime), i32], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _nbytes(x) -> int:
    return x.numel() * x.element_size()


def _stream(s) -> int | None:
    if s is None:
        try:
            import torch

            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except ImportError:
            pass
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ok(rc: int, where: str) -> None:
    if rc != 0:
        raise Csa2Error(rc, where)


# ----------------------------------------------------------------------------- planes

@dataclass
class Planes:
    """Device planes of one Full layer's global KV plus the C struct that points at them."""
    kv_codes: object
    kv_scales: object
    ix_codes: object
    ix_scales: object
    seq_stride: int

    @property
    def c(self) -> KVPlanes:
        return KVPlanes(_ptr(self.kv_codes), _ptr(self.kv_scales), _ptr(self.ix_codes),
                        _ptr(self.ix_scales), self.seq_stride)

    @staticmethod
    def empty(n_seq: int, seq_stride: int, device="cuda") -> "Planes":
        import torch

        n = n_seq * seq_stride
        u8 = dict(dtype=torch.uint8, device=device)
        return Planes(torch.empty((n, 256), **u8), torch.empty((n, 32), **u8),
                      torch.empty((n, 64), **u8), torch.empty((n, 4), **u8), seq_stride)

    def nbytes(self) -> int:
        return sum(_nbytes(t) for t in (self.kv_codes, self.kv_scales, self.ix_codes, self.ix_scales))


def workspace(nbytes: int, device="cuda"):
    """A device workspace (torch allocations are at least 256-byte aligned)."""
    import torch

    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ----------------------------------------------------------------------------- entry points

def quantize_entries(planes: Planes, Cbar, KI, n: int, e0: int = 0, stream=None) -> None:
    _ok(lib().csa2_quantize_entries(_ptr(Cbar), _ptr(KI), n, ctypes.byref(planes.c), e0,
                                    _stream(stream)), "csa2_quantize_entries")


def quantize_index_query(q, n_rows: int, out, stream=None) -> None:
    """MXFP4 indexer query: q bf16 [n_rows][128] -> out bf16 (may be q) holding the values of
    its E2M1 codes under one E8M0 scale per 32 channels."""
    _ok(lib().csa2_quantize_index_query(_ptr(q), n_rows, _ptr(out), _stream(stream)),
        "csa2_quantize_index_query")


def cache_write_workspace_size(T: int, d_model: int, m: int) -> int:
    return lib().csa2_cache_write_workspace_size(T, d_model, m)


def cache_write(H, T: int, d_model: int, Wkv, Wz, Wik, m: int, planes: Planes, seq: int,
                entry_offset: int, ws, stream=None, kv_nr: NormRope | None = None,
                pos_first: int = 0) -> None:
    """kv_nr (norm_rope(...)): RMSNorm / RoPE of the main-KV copy; entry j of the call at
    position pos_first + j * m."""
    _ok(lib().csa2_cache_write(_ptr(H), T, d_model, _ptr(Wkv), _ptr(Wz), _ptr(Wik), m,
                               ctypes.byref(planes.c), seq, entry_offset,
                               ctypes.byref(kv_nr) if kv_nr is not None else None, int(pos_first),
                               _ptr(ws), _nbytes(ws), _stream(stream)), "csa2_cache_write")


def cache_append_workspace_size(G: int, d_model: int, m: int) -> int:
    return lib().csa2_cache_append_workspace_size(G, d_model, m)


def cache_append(H, G: int, d_model: int, Wkv, Wz, Wik, m: int, planes: Planes, n_slots: int, slot, entry,
                 ws, kv_nr: NormRope | None = None, pos=None, stream=None) -> None:
    """Decode-time append: G groups of m tokens (H bf16 [G][m][d_model]); entry g goes to slot
    slot[g], index entry[g] (device int32 / int64 arrays), at position pos[g] with RoPE."""
    _ok(lib().csa2_cache_append(_ptr(H), G, d_model, _ptr(Wkv), _ptr(Wz), _ptr(Wik), m,
                                ctypes.byref(planes.c), n_slots, _ptr(slot), _ptr(entry),
                                ctypes.byref(kv_nr) if kv_nr is not None else None, _ptr(pos), _ptr(ws),
                                _nbytes(ws), _stream(stream)), "csa2_cache_append")


def swa_append(x, R: int, pos, n_queries: int, ring, n_win: int, query=None, nr: NormRope | None = None,
               stream=None, ring_pos=None) -> None:
    """Window ring write: row r of x (fp32 [R][512]) -> E4M3 into ring[query[r] or r][pos[r] % n_win];
    ring_pos (int64 [n_queries][n_win], optional) records the rows' positions."""
    _ok(lib().csa2_swa_append(_ptr(x), R, _ptr(query), _ptr(pos), n_queries,
                              ctypes.byref(nr) if nr is not None else None, _ptr(ring), _ptr(ring_pos), n_win,
                              _stream(stream)), "csa2_swa_append")


def index_topk_workspace_size(B: int, n_max: int, k: int, block: int = 8,
                              n_blocks_keep: int = 0) -> int:
    return lib().csa2_index_topk_workspace_size(B, n_max, k, block, n_blocks_keep)


def index_topk(planes: Planes, B: int, n_entries, n_max: int, qidx, w, k: int, mode: int,
               topk_out, ws, block: int = 8, n_blocks_keep: int = 0, pool_in=None, pool_out=None,
               scores_out=None, stream=None) -> None:
    _ok(lib().csa2_index_topk(ctypes.byref(planes.c), B, _ptr(n_entries), n_max, _ptr(qidx), _ptr(w),
                              k, mode, block, n_blocks_keep, _ptr(pool_in), _ptr(topk_out),
                              _ptr(pool_out), _ptr(scores_out), _ptr(ws), _nbytes(ws),
                              _stream(stream)), "csa2_index_topk")


@dataclass
class PoolStage:
    """Staged indexer keys of a candidate pool: codes [B][keep*block][64], scales [B][keep*block][4]."""
    codes: object
    scales: object

    @staticmethod
    def empty(B: int, n_blocks_keep: int, block: int = 8, device="cuda") -> "PoolStage":
        import torch

        n = B * n_blocks_keep * block
        u8 = dict(dtype=torch.uint8, device=device)
        return PoolStage(torch.empty((n, 64), **u8), torch.empty((n, 4), **u8))


def pool_stage(planes: Planes, B: int, n_entries, n_max: int, pool, stage: PoolStage, block: int = 8,
               n_blocks_keep: int = 0, stream=None) -> None:
    """Gathers the pool's blocks of indexer keys once (csa2_pool_stage), for index_topk_staged."""
    _ok(lib().csa2_pool_stage(ctypes.byref(planes.c), B, _ptr(n_entries), n_max, block, n_blocks_keep,
                              _ptr(pool), _ptr(stage.codes), _ptr(stage.scales), _stream(stream)),
        "csa2_pool_stage")


def index_topk_staged(stage: PoolStage, B: int, n_entries, n_max: int, qidx, w, k: int, pool_in, topk_out,
                      ws, block: int = 8, n_blocks_keep: int = 0, scores_out=None, stream=None) -> None:
    """POOL-mode top-k over a pool staged by pool_stage (csa2_index_topk_staged)."""
    _ok(lib().csa2_index_topk_staged(_ptr(stage.codes), _ptr(stage.scales), B, _ptr(n_entries), n_max,
                                     _ptr(qidx), _ptr(w), k, block, n_blocks_keep, _ptr(pool_in),
                                     _ptr(topk_out), _ptr(scores_out), _ptr(ws), _nbytes(ws),
                                     _stream(stream)), "csa2_index_topk_staged")


def index_topk_prefill_workspace_size(Q: int, n_max: int, k: int) -> int:
    return lib().csa2_index_topk_prefill_workspace_size(Q, n_max, k)


def index_topk_prefill(planes: Planes, seq: int, Q: int, n_visible, n_max: int, qidx, w, k: int, topk_out,
                       ws, stream=None) -> None:
    """Prefill indexer: Q queries of slot `seq`, query q sees entries [0, n_visible[q])."""
    _ok(lib().csa2_index_topk_prefill(ctypes.byref(planes.c), seq, Q, _ptr(n_visible), n_max, _ptr(qidx),
                                      _ptr(w), k, _ptr(topk_out), _ptr(ws), _nbytes(ws), _stream(stream)),
        "csa2_index_topk_prefill")


NOALLOC_SCRATCH_BYTES = 32 << 20


def index_topk_noalloc(planes: Planes, B: int, n_entries, n_max: int, qidx, w, k: int, mode: int,
                       topk_out, block: int = 8, n_blocks_keep: int = 0, pool_in=None, pool_out=None,
                       stream=None) -> None:
    """csa2_index_topk without a workspace: scratch lives in a fixed device array
    of NOALLOC_SCRATCH_BYTES inside the library (for callers that cannot allocate)."""
    _ok(lib().csa2_index_topk_noalloc(ctypes.byref(planes.c), B, _ptr(n_entries), n_max, _ptr(qidx),
                                      _ptr(w), k, mode, block, n_blocks_keep, _ptr(pool_in),
                                      _ptr(topk_out), _ptr(pool_out), _stream(stream)),
        "csa2_index_topk_noalloc")


def index_topk_noalloc_check(stream=None) -> tuple[int, int]:
    """Syncs `stream`; (status, detail) of the first device-side error the allocation-free
    calls recorded since the last call began, then clears it (csa2_index_topk_noalloc_check)."""
    d = ctypes.c_int64(0)
    rc = lib().csa2_index_topk_noalloc_check(_stream(stream), ctypes.byref(d))
    return rc, d.value


def sparse_attn_workspace_size(B: int, k: int, n_swa: int) -> int:
    return lib().csa2_sparse_attn_workspace_size(B, k, n_swa)


def sparse_attn_decode(planes: Planes, B: int, topk, k: int, swa, n_swa: int, q,
                       softmax_scale: float, out, ws, lse_out=None, stream=None,
                       q_nr: NormRope | None = None, q_pos=None, sink=None, win: Window | None = None) -> None:
    """q_nr (norm_rope(...)): RMSNorm / RoPE of the query heads, q_pos int64 [B] (needed with
    RoPE; the output turns back by -q_pos); sink fp32 [64] per-head sink logits; win (window(...)):
    only window rows at positions >= lo[b] are seen."""
    _ok(lib().csa2_sparse_attn_decode(ctypes.byref(planes.c), B, _ptr(topk), k, _ptr(swa), n_swa,
                                      _ptr(q), softmax_scale,
                                      ctypes.byref(q_nr) if q_nr is not None else None, _ptr(q_pos),
                                      _ptr(sink), ctypes.byref(win) if win is not None else None, _ptr(out),
                                      _ptr(lse_out), _ptr(ws), _nbytes(ws), _stream(stream)),
        "csa2_sparse_attn_decode")


def dense_attn_workspace_size(B: int, n_max: int, n_swa: int) -> int:
    return lib().csa2_dense_attn_workspace_size(B, n_max, n_swa)


def dense_attn_decode(planes: Planes, B: int, n_entries, n_max: int, swa, n_swa: int, q,
                      softmax_scale: float, out, ws, lse_out=None, stream=None,
                      q_nr: NormRope | None = None, q_pos=None, sink=None, win: Window | None = None) -> None:
    """HCA attention: every entry [0, n_entries[b]) of slot b plus the window rows."""
    _ok(lib().csa2_dense_attn_decode(ctypes.byref(planes.c), B, _ptr(n_entries), n_max, _ptr(swa), n_swa,
                                     _ptr(q), softmax_scale,
                                     ctypes.byref(q_nr) if q_nr is not None else None, _ptr(q_pos),
                                     _ptr(sink), ctypes.byref(win) if win is not None else None, _ptr(out),
                                     _ptr(lse_out), _ptr(ws), _nbytes(ws), _stream(stream)),
        "csa2_dense_attn_decode")


def compress_workspace_size(T: int, d_model: int) -> int:
    return lib().csa2_compress_workspace_size(T, d_model)


def compress_overlap(H, T: int, d_model: int, Wa_kv, Wb_kv, Wa_z, Wb_z, Ba, Bb, m: int, out, ws,
                     stream=None, width: int = 512) -> None:
    """Two-path overlapping compressor: W_* [d_model][width], out fp32 [T/m][width] (width 512: main
    latents, 128: V4 indexer keys)."""
    _ok(lib().csa2_compress_overlap(_ptr(H), T, d_model, _ptr(Wa_kv), _ptr(Wb_kv), _ptr(Wa_z), _ptr(Wb_z),
                                    _ptr(Ba), _ptr(Bb), m, width, _ptr(out), _ptr(ws), _nbytes(ws),
                                    _stream(stream)), "csa2_compress_overlap")


def compress_hca(H, T: int, d_model: int, Wkv, Wz, Bp, m: int, out, ws, stream=None, width: int = 512) -> None:
    """HCA compressor: out fp32 [T/m][width]."""
    _ok(lib().csa2_compress_hca(_ptr(H), T, d_model, _ptr(Wkv), _ptr(Wz), _ptr(Bp), m, width, _ptr(out),
                                _ptr(ws), _nbytes(ws), _stream(stream)), "csa2_compress_hca")


def check(ws, stream=None) -> tuple[int, int]:
    """(status, detail) of the device-side error word of `ws`, cleared afterwards."""
    d = ctypes.c_int64(0)
    rc = lib().csa2_check(_ptr(ws), _stream(stream), ctypes.byref(d))
    return rc, d.value


def selftest_wait_timeout(budget_cycles: int, ws, stream=None) -> None:
    """Runs the bounded-wait self-test; csa2.check(ws) then reports the timeout."""
    _ok(lib().csa2_selftest_wait_timeout(int(budget_cycles), _ptr(ws), _nbytes(ws), _stream(stream)),
        "csa2_selftest_wait_timeout")


def selftest_codec_division(ws, stream=None) -> tuple[int, int]:
    """(differing quotients, comparisons) of the codec's division against the correctly
    rounded one over every positive E4M3 scale and fp32 significand in its range."""
    bad, n = ctypes.c_int64(0), ctypes.c_int64(0)
    _ok(lib().csa2_selftest_codec_division(_ptr(ws), _nbytes(ws), ctypes.byref(bad), ctypes.byref(n),
                                           _stream(stream)),
        "csa2_selftest_codec_division")
    return bad.value, n.value


def selftest_encode_sweep(ws, chunk0: int = 0, nchunks: int = 4096, stream=None):
    """uint64 [nchunks, 2]: per chunk of 2^20 fp32 bit patterns (c << 20 | i), the sums of
    the codec's E2M1 codes and E4M3 bytes of its non-NaN values weighted by 2 i + 1
    (mod 2^64) -- csa2_selftest_encode_sweep."""
    import numpy as np

    out = np.zeros((nchunks, 2), np.uint64)
    _ok(lib().csa2_selftest_encode_sweep(chunk0, nchunks, _ptr(ws), _nbytes(ws), out.ctypes.data,
                                         _stream(stream)), "csa2_selftest_encode_sweep")
    return out


def timing_enable(on: bool) -> None:
    """Switches per-kernel event timing on or off; discards the totals so far."""
    _ok(lib().csa2_timing_enable(1 if on else 0), "csa2_timing_enable")


def kernel_times() -> dict[str, tuple[int, float]]:
    """{kernel name: (launches, summed device ms)} since the last timing_enable (waits for them)."""
    n = lib().csa2_kernel_times(None, 0)
    if n < 0:
        raise Csa2Error(4, "csa2_kernel_times")
    arr = (KernelTime * max(n, 1))()
    n = lib().csa2_kernel_times(arr, n)
    if n < 0:
        raise Csa2Error(4, "csa2_kernel_times")
    return {arr[i].name.decode(): (int(arr[i].launches), float(arr[i].total_ms)) for i in range(n)}


def status_string(s: int) -> str:
    return lib().csa2_status_string(s).decode()


def v41_layer_table() -> dict[str, list[int]]:
    arrs = {k: (ctypes.c_int32 * 40)() for k in ("mode", "m", "kv_src", "topk_src", "pool_src")}
    _ok(lib().csa2_v41_layer_table(40, *[ctypes.addressof(a) for a in arrs.values()]),
        "csa2_v41_layer_table")
    return {k: list(a) for k, a in arrs.items()}
