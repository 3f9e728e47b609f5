"""Seeded synthetic inputs for the CSA2 decode and cache-write workloads.

This module is the one thing the oracle side and the CUDA side share: it draws
the random inputs (never any of the method's arithmetic).  The generator is a
counter-based SplitMix64 stream per (seed, tensor id); element i of a tensor is
a pure function of (seed, tensor id, i), so any slice of any tensor can be
regenerated on its own, on the host (``synth_host.c``) or on the device
(``synth_dev.cu``), with identical bits.  The definition is written out in
``synth_core.h``.

Workload recipes (shapes and distributions) live in :mod:`synth.workloads`.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(_HERE, "libcsa2synth_host.so")
DEV_LIB = os.path.join(_HERE, "libcsa2synth_dev.so")

_host = None
_dev = None


def _load_host():
    global _host
    if _host is None:
        if not os.path.exists(HOST_LIB):
            from . import build as _b

            _b.build_host()
        lib = ctypes.CDLL(HOST_LIB)
        u64, i64, i32, f32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        vp = ctypes.c_void_p
        lib.syn_stream_key.argtypes = [u64, u64]
        lib.syn_stream_key.restype = u64
        lib.syn_host_normal_f32.argtypes = [u64, u64, u64, i64, f32, vp, ctypes.c_int]
        lib.syn_host_normal_bf16.argtypes = [u64, u64, u64, i64, f32, vp, ctypes.c_int]
        lib.syn_host_uniform_f32.argtypes = [u64, u64, u64, i64, vp, ctypes.c_int]
        lib.syn_host_e4m3_normal.argtypes = [u64, u64, u64, i64, f32, vp, ctypes.c_int]
        lib.syn_host_keys.argtypes = [u64, u64, u64, u64, i64, i32, f32, vp, vp, ctypes.c_int]
        for f in ("syn_host_normal_f32", "syn_host_normal_bf16", "syn_host_uniform_f32",
                  "syn_host_e4m3_normal", "syn_host_keys"):
            getattr(lib, f).restype = None
        _host = lib
    return _host


def _load_dev():
    global _dev
    if _dev is None:
        if not os.path.exists(DEV_LIB):
            raise RuntimeError(
                f"device generator library missing: {DEV_LIB}; run __graft_entry__.build()")
        lib = ctypes.CDLL(DEV_LIB)
        u64, i64, i32, f32, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                  ctypes.c_void_p)
        lib.syn_dev_normal_f32.argtypes = [u64, u64, u64, i64, f32, vp, vp]
        lib.syn_dev_normal_bf16.argtypes = [u64, u64, u64, i64, f32, vp, vp]
        lib.syn_dev_uniform_f32.argtypes = [u64, u64, u64, i64, vp, vp]
        lib.syn_dev_e4m3_normal.argtypes = [u64, u64, u64, i64, f32, vp, vp]
        lib.syn_dev_keys.argtypes = [u64, u64, u64, u64, i64, i32, f32, vp, vp, vp]
        for f in ("syn_dev_normal_f32", "syn_dev_normal_bf16", "syn_dev_uniform_f32",
                  "syn_dev_e4m3_normal", "syn_dev_keys"):
            getattr(lib, f).restype = ctypes.c_int
        _dev = lib
    return _dev


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------------------- host fills

def stream_key(seed: int, tid: int) -> int:
    return int(_load_host().syn_stream_key(seed, tid))


def normal_f32(seed: int, tid: int, n: int, offset: int = 0, scale: float = 1.0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load_host().syn_host_normal_f32(seed, tid, offset, n, scale, _ptr(out), _threads())
    return out


def normal_bf16(seed: int, tid: int, n: int, offset: int = 0, scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of scale * N(0,1), rounded to nearest even."""
    out = np.empty(n, np.uint16)
    _load_host().syn_host_normal_bf16(seed, tid, offset, n, scale, _ptr(out), _threads())
    return out


def uniform_f32(seed: int, tid: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, np.float32)
    _load_host().syn_host_uniform_f32(seed, tid, offset, n, _ptr(out), _threads())
    return out


def e4m3_normal(seed: int, tid: int, n: int, offset: int = 0, scale: float = 1.0) -> np.ndarray:
    """FP8 E4M3 bytes of scale * N(0,1) (input synthesis for sliding-window rows)."""
    out = np.empty(n, np.uint8)
    _load_host().syn_host_e4m3_normal(seed, tid, offset, n, scale, _ptr(out), _threads())
    return out


def keys_f32(seed: int, tid: int, tid_hot: int, n: int, dim: int, offset: int = 0,
             hot_prob: float = 0.0, hotvec: np.ndarray | None = None) -> np.ndarray:
    """Rows of N(0,1) keys; a row is 'hot' with probability hot_prob and gets hotvec added."""
    out = np.empty(n, np.float32)
    hv = None
    if hotvec is not None:
        hv = np.ascontiguousarray(hotvec, np.float32)
        assert hv.shape == (dim,)
    _load_host().syn_host_keys(seed, tid, tid_hot, offset, n, dim, hot_prob,
                               None if hv is None else _ptr(hv), _ptr(out), _threads())
    return out


# ----------------------------------------------------------------------------- device fills

def _chk(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what}: CUDA error {rc}")


def dev_normal_f32(seed, tid, n, out_ptr, stream=0, offset=0, scale=1.0):
    _chk(_load_dev().syn_dev_normal_f32(seed, tid, offset, n, scale, out_ptr, stream), "normal_f32")


def dev_normal_bf16(seed, tid, n, out_ptr, stream=0, offset=0, scale=1.0):
    _chk(_load_dev().syn_dev_normal_bf16(seed, tid, offset, n, scale, out_ptr, stream), "normal_bf16")


def dev_uniform_f32(seed, tid, n, out_ptr, stream=0, offset=0):
    _chk(_load_dev().syn_dev_uniform_f32(seed, tid, offset, n, out_ptr, stream), "uniform_f32")


def dev_e4m3_normal(seed, tid, n, out_ptr, stream=0, offset=0, scale=1.0):
    _chk(_load_dev().syn_dev_e4m3_normal(seed, tid, offset, n, scale, out_ptr, stream), "e4m3")


def dev_keys_f32(seed, tid, tid_hot, n, dim, out_ptr, stream=0, offset=0, hot_prob=0.0,
                 hotvec_ptr=None):
    _chk(_load_dev().syn_dev_keys(seed, tid, tid_hot, offset, n, dim, hot_prob, hotvec_ptr,
                                  out_ptr, stream), "keys")


def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    return (np.asarray(u16, np.uint16).astype(np.uint32) << 16).view(np.float32)
