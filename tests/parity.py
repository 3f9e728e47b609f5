"""Parity rules between the CUDA path and the oracle.

Top-k: the GPU set must hold every entry whose oracle score exceeds the
oracle's k-th score tau by more than 1e-3 relative, and no entry below tau by
more than that; it has exactly min(k, valid) distinct entries, ascending, -1
padded.  Attention: max |gpu - oracle| <= 1e-2 * RMS(oracle) per query.
Cache bytes: identical for the codec on identical fp32 inputs; for the cache
write, identical in every group whose rounding decisions lie farther from the
oracle's pre-quantization values than the error bound of the GPU's fp32
accumulation (test_gpu_cache_write.py states the bound).
"""
from __future__ import annotations

import numpy as np

TOPK_REL = 1e-3
ATTN_REL = 1e-2


def check_topk(gpu: np.ndarray, scores: np.ndarray, k: int, valid: np.ndarray | None = None,
               rel: float = TOPK_REL, what: str = "topk") -> None:
    """gpu: [k] chosen ids; scores: oracle score per id (len n); valid: bool per id."""
    gpu = np.asarray(gpu)
    n = scores.shape[0]
    if valid is None:
        valid = np.ones(n, bool)
    ids = np.nonzero(valid)[0]
    want = min(k, ids.size)
    chosen = gpu[gpu >= 0]
    assert chosen.size == want, f"{what}: {chosen.size} chosen, expected {want}"
    assert np.all(gpu[want:] == -1), f"{what}: padding"
    assert np.all(np.diff(chosen) > 0), f"{what}: not strictly ascending"
    assert np.all(valid[chosen]), f"{what}: invalid id chosen"
    if want == 0:
        return
    vs = scores[ids]
    tau = np.sort(vs)[::-1][want - 1]
    band = rel * abs(tau)
    must = ids[vs > tau + band]
    missing = np.setdiff1d(must, chosen)
    assert missing.size == 0, f"{what}: {missing.size} clearly-above entries missing, e.g. {missing[:5]}"
    low = chosen[scores[chosen] < tau - band]
    assert low.size == 0, f"{what}: {low.size} clearly-below entries chosen, e.g. {low[:5]}"


def check_attention(gpu: np.ndarray, ref: np.ndarray, rel: float = ATTN_REL, what="attn") -> float:
    """Per query: max abs error <= rel * RMS of the oracle output.  Returns the worst ratio."""
    gpu = np.asarray(gpu, np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    worst = 0.0
    for b in range(ref.shape[0]):
        rms = np.sqrt(np.mean(ref[b] ** 2))
        err = np.max(np.abs(gpu[b] - ref[b]))
        if rms == 0:
            assert err == 0, f"{what}[{b}]: nonzero output where the oracle is 0"
            continue
        worst = max(worst, err / rms)
        assert err <= rel * rms, f"{what}[{b}]: max err {err:.3e} > {rel} * rms {rms:.3e}"
    return worst
