"""Pins of the oracle's sparse MQA + sliding-window attention: a dense numpy
softmax-attention over explicit rows (k = N), closed forms (one row, equal
logits), and permutation invariance."""
import numpy as np
import pytest

import synth
from synth.workloads import attn_query, main_latents, swa_rows


def _kv(oracle_mod, n, seed=0):
    return oracle_mod.quantize_main(main_latents(seed, 0, 1, n, 0, 0, n))


def _dense(rows: np.ndarray, q: np.ndarray, scale: float):
    """Textbook softmax(scale q X^T) X with a log-sum-exp, fp64, numpy only."""
    lg = scale * (q @ rows.T)
    m = lg.max(1, keepdims=True)
    p = np.exp(lg - m)
    den = p.sum(1, keepdims=True)
    return (p / den) @ rows, (m + np.log(den))[:, 0]


def _e4m3(b):
    import torch

    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_k_equals_n_is_dense(oracle_mod):
    n = 96
    kc, ks = _kv(oracle_mod, n)
    swa = swa_rows(0, 0, 1, 16)[0]
    q = attn_query(0, 0, 1)[0]
    topk = np.arange(n, dtype=np.int32)
    out, lse = oracle_mod.attention(kc, ks, topk, swa, q, 1 / np.sqrt(512))
    rows = np.concatenate([oracle_mod.dequant_main(kc, ks), _e4m3(swa)])
    ref, rlse = _dense(rows, synth.bf16_to_f32(q).astype(np.float64), 1 / np.sqrt(512))
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, rlse, rtol=1e-12, atol=1e-12)


def test_single_row_returns_row(oracle_mod):
    kc, ks = _kv(oracle_mod, 10)
    q = attn_query(0, 1, 1)[0]
    out, _ = oracle_mod.attention(kc, ks, np.array([7, -1, -1], np.int32),
                                  np.zeros((0, 512), np.uint8), q, 0.1)
    row = oracle_mod.dequant_main(kc[7:8], ks[7:8])[0]
    assert np.array_equal(out, np.broadcast_to(row, out.shape))


def test_equal_logits_give_mean(oracle_mod):
    kc, ks = _kv(oracle_mod, 40)
    q = np.zeros((64, 512), np.uint16)  # q = 0 -> all logits equal
    sel = np.array([3, 9, 11, 30], np.int32)
    swa = swa_rows(0, 2, 1, 4)[0]
    out, lse = oracle_mod.attention(kc, ks, sel, swa, q, 1.0)
    rows = np.concatenate([oracle_mod.dequant_main(kc[sel], ks[sel]), _e4m3(swa)])
    assert np.allclose(out, rows.mean(0)[None, :], rtol=1e-14, atol=1e-14)
    assert np.allclose(lse, np.log(8.0))


def test_permutation_invariance(oracle_mod):
    kc, ks = _kv(oracle_mod, 200)
    q = attn_query(0, 3, 1)[0]
    rng = np.random.default_rng(0)
    sel = rng.choice(200, 64, replace=False).astype(np.int32)
    swa = swa_rows(0, 3, 1, 8)[0]
    a, la = oracle_mod.attention(kc, ks, sel, swa, q, 0.05)
    b, lb = oracle_mod.attention(kc, ks, rng.permutation(sel), swa, q, 0.05)
    assert np.allclose(a, b, rtol=1e-13, atol=1e-14)
    assert np.allclose(la, lb, rtol=1e-14)


def test_padding_entries_skipped(oracle_mod):
    kc, ks = _kv(oracle_mod, 50)
    q = attn_query(0, 4, 1)[0]
    swa = swa_rows(0, 4, 1, 2)[0]
    sel = np.array([1, 2, 3], np.int32)
    a, _ = oracle_mod.attention(kc, ks, sel, swa, q, 0.05)
    b, _ = oracle_mod.attention(kc, ks, np.array([1, -1, 2, -1, 3], np.int32), swa, q, 0.05)
    assert np.array_equal(a, b)


def test_empty_gives_zero(oracle_mod):
    kc, ks = _kv(oracle_mod, 4)
    out, lse = oracle_mod.attention(kc, ks, np.full(4, -1, np.int32), np.zeros((0, 512), np.uint8),
                                    attn_query(0, 5, 1)[0], 0.05)
    assert np.all(out == 0) and np.all(lse == -np.inf)
