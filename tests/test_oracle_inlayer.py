"""Pins of the oracle's in-layer math around the path ("DeepSeek-V4: Towards Highly
Efficient Million-Token Context Intelligence", CSA, other details: RMSNorm of each query
head and compressed entry, RoPE on the last 64 channels of query, KV and output with the
output turned back by -t, the attention sink; "DeepSeek-V4.1-Flash", 2.4.4: the cache is
quantized after RoPE).  Pinned by what the definitions fix: the RMS of a normalised row,
scale invariance, norm-preserving rotations that compose and invert, the relative-position
property the pages state (R_-t o_t = sum_s a_ts R_(s-t) e_s: shifting every position by
the same amount leaves the turned-back output unchanged), closed forms of the sink, and
the plain path when every extra is off."""
import numpy as np
import pytest

import synth
from synth.workloads import attn_query, main_latents, swa_rows

D = 512
R0 = D - 64  # first rotated channel


def _rows(n, seed=1):
    return np.random.default_rng(seed).standard_normal((n, D))


def test_rmsnorm_unit_rms_and_scale_invariance(oracle_mod):
    x = _rows(5)
    y = oracle_mod.rmsnorm(x, eps=0.0)
    assert np.allclose((y ** 2).mean(1), 1.0, rtol=0, atol=1e-13)
    assert np.allclose(oracle_mod.rmsnorm(3.5 * x, eps=0.0), y, rtol=0, atol=1e-13)
    ms = (x ** 2).mean(1)
    ye = oracle_mod.rmsnorm(x, eps=0.25)
    assert np.allclose((ye ** 2).mean(1), ms / (ms + 0.25), rtol=1e-13, atol=0)
    w = np.linspace(-2, 2, D).astype(np.float32)
    assert np.allclose(oracle_mod.rmsnorm(x, w, eps=0.0), y * w.astype(np.float64), rtol=0, atol=1e-13)


def test_rope_touches_only_the_last_64_and_keeps_pair_norms(oracle_mod):
    x = _rows(3)
    y = oracle_mod.rope(x, 12345.0)
    assert np.array_equal(y[:, :R0], x[:, :R0])
    pn = lambda a: np.hypot(a[:, R0::2], a[:, R0 + 1::2])
    assert np.allclose(pn(y), pn(x), rtol=1e-13, atol=0)
    assert not np.allclose(y[:, R0:], x[:, R0:])


def test_rope_angles_of_single_pairs(oracle_mod):
    # pair i turns by pos * 10000^(-i/32): pair 0 by pos radians, pair 16 by pos/100,
    # counter-clockwise (a, b) -> (a cos - b sin, a sin + b cos)
    for i, theta in ((0, 1.0), (16, 0.01), (31, 1e4 ** (-31 / 32))):
        x = np.zeros(D)
        x[R0 + 2 * i] = 1.0
        y = oracle_mod.rope(x, 1.0)
        assert y[R0 + 2 * i] == pytest.approx(np.cos(theta), abs=1e-15)
        assert y[R0 + 2 * i + 1] == pytest.approx(np.sin(theta), abs=1e-15)
        x[R0 + 2 * i], x[R0 + 2 * i + 1] = 0.0, 1.0
        y = oracle_mod.rope(x, 1.0)
        assert y[R0 + 2 * i] == pytest.approx(-np.sin(theta), abs=1e-15)


def test_rope_composes_and_inverts(oracle_mod):
    x = _rows(2, 3)
    assert np.allclose(oracle_mod.rope(oracle_mod.rope(x, 777.0), -777.0), x, rtol=0, atol=1e-12)
    a = oracle_mod.rope(oracle_mod.rope(x, 100.0), 23.0)
    assert np.allclose(a, oracle_mod.rope(x, 123.0), rtol=0, atol=1e-11)


def test_rope_dot_depends_on_the_position_difference(oracle_mod):
    a, b = _rows(1, 4)[0], _rows(1, 5)[0]
    d0 = oracle_mod.rope(a, 40.0) @ oracle_mod.rope(b, 15.0)
    d1 = oracle_mod.rope(a, 40.0 + 9000.0) @ oracle_mod.rope(b, 15.0 + 9000.0)
    assert d0 == pytest.approx(d1, rel=1e-12)
    assert d0 != pytest.approx(oracle_mod.rope(a, 41.0) @ oracle_mod.rope(b, 15.0), rel=1e-9)


def test_turned_back_output_is_relative(oracle_mod):
    """Entries rotated at their positions p_s + shift, the query at t + shift: the output
    turned back by -(t + shift) is the same for every shift."""
    e = _rows(40, 6) * 0.5
    pos = np.arange(40) * 4.0 + 3.0
    q = attn_query(3, 0, 1)[0]
    t = 170.0
    outs = []
    for shift in (0.0, 1000.0, 123456.0):
        X = np.stack([oracle_mod.rope(e[s], pos[s] + shift) for s in range(40)])
        o, lse = oracle_mod.attention_rows(X, q, 1 / np.sqrt(512), qpos=t + shift)
        outs.append((o, lse))
    for o, lse in outs[1:]:
        assert np.allclose(o, outs[0][0], rtol=1e-9, atol=1e-11)
        assert np.allclose(lse, outs[0][1], rtol=1e-11, atol=1e-11)
    # without the turn back the output keeps the absolute position
    absolute = [oracle_mod.rope(o, t + shift) for (o, _), shift in zip(outs, (0.0, 1000.0))]
    assert not np.allclose(absolute[0][:, R0:], absolute[1][:, R0:], atol=1e-6)
    assert np.allclose(absolute[0][:, :R0], absolute[1][:, :R0], rtol=1e-9, atol=1e-11)


def test_query_norm_is_scale_invariant(oracle_mod):
    X = _rows(30, 7)
    q = attn_query(4, 0, 1)[0]
    qf = synth.bf16_to_f32(q)
    q2 = ((qf * 2.0).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # exact: a power of two
    w = np.full(D, 0.7, np.float32)
    o1, l1 = oracle_mod.attention_rows(X, q, 0.05, q_norm_weight=w, eps=0.0)
    o2, l2 = oracle_mod.attention_rows(X, q2, 0.05, q_norm_weight=w, eps=0.0)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-13) and np.allclose(l1, l2, rtol=1e-12)
    o3, _ = oracle_mod.attention_rows(X, q, 0.05)
    assert not np.allclose(o1, o3, atol=1e-6)


def test_sink_closed_form_on_equal_logits(oracle_mod):
    """n equal rows x: every logit is L, so a = e^L / (n e^L + e^z) and out = n a x."""
    n = 7
    x = np.random.default_rng(8).standard_normal(D)
    X = np.tile(x, (n, 1))
    q = attn_query(5, 0, 1)[0]
    qf = synth.bf16_to_f32(q).astype(np.float64)
    scale = 0.03
    L = scale * (qf @ x)
    z = np.linspace(-3, 3, 64).astype(np.float32)
    o, lse = oracle_mod.attention_rows(X, q, scale, sink=z)
    frac = n * np.exp(L) / (n * np.exp(L) + np.exp(z.astype(np.float64)))
    assert np.allclose(o, frac[:, None] * x[None, :], rtol=1e-12, atol=1e-14)
    assert np.allclose(lse, np.logaddexp(np.log(n) + L, z.astype(np.float64)), rtol=1e-13, atol=1e-13)
    # a sink far below the logits changes nothing; with no rows only the sink is left
    o0, l0 = oracle_mod.attention_rows(X, q, scale)
    ofar, lfar = oracle_mod.attention_rows(X, q, scale, sink=np.full(64, -1e30, np.float32))
    assert np.allclose(ofar, o0, rtol=1e-15, atol=0) and np.allclose(lfar, l0, rtol=1e-15)
    oe, le = oracle_mod.attention_rows(np.zeros((0, D)), q, scale, sink=z)
    assert np.all(oe == 0) and np.allclose(le, z.astype(np.float64))


def test_extras_off_is_the_plain_path(oracle_mod):
    kc, ks = oracle_mod.quantize_main(main_latents(0, 0, 1, 64, 0, 0, 64))
    swa = swa_rows(0, 0, 1, 8)[0]
    q = attn_query(0, 0, 1)[0]
    topk = np.arange(64, dtype=np.int32)[::-1].copy()
    a = oracle_mod.attention(kc, ks, topk, swa, q, 0.044)
    b = oracle_mod.attention(kc, ks, topk, swa, q, 0.044, q_norm_weight=None, qpos=None, sink=None)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_cache_write_quantizes_the_normalised_rotated_copy(oracle_mod):
    """Entry j: RMSNorm of its pooled latent, turned to position pos_first + j m, then
    quantized; the indexer key keeps the pooled latent."""
    rng = np.random.default_rng(9)
    bits = lambda a: (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    T, d, m = 12, 64, 2
    H = bits(rng.standard_normal((T, d)).astype(np.float32))
    Wkv = bits((rng.standard_normal((d, D)) / 8).astype(np.float32))
    Wz = bits((rng.standard_normal((d, D)) / 8).astype(np.float32))
    Wik = bits((rng.standard_normal((D, 128)) / 8).astype(np.float32))
    w = (1.0 + 0.5 * rng.standard_normal(D)).astype(np.float32)
    plain = oracle_mod.cache_write(H, Wkv, Wz, Wik, m, return_prequant=True)
    got = oracle_mod.cache_write(H, Wkv, Wz, Wik, m, return_prequant=True, norm_weight=w, eps=1e-6,
                                 rope=True, pos_first=7.0)
    cb, att = got[4], got[6]
    assert np.array_equal(cb, plain[4])                      # the pooled latent is unchanged
    assert np.array_equal(got[2], plain[2]) and np.array_equal(got[3], plain[3])  # indexer key too
    for j in range(T // m):
        back = oracle_mod.rope(att[j], -(7.0 + j * m))          # turned back to position 0
        assert np.allclose(back, oracle_mod.rmsnorm(cb[j], w, 1e-6), rtol=1e-12, atol=1e-12)
    assert np.allclose((oracle_mod.rmsnorm(cb, None, 0.0) ** 2).mean(1), 1.0, atol=1e-12)
    kc, ks = oracle_mod.quantize_main(att.astype(np.float32))
    assert np.array_equal(got[0], kc) and np.array_equal(got[1], ks)


def test_swa_row_encodes_the_normalised_rotated_value(oracle_mod):
    x = _rows(1, 11)[0] * 3.0
    plain, pre = oracle_mod.swa_row(x)
    assert np.array_equal(pre, x)
    assert np.array_equal(plain, oracle_mod.e4m3_encode_array(x.astype(np.float32)))
    w = np.linspace(0.5, 1.5, D).astype(np.float32)
    out, pre = oracle_mod.swa_row(x, w, 1e-6, pos=4321.0)
    assert np.allclose(oracle_mod.rope(pre, -4321.0), oracle_mod.rmsnorm(x, w, 1e-6), rtol=1e-12, atol=1e-12)
    assert np.array_equal(out, oracle_mod.e4m3_encode_array(pre.astype(np.float32)))
    # E4M3 keeps 3 mantissa bits: the decoded row is within 2^-4 relative of the value (or saturated)
    dec = np.array([oracle_mod.e4m3_value(int(v)) for v in out])
    ok = np.abs(pre) < 448
    assert np.all(np.abs(dec[ok] - pre[ok]) <= 2.0 ** -4 * np.abs(pre[ok]) + 2.0 ** -10)
