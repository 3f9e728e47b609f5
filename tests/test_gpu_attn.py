"""csa2_sparse_attn_decode against the oracle: within 1e-2 x RMS per query, on
selections from the oracle's own top-k, with padding, duplicates, k = N,
SWA-only and empty cases, and the out-of-range error report."""
import numpy as np
import pytest

from gpu_common import SmallCache, csa2, require_gpu, to_dev, torch
from parity import check_attention
from synth import workloads as W

pytestmark = pytest.mark.gpu
SCALE = 1.0 / np.sqrt(512.0)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(scope="module")
def cache(oracle_mod):
    return SmallCache(oracle_mod, 1, 2, 3000, stride=3072)


def _attn(c, topk, swa, q, k, n_swa, lse=True):
    B = topk.shape[0]
    out = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
    lse_t = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.sparse_attn_workspace_size(B, k, n_swa))
    swa_c = np.ascontiguousarray(swa[:, :n_swa])  # [B][n_swa][512] contiguous
    csa2.sparse_attn_decode(c.planes, B, to_dev(topk.astype(np.int32)), k,
                            to_dev(swa_c) if n_swa else None, n_swa, to_dev(q.view(np.int16)), SCALE,
                            out, ws, lse_out=lse_t if lse else None)
    st, det = csa2.check(ws)
    return out.cpu().numpy(), lse_t.cpu().numpy(), st, det


def _oracle(oracle_mod, c, topk, swa, q, n_swa):
    outs, lses = [], []
    for b in range(topk.shape[0]):
        kvc, kvs, _, _ = c.oracle_slot(b)
        o, l = oracle_mod.attention(kvc, kvs, topk[b], swa[b][:n_swa], q[b], SCALE)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _oracle_topk(oracle_mod, c, k, layer=0):
    q, w = W.index_query(1, layer, c.B)
    sel = []
    for b in range(c.B):
        _, _, ixc, ixs = c.oracle_slot(b)
        sel.append(oracle_mod.topk(oracle_mod.index_scores(ixc, ixs, q[b], w[b]), k))
    return np.stack(sel)


@pytest.mark.parametrize("k,n_swa", [(512, 128), (512, 0), (100, 17), (2048, 128)])
def test_attention_matches_oracle(cache, oracle_mod, k, n_swa):
    c = cache
    topk = _oracle_topk(oracle_mod, c, k)
    q = W.attn_query(1, 0, c.B)
    swa = W.swa_rows(1, 0, c.B, 128)
    out, lse, st, _ = _attn(c, topk, swa, q, k, n_swa)
    assert st == 0
    ref, rlse = _oracle(oracle_mod, c, topk, swa, q, n_swa)
    check_attention(out, ref)
    assert np.allclose(lse, rlse, rtol=1e-4, atol=1e-4)


def test_k_equals_n_dense(oracle_mod):
    c = SmallCache(oracle_mod, 2, 1, 640)
    topk = np.arange(640, dtype=np.int32)[None, :]
    q = W.attn_query(2, 0, 1)
    swa = W.swa_rows(2, 0, 1, 128)
    out, _, st, _ = _attn(c, topk, swa, q, 640, 128)
    ref, _ = _oracle(oracle_mod, c, topk, swa, q, 128)
    assert st == 0
    check_attention(out, ref)


def test_padding_duplicates_and_swa_only(cache, oracle_mod):
    c = cache
    q = W.attn_query(1, 3, c.B)
    swa = W.swa_rows(1, 3, c.B, 128)
    rng = np.random.default_rng(0)
    topk = rng.integers(0, 3000, (c.B, 512)).astype(np.int32)  # duplicates allowed
    topk[:, ::3] = -1
    out, _, st, _ = _attn(c, topk, swa, q, 512, 64)
    ref, _ = _oracle(oracle_mod, c, topk, swa, q, 64)
    assert st == 0
    check_attention(out, ref)
    none = np.full((c.B, 512), -1, np.int32)
    out, lse, st, _ = _attn(c, none, swa, q, 512, 128)
    ref, rl = _oracle(oracle_mod, c, none, swa, q, 128)
    check_attention(out, ref)
    out, lse, st, _ = _attn(c, none, swa, q, 512, 0)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_out_of_range_index_reported(cache):
    c = cache
    q = W.attn_query(1, 4, c.B)
    swa = W.swa_rows(1, 4, c.B, 128)
    topk = np.tile(np.arange(512, dtype=np.int32), (c.B, 1))
    topk[1, 7] = 3072 + 5  # beyond the slot
    _, _, st, det = _attn(c, topk, swa, q, 512, 128)
    assert st == 6 and det == 3077


def _extras(B, seed):
    rng = np.random.default_rng(seed)
    w = (1.0 + 0.3 * rng.standard_normal(512)).astype(np.float32)
    pos = (1_000_003 + 37 * np.arange(B)).astype(np.int64)  # millions: the fp64 angle path
    sink = (2.0 * rng.standard_normal(64)).astype(np.float32)
    return w, pos, sink


def _lse_bound(oracle_mod, c, topk, swa, q, n_swa, w, pos):
    """Each logit moves by at most scale * 2^-11 * sum_c |q'_c x_c| when q' (normalised and
    rotated in fp32) is rounded to f16 (2^-12 relative) plus its fp32 arithmetic (2^-12,
    generously); lse moves by at most the largest logit change of its query."""
    import synth

    bounds = []
    for b in range(topk.shape[0]):
        kvc, kvs, _, _ = c.oracle_slot(b)
        idx = topk[b][topk[b] >= 0]
        X = np.concatenate([oracle_mod.dequant_main(kvc[idx], kvs[idx]),
                            _e4m3_rows(swa[b][:n_swa])]) if n_swa else oracle_mod.dequant_main(kvc[idx], kvs[idx])
        qf = synth.bf16_to_f32(q[b]).astype(np.float64)
        qn = oracle_mod.rope(oracle_mod.rmsnorm(qf, w, 1e-6), float(pos[b]))
        bounds.append(SCALE * 2.0 ** -11 * (np.abs(qn) @ np.abs(X).T).max(1))
    return np.stack(bounds)


def _e4m3_rows(b):
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("B", [2, 80])
def test_attention_with_norm_rope_sink(oracle_mod, B):
    """Query RMSNorm + RoPE at positions near 10^6, the output turned back, a sink per head:
    batch 2 splits each query over several CTAs (the merge adds the sink), batch 80 runs a
    query in one CTA."""
    n = 700
    c = SmallCache(oracle_mod, 6, B, n)
    k, n_swa = 512, 128
    rng = np.random.default_rng(B)
    topk = np.sort(np.stack([rng.choice(n, k, replace=False) for _ in range(B)]), 1).astype(np.int32)
    topk[:, 5] = -1
    q = W.attn_query(6, 1, B)
    swa = W.swa_rows(6, 1, B, 128)
    w, pos, sink = _extras(B, B + 1)
    out = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.sparse_attn_workspace_size(B, k, n_swa))
    w_d = to_dev(w)
    csa2.sparse_attn_decode(c.planes, B, to_dev(topk), k, to_dev(np.ascontiguousarray(swa)), n_swa,
                            to_dev(q.view(np.int16)), SCALE, out, ws, lse_out=lse,
                            q_nr=csa2.norm_rope(w_d, 1e-6, True, 10000.0), q_pos=to_dev(pos),
                            sink=to_dev(sink))
    assert csa2.check(ws)[0] == 0
    got, glse = out.cpu().numpy(), lse.cpu().numpy()
    ref, rlse = [], []
    for b in range(B):
        kvc, kvs, _, _ = c.oracle_slot(b)
        o, l_ = oracle_mod.attention(kvc, kvs, topk[b], swa[b], q[b], SCALE, q_norm_weight=w, eps=1e-6,
                                     qpos=float(pos[b]), sink=sink)
        ref.append(o)
        rlse.append(l_)
    ref, rlse = np.stack(ref), np.stack(rlse)
    check_attention(got, ref)
    bound = _lse_bound(oracle_mod, c, topk, swa, q, n_swa, w, pos)
    assert np.all(np.abs(glse - rlse) <= bound + 1e-5 * np.abs(rlse) + 1e-5)
    # the sink takes weight: a sink far above every logit drives the output to zero
    csa2.sparse_attn_decode(c.planes, B, to_dev(topk), k, to_dev(np.ascontiguousarray(swa)), n_swa,
                            to_dev(q.view(np.int16)), SCALE, out, ws, lse_out=lse,
                            q_nr=csa2.norm_rope(w_d, 1e-6, True, 10000.0), q_pos=to_dev(pos),
                            sink=to_dev(np.full(64, 1e4, np.float32)))
    assert np.abs(out.cpu().numpy()).max() < 1e-30
    assert np.allclose(lse.cpu().numpy(), 1e4, rtol=1e-6)
