"""Decode-time writes against the oracle: csa2_cache_append (each group of m tokens makes
one entry of its own slot, computed as the prefill write computes it) and csa2_swa_append
(one E4M3 window row per token into a ring), with and without RMSNorm / RoPE."""
import numpy as np
import pytest

from gpu_common import SmallCache, csa2, require_gpu, to_dev, torch
from synth import workloads as W
from test_gpu_cache_write import U, _decided_index, _decided_main, _error_bounds, _norm_rope_bounds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _e4m3_mids(oracle_mod):
    return np.array([0.5 * (oracle_mod.e4m3_value(c) + oracle_mod.e4m3_value(c + 1)) for c in range(126)])


@pytest.mark.parametrize("m,nr", [(1, False), (2, True), (1, True)])
def test_cache_append_matches_the_write_of_each_group(oracle_mod, m, nr):
    d, G, n_slots, stride = 1024, 6, 4, 50
    H, Wkv, Wz, Wik = W.cache_write_inputs(7, G * m, d)
    slots = np.array([0, 3, 1, 3, 2, 0], np.int32)
    entries = np.array([7, 0, 49, 12, 3, 8], np.int64)
    pos = entries * m + (m - 1) + 1_000_000
    w = (1.0 + 0.3 * np.random.default_rng(m).standard_normal(512)).astype(np.float32)
    P = csa2.Planes.empty(n_slots, stride)
    for t in (P.kv_codes, P.kv_scales, P.ix_codes, P.ix_scales):
        t.fill_(0xA5)
    ws = csa2.workspace(csa2.cache_append_workspace_size(G, d, m))
    kv_nr = csa2.norm_rope(to_dev(w), 1e-6, True, 10000.0) if nr else None
    csa2.cache_append(to_dev(H.view(np.int16)), G, d, to_dev(Wkv.view(np.int16)), to_dev(Wz.view(np.int16)),
                      to_dev(Wik.view(np.int16)), m, P, n_slots, to_dev(slots), to_dev(entries), ws,
                      kv_nr=kv_nr, pos=to_dev(pos) if nr else None)
    assert csa2.check(ws)[0] == 0
    planes = [t.cpu().numpy() for t in (P.kv_codes, P.kv_scales, P.ix_codes, P.ix_scales)]
    mids = _e4m3_mids(oracle_mod)
    written = set()
    for g in range(G):
        Hg = H[g * m:(g + 1) * m]
        kvc, kvs, ixc, ixs, cb, ki, att = oracle_mod.cache_write(
            Hg, Wkv, Wz, Wik, m, return_prequant=True, norm_weight=w if nr else None, eps=1e-6, rope=nr,
            pos_first=float(pos[g]), pos_step=float(m))
        eCb, eKI = _error_bounds(Hg, Wkv, Wz, Wik, m, cb)
        eAtt = _norm_rope_bounds(cb, att, eCb, w, 1e-6) if nr else eCb
        row = int(slots[g]) * stride + int(entries[g])
        written.add(row)
        got = [p[row:row + 1] for p in planes]
        dm = _decided_main(att.astype(np.float32).astype(np.float64), eAtt, mids, oracle_mod)
        di = _decided_index(ki.astype(np.float32).astype(np.float64), eKI)
        for (gc, gs, rc, rs, dec, gb) in ((got[0], got[1], kvc, kvs, dm, 8), (got[2], got[3], ixc, ixs, di, 16)):
            same = (gc.reshape(1, -1, gb) == rc.reshape(1, -1, gb)).all(-1) & (gs == rs)
            assert not (dec & ~same).any(), f"group {g}: decided quantization groups differ"
    untouched = [r for r in range(n_slots * stride) if r not in written]
    assert np.all(planes[1][untouched] == 0xA5) and np.all(planes[3][untouched] == 0xA5)
    # a destination outside the planes is skipped and reported
    bad = entries.copy()
    bad[2] = stride
    csa2.cache_append(to_dev(H.view(np.int16)), G, d, to_dev(Wkv.view(np.int16)), to_dev(Wz.view(np.int16)),
                      to_dev(Wik.view(np.int16)), m, P, n_slots, to_dev(slots), to_dev(bad), ws,
                      kv_nr=kv_nr, pos=to_dev(pos) if nr else None)
    st, det = csa2.check(ws)
    assert st == 6 and det == stride


def _decided_e4m3(pre32, e, mids):
    """Elements whose E4M3 code is fixed within the bound e (saturated values stay decided)."""
    a = np.abs(pre32)
    dist = np.abs(a[..., None] - mids).min(-1)
    return (dist > e) | (a - e > 464.0)


@pytest.mark.parametrize("nr", [False, True])
def test_swa_append_ring(oracle_mod, nr):
    R, nq, n_win = 10, 3, 8
    rng = np.random.default_rng(5)
    x = (2.5 * rng.standard_normal((R, 512))).astype(np.float32)
    x[0, :16] = 500.0                                   # saturating values
    query = np.array([0, 1, 2, 0, 1, 2, 0, 1, 2, 0], np.int32)
    pos = np.array([0, 1, 2, 9, 12, 1_000_003, 3, -5, 7, 14], np.int64)  # 9 -> slot 1, -5 skipped
    w = (1.0 + 0.3 * rng.standard_normal(512)).astype(np.float32)
    ring = torch.full((nq, n_win, 512), 0xA5, dtype=torch.uint8, device="cuda")
    csa2.swa_append(to_dev(x), R, to_dev(pos), nq, ring, n_win, query=to_dev(query),
                    nr=csa2.norm_rope(to_dev(w), 1e-6, True, 10000.0) if nr else None)
    torch.cuda.synchronize()
    got = ring.cpu().numpy()
    mids = _e4m3_mids(oracle_mod)
    seen = set()
    for r in range(R):
        if pos[r] < 0:
            continue
        slot = (int(query[r]), int(pos[r] % n_win))
        assert slot not in seen
        seen.add(slot)
        ref, pre = oracle_mod.swa_row(x[r].astype(np.float64), w if nr else None, 1e-6,
                                      pos=float(pos[r]) if nr else None)
        g = got[slot[0], slot[1]]
        if not nr:
            assert np.array_equal(g, ref)               # the same fp32 value, the same encoder
        else:
            y = pre
            e = 32.0 * U * np.abs(y)
            ep = e[448::2] + e[449::2] + (3e-7 + 4.0 * U) * (np.abs(y[448::2]) + np.abs(y[449::2]))
            e[448::2] = ep
            e[449::2] = ep
            dec = _decided_e4m3(pre.astype(np.float32).astype(np.float64), e, mids)
            assert np.array_equal(g[dec], ref[dec])
            assert dec.mean() > 0.9
    for q in range(nq):
        for s in range(n_win):
            if (q, s) not in seen:
                assert np.all(got[q, s] == 0xA5)
    # the ring is the attention's window input: the order of its rows does not matter
    assert csa2.sparse_attn_workspace_size(nq, 0, n_win) > 0


def test_swa_append_records_positions():
    R, nq, n_win = 10, 3, 8
    x = np.random.default_rng(6).standard_normal((R, 512)).astype(np.float32)
    query = np.array([0, 1, 2, 0, 1, 2, 0, 1, 2, 0], np.int32)
    pos = np.array([0, 1, 2, 9, 12, 1_000_003, 3, -5, 7, 14], np.int64)
    ring = torch.zeros((nq, n_win, 512), dtype=torch.uint8, device="cuda")
    ring_pos = torch.full((nq, n_win), -1, dtype=torch.int64, device="cuda")
    csa2.swa_append(to_dev(x), R, to_dev(pos), nq, ring, n_win, query=to_dev(query), ring_pos=ring_pos)
    torch.cuda.synchronize()
    ref = np.full((nq, n_win), -1, np.int64)
    for r in range(R):
        if pos[r] >= 0:
            ref[query[r], pos[r] % n_win] = pos[r]
    assert np.array_equal(ring_pos.cpu().numpy(), ref)


def test_bounded_replay_window(oracle_mod):
    """SWA bounded replay ("DeepSeek-V4.1-Flash: pushing the limits of KV cache compression",
    section 6): after a replay from position s the query at position i sees the window rows
    at [max(s, i - n_win + 1), i] only.  The ring holds stale rows from before s beside the
    replayed ones; with the window bounds the attention equals the oracle's over exactly the
    visible rows (built on the host with the oracle's own row encoder)."""
    from parity import check_attention

    n_win, B, N, k = 128, 2, 700, 64
    c = SmallCache(oracle_mod, 13, B, N)
    rng = np.random.default_rng(13)
    q = W.attn_query(13, 0, B)
    topk = np.sort(np.stack([rng.choice(N, k, replace=False) for _ in range(B)]), axis=1).astype(np.int32)
    i_pos = np.array([1150, 1130], np.int64)   # the queries' positions
    s_rep = np.array([1100, 1000], np.int64)   # where each query's replay started
    ring = np.zeros((B, n_win, 512), np.uint8)
    ring_pos = np.full((B, n_win), -1, np.int64)
    for b in range(B):
        # stale rows (a pre-miss window), then the replay from s_rep[b] up to the query
        for p in list(range(int(i_pos[b]) - 250, int(s_rep[b]))) + list(range(int(s_rep[b]), int(i_pos[b]) + 1)):
            row, _ = oracle_mod.swa_row(2.0 * rng.standard_normal(512))
            ring[b, p % n_win] = row
            ring_pos[b, p % n_win] = p
    lo = np.maximum(s_rep, i_pos - n_win + 1)
    out = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, 64), dtype=torch.float32, device="cuda")
    ws = csa2.workspace(csa2.sparse_attn_workspace_size(B, k, n_win))
    win = csa2.window(to_dev(ring_pos), to_dev(lo))
    scale = 1.0 / np.sqrt(512.0)
    csa2.sparse_attn_decode(c.planes, B, to_dev(topk), k, to_dev(ring), n_win, to_dev(q.view(np.int16)), scale, out,
                            ws, lse_out=lse, win=win)
    assert csa2.check(ws)[0] == 0
    got, glse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        vis = ring_pos[b] >= lo[b]
        assert vis.sum() == min(n_win, i_pos[b] - lo[b] + 1)
        kvc, kvs, _, _ = c.oracle_slot(b)
        ro, rl = oracle_mod.attention(kvc, kvs, topk[b], ring[b][vis], q[b], scale)
        check_attention(got[b:b + 1], ro[None])
        assert np.allclose(glse[b], rl, rtol=1e-4, atol=1e-4)
    # a bound above every row: no window at all (and no entries: out = 0, lse = -inf)
    none = csa2.window(to_dev(ring_pos), to_dev(np.full(B, 10**9, np.int64)))
    csa2.sparse_attn_decode(c.planes, B, to_dev(topk), 0, to_dev(ring), n_win, to_dev(q.view(np.int16)), scale, out,
                            ws, lse_out=lse, win=none)
    assert csa2.check(ws)[0] == 0
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
