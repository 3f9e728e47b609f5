"""Failure detection without a GPU fault, and the cache as resumable state.

The bounded-wait self-test makes a device wait run out on a barrier nothing
completes: the kernel records CSA2_ERR_DEVICE_TIMEOUT in the workspace and exits,
the host reads it through csa2_check, and the context keeps working.  The cache
planes are plain caller-owned bytes: dumped to the host and loaded into a fresh
allocation they give the same top-k and attention, bit for bit."""
import numpy as np
import pytest

from gpu_common import SmallCache, csa2, require_gpu, to_dev, torch
from synth import workloads as W

pytestmark = pytest.mark.gpu
TIMEOUT = 5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("budget", [0, 2_000_000])
def test_wait_runs_out_and_is_reported(budget):
    ws = csa2.workspace(256)
    csa2.selftest_wait_timeout(budget, ws)
    st, detail = csa2.check(ws)
    assert st == TIMEOUT and detail >= budget
    assert csa2.check(ws)[0] == 0  # the check cleared it


def test_context_usable_after_timeout(oracle_mod):
    ws = csa2.workspace(256)
    csa2.selftest_wait_timeout(1_000_000, ws)
    assert csa2.check(ws)[0] == TIMEOUT
    x = np.random.default_rng(0).standard_normal((8, 512)).astype(np.float32)
    P = csa2.Planes.empty(1, 8)
    csa2.quantize_entries(P, to_dev(x), to_dev(np.zeros((8, 128), np.float32)), 8, 0)
    torch.cuda.synchronize()
    codes, scales = oracle_mod.quantize_main(x)
    assert np.array_equal(P.kv_codes.cpu().numpy(), codes) and np.array_equal(P.kv_scales.cpu().numpy(), scales)


def _decode(planes, B, N, q, w, qa, swa):
    ne = torch.full((B,), N, dtype=torch.int32, device="cuda")
    topk = torch.empty((B, 512), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_workspace_size(B, N, 512, 8, 64))
    csa2.index_topk(planes, B, ne, N, q, w, 512, csa2.TOPK_HIER_BUILD, topk, ws, 8, 64)
    out = torch.empty((B, 64, 512), dtype=torch.float32, device="cuda")
    wa = csa2.workspace(csa2.sparse_attn_workspace_size(B, 512, 128))
    csa2.sparse_attn_decode(planes, B, topk, 512, swa, 128, qa, 1.0 / np.sqrt(512.0), out, wa)
    assert csa2.check(ws)[0] == 0 and csa2.check(wa)[0] == 0
    return topk.cpu().numpy(), out.cpu().numpy()


def test_cache_dump_and_reload_gives_identical_decode(oracle_mod):
    B, N = 2, 3000
    c = SmallCache(oracle_mod, 12, B, N)
    qi, wi = W.index_query(12, 0, B)
    q, w = to_dev(qi.view(np.int16)), to_dev(wi)
    qa = to_dev(W.attn_query(12, 0, B).view(np.int16))
    swa = to_dev(np.ascontiguousarray(W.swa_rows(12, 0, B, 128)))
    t0, o0 = _decode(c.planes, B, N, q, w, qa, swa)
    dump = [t.cpu().numpy().copy() for t in (c.planes.kv_codes, c.planes.kv_scales, c.planes.ix_codes,
                                            c.planes.ix_scales)]
    fresh = csa2.Planes.empty(B, N)
    for dst, src in zip((fresh.kv_codes, fresh.kv_scales, fresh.ix_codes, fresh.ix_scales), dump):
        dst.copy_(torch.from_numpy(src))
    t1, o1 = _decode(fresh, B, N, q, w, qa, swa)
    assert np.array_equal(t0, t1) and np.array_equal(o0, o1)
