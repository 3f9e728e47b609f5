"""Per-kernel device timing of the library: while enabled, every launch of the
indexer call is counted with a positive device time; once disabled nothing more
is recorded."""
import numpy as np
import pytest

import compressed_sparse_attention_nvfp4_gb300 as csa2
from synth import workloads as W

pytestmark = pytest.mark.gpu


def test_kernel_times_count_launches(oracle_mod):
    from gpu_common import SmallCache, require_gpu, to_dev, torch

    require_gpu()
    B, n_max, k, keep = 2, 3000, 64, 100
    q, w = W.index_query(7, 0, B)
    c = SmallCache(oracle_mod, 7, B, n_max)
    ne = to_dev(np.array([n_max, n_max], np.int32))
    qd, wd = to_dev(q.view(np.int16)), to_dev(w)
    topk = torch.empty((B, k), dtype=torch.int32, device="cuda")
    ws = csa2.workspace(csa2.index_topk_workspace_size(B, n_max, k, 8, keep))
    csa2.timing_enable(True)
    try:
        for _ in range(3):
            csa2.index_topk(c.planes, B, ne, n_max, qd, wd, k, csa2.TOPK_HIER_BUILD, topk, ws, 8, keep)
        torch.cuda.synchronize()
        t = csa2.kernel_times()
    finally:
        csa2.timing_enable(False)
    assert t["k_scan_tc"][0] == 3 and t["k_scan_tc"][1] > 0.0
    assert sum(n for name, (n, _) in t.items() if name.startswith("k_select")) == 6  # pool + tokens
    csa2.index_topk(c.planes, B, ne, n_max, qd, wd, k, csa2.TOPK_HIER_BUILD, topk, ws, 8, keep)
    torch.cuda.synchronize()
    assert csa2.kernel_times() == {}
    assert csa2.check(ws)[0] == 0
