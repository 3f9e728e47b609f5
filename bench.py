#!/usr/bin/env python3
"""CSA2 decode benchmark on one GB300.

Default workload: batch 32 decode queries, each over its own 1,048,576-entry
decoder Full-layer cache (m = 1, 356 B/entry, 11.95 GB resident), hierarchical
indexer (131,072 blocks of 8 -> top 2,048 blocks -> token top-512) followed by
64-head x 512 sparse MQA over the 512 selected entries plus a 128-row FP8
sliding window.  One step = one csa2_index_topk(HIER_BUILD) + one
csa2_sparse_attn_decode over the whole batch.  Metric: decode queries/s.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA2 decode queries/s at 1M ctx; achieved HBM GB/s vs GB300 peak"
UNIT = "queries/s"
WORKLOAD = ("batch 32 decode queries, 1,048,576-entry decoder Full-layer FP4 cache per query (m=1), "
            "hierarchical indexer 131,072 blocks -> 2,048 blocks -> top-512, "
            "64x512 sparse MQA over 512 selected + 128 FP8 SWA rows")
B, N, K_TOP, KEEP, BLOCK, NSWA, SEED = 32, 1 << 20, 512, 2048, 8, 128, 2
IDX_BYTES, MAIN_BYTES, SWA_ROW = 68, 288, 512


def kernel_fingerprint() -> str:
    """Hash of the sources of the scan kernel, to match ncu traffic records."""
    h = hashlib.sha256()
    for f in ("index_scan.cu", "index_scan.cuh", "ptx.cuh", "codec.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "compressed_sparse_attention_nvfp4_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(fp: str):
    """DRAM bytes per k_scan_tc launch from profiles/traffic_scan.txt if taken on these sources."""
    path = os.path.join(ROOT, "profiles", "traffic_scan.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split("#", 1)[0].split()
        if len(parts) >= 2 and parts[0] == fp:
            return float(parts[1])
    return None


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth (context next to the measured peak)


def host_cpu() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    import platform
    import subprocess

    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


NVML_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                    0x40: "hw_thermal_slowdown"}


class NvmlQueries:
    """Read-only NVML queries (ctypes on the driver's libnvidia-ml): the SM clock, its
    maximum, the power draw and the active clock-event reasons of one GPU."""

    def __init__(self, uuid=None, index=0, lib=None):
        import ctypes

        self.ct = ctypes
        self.L = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
        if self.L.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if uuid:
            rc = self.L.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid.encode()), ctypes.byref(self.h))
        if rc != 0:
            rc = self.L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the device")
        v = ctypes.c_uint(0)
        self.max_mhz = float(v.value) if self.L.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(v)) == 0 else None
        self._reasons = getattr(self.L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.L.nvmlDeviceGetCurrentClocksThrottleReasons

    def sample(self, with_power: bool):
        """(sm_mhz, power_w or None, reason mask) now."""
        ct = self.ct
        mhz, mw, mask = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        if self.L.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) != 0:  # NVML_CLOCK_SM
            return None
        if self._reasons(self.h, ct.byref(mask)) != 0:
            return None
        pw = None
        if with_power and self.L.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw)) == 0:
            pw = mw.value / 1000.0
        return float(mhz.value), pw, int(mask.value)


def cuda_uuid(local_rank: int):
    """NVML's UUID string of the CUDA device (None if torch does not report one)."""
    try:
        import torch

        u = getattr(torch.cuda.get_device_properties(local_rank), "uuid", None)
    except Exception:  # noqa: BLE001
        return None
    if u is None:
        return None
    u = str(u)
    return u if u.startswith("GPU-") else "GPU-" + u


def physical_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p.strip() for p in vis.split(",") if p.strip()]
    if local_rank < len(parts) and parts[local_rank].isdigit():
        return int(parts[local_rank])
    return local_rank


class FastClockSampler:
    """SM clock and clock-event reasons sampled every `period_s` (default 1 ms) by a thread
    calling NVML directly, so that even a timed region of a few milliseconds holds several
    samples.  mark() opens the timed region and stop() closes it; summary() reports the
    samples between the two only.  `queries` is an NvmlQueries (or a stand-in in tests)."""

    def __init__(self, queries, period_s: float = 0.001):
        self.q = queries
        self.period = period_s
        self.samples = []  # (sm_mhz, power_w, mask)
        self.lo = self.hi = None
        self._run = False
        self._thread = None

    def _loop(self):
        n = 0
        while self._run:
            s = self.q.sample(with_power=(n % 20 == 0))
            if s is not None:
                self.samples.append(s)
            n += 1
            time.sleep(self.period)

    def __enter__(self):
        self._run = True
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5.0:
            time.sleep(0.001)
        return self

    def __exit__(self, *a):
        self._run = False
        if self._thread:
            self._thread.join(timeout=5.0)

    def mark(self):
        self.lo = len(self.samples)

    def stop(self):
        self.hi = len(self.samples)

    def summary(self):
        lo = self.lo or 0
        hi = self.hi if self.hi is not None else len(self.samples)
        rows = self.samples[lo:hi]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.q.max_mhz, "reasons": ["no samples"]}
        reasons = sorted({name for _, _, m in rows for bit, name in NVML_REASON_BITS.items() if m & bit})
        pw = [p for _, p, _ in rows if p is not None]
        out = {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": self.q.max_mhz,
               "sm_mhz_min": min(r[0] for r in rows), "reasons": reasons, "samples": len(rows),
               "window": "timed region only", "source": f"NVML every {self.period * 1e3:g} ms"}
        if pw:
            out["power_w_max"] = max(pw)
        return out


def clock_sampler(local_rank: int):
    """The fast NVML sampler when the driver's NVML loads, else nvidia-smi every 200 ms."""
    try:
        return FastClockSampler(NvmlQueries(cuda_uuid(local_rank), physical_index(local_rank)))
    except (OSError, AttributeError):
        return ClockSampler(physical_index(local_rank))


class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running (the fallback when
    NVML cannot be loaded directly)."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None
        self.offset = 0  # samples before this file offset were taken before the timed region
        self.end = None  # file size when the timed region closed

    def mark(self):
        """Call at the start of the timed region: later samples only are summarised."""
        if self.proc:
            self.offset = os.path.getsize(self.file.name)

    def stop(self):
        """Call at the end of the timed region: later samples are not summarised."""
        if self.proc:
            self.end = os.path.getsize(self.file.name)

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        # start timing only once the sampler is up: nvidia-smi's startup can hold the
        # driver for a second or more, which would land inside a short timed region
        t0 = time.time()
        while self.proc and self.proc.poll() is None and time.time() - t0 < 15.0:
            if os.path.getsize(self.file.name) > 0:
                break
            time.sleep(0.05)
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as fh:
            fh.seek(self.offset)
            text = fh.read() if self.end is None else fh.read(max(self.end - self.offset, 0))
            lines = text.splitlines()
        if self.offset and lines:
            lines = lines[1:]  # may be a sample cut at the offset
        for line in lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) >= 8:
                try:
                    rows.append((float(f[0]), float(f[1]), f[4:8]))
                except ValueError:
                    pass
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "window": "timed region only",
                "source": "nvidia-smi every 200 ms"}


# ----------------------------------------------------------------------------- oracle sample

def oracle_planes_query(b: int, threads: int):
    """The oracle's encoding of query b's whole 1,048,576-entry cache, and its inputs."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from synth import workloads as W

    q, w = W.index_query(SEED, 0, B)
    hv = W.hot_vectors(q, w, 3.0)
    chunk = 1 << 16

    def encode(j0):
        cnt = min(chunk, N - j0)
        kv = oracle.quantize_main(W.main_latents(SEED, 0, B, N, b, j0, cnt))
        ix = oracle.quantize_index(W.index_latents(SEED, 0, B, N, b, j0, cnt, 0.02, hv[b]))
        return j0, kv, ix

    kvc = np.empty((N, 256), np.uint8)
    kvs = np.empty((N, 32), np.uint8)
    ixc = np.empty((N, 64), np.uint8)
    ixs = np.empty((N, 4), np.uint8)
    with ThreadPoolExecutor(threads) as ex:
        for j0, (c1, s1), (c2, s2) in ex.map(encode, range(0, N, chunk)):
            kvc[j0:j0 + c1.shape[0]], kvs[j0:j0 + c1.shape[0]] = c1, s1
            ixc[j0:j0 + c2.shape[0]], ixs[j0:j0 + c2.shape[0]] = c2, s2
    return (kvc, kvs, ixc, ixs), q[b], w[b], W.attn_query(SEED, 0, B)[b], W.swa_rows(SEED, 0, B)[b]


def oracle_query_path(planes, q, w, qa, swa, threads, scores=None):
    """One query's whole path in the oracle: scores (unless given), block maxima, pool,
    top-512 within the pool, attention over the selection and the window."""
    import oracle

    kvc, kvs, ixc, ixs = planes
    s = oracle.index_scores(ixc, ixs, q, w, nthreads=threads) if scores is None else scores
    pool = oracle.hier_pool(oracle.block_max(s, BLOCK), KEEP)
    sel = oracle.pool_topk(s, pool, BLOCK, K_TOP)
    oracle.attention(kvc, kvs, sel, swa, qa, 1 / math.sqrt(512))


def oracle_sample(n_queries: int, steps: int, warmup: int = 0):
    """Time the CPU oracle on `n_queries` of the workload's queries (full 1M-entry caches),
    after `warmup` untimed passes.  Returns (queries/s, threads, description).  Setup (input
    synthesis, encoding) is untimed."""
    threads = os.cpu_count() or 1
    data = [oracle_planes_query(b, threads) for b in range(n_queries)]
    for _ in range(warmup):
        for d in data:
            oracle_query_path(*d, threads)
    t0 = time.perf_counter()
    for _ in range(steps):
        for d in data:
            oracle_query_path(*d, threads)
    dt = time.perf_counter() - t0
    desc = (f"{n_queries} of the {B} queries at the full 1,048,576-entry context, {steps} pass(es): "
            f"oracle scores (fp64, {threads} threads), block max, pool, top-512, attention")
    return n_queries * steps / dt, threads, desc


REF_BUDGET_S = 150.0  # timed CPU work of the reference arm, at most


def oracle_reference_steps(steps: int, warmup: int):
    """The reference arm: `steps` timed steps of the oracle after `warmup` untimed ones.
    A step is one query's whole path (query 0 of the workload, full context) while
    steps x (one query's time) fits REF_BUDGET_S; beyond that each step scores one of f
    equal slices of the query's entries, and every f-th step also runs the selection and
    attention of the query just completed, so that f steps do one query's work.
    Returns (queries/s, threads, description, f)."""
    import numpy as np

    import oracle

    threads = os.cpu_count() or 1
    planes, q, w, qa, swa = oracle_planes_query(0, threads)
    t_q = None
    for i in range(max(warmup, 1)):  # at least one untimed pass, which also sizes the steps
        t0 = time.perf_counter()
        oracle_query_path(planes, q, w, qa, swa, threads)
        t_q = time.perf_counter() - t0
    f = max(1, math.ceil(steps * t_q / REF_BUDGET_S))
    kvc, kvs, ixc, ixs = planes
    bounds = [N * i // f for i in range(f + 1)]
    scores = np.empty(N, np.float64)
    t0 = time.perf_counter()
    for st in range(steps):
        if f == 1:
            oracle_query_path(planes, q, w, qa, swa, threads)
            continue
        sl = st % f
        lo, hi = bounds[sl], bounds[sl + 1]
        scores[lo:hi] = oracle.index_scores(ixc[lo:hi], ixs[lo:hi], q, w, nthreads=threads)
        if sl == f - 1:
            oracle_query_path(planes, q, w, qa, swa, threads, scores=scores)
    dt = time.perf_counter() - t0
    if f == 1:
        desc = (f"query 0 of the {B} at the full 1,048,576-entry context, one query per step: oracle scores "
                f"(fp64, {threads} threads), block max, pool, top-512, attention")
    else:
        desc = (f"query 0 of the {B} at the full 1,048,576-entry context; each step scores 1/{f} of its "
                f"entries (fp64, {threads} threads) and every {f}th step runs the block max, pool, top-512 and "
                f"attention of the completed query, so {f} steps = one query (rate = steps / {f} / time)")
    return steps / f / dt, threads, desc, f


# ----------------------------------------------------------------------------- GPU arm

CW_T, CW_D, CW_M, CW_SEED = 131072, 5120, 2, 3
CW_WORKLOAD = ("prefill cache write: T=131,072 tokens x d_model 5120, m=2 -> 65,536 entries "
               "(C,Z = H[W_KV|W_Z], softmax pooling, K^I = Cbar W_IK, codec; 23.3 MB of cache)")


def run_cache_write(dev, st, calls: int, warmup: int):
    """The prefill cache write (one csa2_cache_write call per step) on seeded device inputs:
    ms per call, whole-call TFLOP/s, and k_cw_tc's own TFLOP/s against the measured bf16 peak."""
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    import synth
    from synth import workloads as W

    T, d, m = CW_T, CW_D, CW_M
    n = T // m
    H = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    Wkv = torch.empty((d, 512), dtype=torch.bfloat16, device=dev)
    Wz = torch.empty((d, 512), dtype=torch.bfloat16, device=dev)
    Wik = torch.empty((512, 128), dtype=torch.bfloat16, device=dev)
    ss = st.cuda_stream
    synth.dev_normal_bf16(CW_SEED, W.TID_H, T * d, H.data_ptr(), ss)
    synth.dev_normal_bf16(CW_SEED, W.TID_WKV, d * 512, Wkv.data_ptr(), ss, scale=1.0 / math.sqrt(d))
    synth.dev_normal_bf16(CW_SEED, W.TID_WZ, d * 512, Wz.data_ptr(), ss, scale=1.0 / math.sqrt(d))
    synth.dev_normal_bf16(CW_SEED, W.TID_WIK, 512 * 128, Wik.data_ptr(), ss, scale=1.0 / math.sqrt(512))
    P = csa2.Planes.empty(1, n, dev)
    ws = csa2.workspace(csa2.cache_write_workspace_size(T, d, m), dev)
    torch.cuda.synchronize()

    def call():
        csa2.cache_write(H, T, d, Wkv, Wz, Wik, m, P, 0, 0, ws, stream=st)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    assert csa2.check(ws, st)[0] == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(calls):
        call()
    b.record(st)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / calls
    csa2.timing_enable(True)
    for _ in range(calls):
        call()
    torch.cuda.synchronize()
    kt = csa2.kernel_times()
    csa2.timing_enable(False)
    assert csa2.check(ws, st)[0] == 0
    gemm_flop = 2.0 * T * d * 2 * 512
    all_flop = gemm_flop + 2.0 * n * 512 * 128
    tc_n, tc_ms = kt.get("k_cw_tc", (0, 0.0))
    tc_avg = tc_ms / max(tc_n, 1)
    achieved = gemm_flop / (tc_avg * 1e-3) / 1e12 if tc_n else 0.0
    peak, kind = tensor_peak()
    return {
        "workload": CW_WORKLOAD, "calls": calls, "ms_per_call": round(ms, 4),
        "tflops_per_call": round(all_flop / (ms * 1e-3) / 1e12, 1),
        "kernels_ms_per_launch": {k: round(t / max(c, 1), 4) for k, (c, t) in sorted(kt.items())},
        "roofline": {"kernel": "k_cw_tc (bf16 tcgen05 GEMM + pooling)", "bound": "tensor",
                     "achieved": round(achieved, 1), "peak": peak, "peak_kind": kind, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4) if peak else None,
                     "algorithmic_flop_per_launch": gemm_flop, "launch_ms": round(tc_avg, 4)},
    }


ST_B, ST_CTX, ST_SEED = 128, 262144, 4
ST_WORKLOAD = ("40-layer V4.1 decode step: batch 128 at a 262,144-token context; layers 0-1 SWA only, "
               "encoder 3 x (Full + 5 Reuse) at m=2 (131,072 entries), decoder (Full + 3 Reuse) + "
               "4 x (Reindex + 3 Reuse) at m=1 (262,144 entries, 2,048-block pool), top-512 + 128-row "
               "FP8 window in every layer")


def run_step40(dev, st, steps: int, warmup: int):
    """One decode step over the 40-layer schedule (schedule.run_step) on seeded device inputs."""
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    from compressed_sparse_attention_nvfp4_gb300 import schedule as SCH
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    B, T = ST_B, ST_CTX
    t = csa2.v41_layer_table()
    full = [l for l in range(40) if t["mode"][l] == csa2.LAYER_FULL]
    n_of = {f: T // t["m"][f] for f in full}
    with torch.cuda.stream(st):
        kv, ne, nm = {}, {}, {}
        for f in full:
            kv[f] = csa2.Planes.empty(B, n_of[f], dev)
            WL.fill_planes(kv[f], ST_SEED, f, B, n_of[f], stream=st)
            ne[f] = torch.full((B,), n_of[f], dtype=torch.int32, device=dev)
            nm[f] = n_of[f]
        qidx, w, q, swa, out = {}, {}, {}, {}, {}
        for l in range(40):
            if t["mode"][l] in (csa2.LAYER_FULL, csa2.LAYER_REINDEX):
                qidx[l], w[l], _, _ = WL.index_query_dev(ST_SEED, l, B, dev)
            q[l], _ = WL.attn_query_dev(ST_SEED, l, B, dev)
            swa[l] = WL.swa_dev(ST_SEED, l, B, NSWA, dev, stream=st)
            out[l] = torch.empty((B, 64, 512), dtype=torch.float32, device=dev)
        buf = SCH.StepBuffers(B=B, kv=kv, n_entries=ne, n_max=nm, qidx=qidx, w=w, q=q, swa=swa, out=out,
                              k=K_TOP, n_blocks_keep=KEEP)
        SCH.allocate_scratch(buf, dev)
        # a second batch's outputs and scratch: two independent batches in flight on two
        # streams (the inputs are shared; each batch writes its own outputs and workspaces)
        import dataclasses
        buf2 = dataclasses.replace(buf, out={l: torch.empty_like(o) for l, o in out.items()}, topk={}, pool={},
                                   stage={})
        SCH.allocate_scratch(buf2, dev)
        st2 = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    for _ in range(warmup):
        SCH.run_step(buf, stream=st)
        SCH.run_step(buf2, stream=st2)
    torch.cuda.synchronize()
    for bb, ss in ((buf, st), (buf2, st2)):
        assert csa2.check(bb.ws_index, ss)[0] == 0 and csa2.check(bb.ws_attn, ss)[0] == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def two_in_flight():  # step s runs batch s % 2 on stream s % 2
        a.record(st)
        st2.wait_event(a)
        for s_i in range(steps):
            n_calls = SCH.run_step(buf if s_i % 2 == 0 else buf2, stream=st if s_i % 2 == 0 else st2)
        j = torch.cuda.Event()
        j.record(st2)
        st.wait_event(j)
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps, n_calls

    def one_in_flight():  # each step after the one before
        a.record(st)
        for _ in range(steps):
            SCH.run_step(buf, stream=st)
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    # the median of three timed runs of the K steps each (the step is short, so one run
    # of a few steps varies by a few per cent from box to box)
    runs = [two_in_flight() for _ in range(3)]
    calls = runs[0][1]
    ms = sorted(r[0] for r in runs)[1]
    ms1 = sorted(one_in_flight() for _ in range(3))[1]
    csa2.timing_enable(True)
    SCH.run_step(buf, stream=st)
    torch.cuda.synchronize()
    kt = csa2.kernel_times()
    csa2.timing_enable(False)
    assert csa2.check(buf.ws_index, st)[0] == 0 and csa2.check(buf.ws_attn, st)[0] == 0
    # algorithmic bytes: every Full layer's keys once, each Reindex layer's pool, and
    # every attention layer's selected entries and window rows
    # the same step replayed from a CUDA graph (captured once; no host work per step)
    graph = {"captured": False}
    try:
        g = SCH.capture_step(buf, st)
        with torch.cuda.stream(st):  # replay() launches on the current stream
            for _ in range(warmup):
                g.replay()
            torch.cuda.synchronize()
            a.record(st)
            for _ in range(steps):
                g.replay()
            b.record(st)
        torch.cuda.synchronize()
        assert csa2.check(buf.ws_index, st)[0] == 0 and csa2.check(buf.ws_attn, st)[0] == 0
        gms = a.elapsed_time(b) / steps
        graph = {"captured": True, "ms_per_step": round(gms, 4), "queries_per_s": round(B / (gms * 1e-3), 1)}
    except Exception as e:  # report, do not fail the bench line
        graph = {"captured": False, "error": str(e)[:200]}
    n_reindex = sum(1 for l in range(40) if t["mode"][l] == csa2.LAYER_REINDEX)
    n_attn_sel = sum(1 for l in range(40) if t["mode"][l] != csa2.LAYER_SWA)
    step_bytes = B * (sum(n_of.values()) * IDX_BYTES + n_reindex * KEEP * BLOCK * IDX_BYTES
                      + n_attn_sel * K_TOP * MAIN_BYTES + 40 * NSWA * SWA_ROW)
    hbm, kind = peaks()
    achieved = step_bytes / (ms * 1e-3) / 1e9
    return {
        "workload": ST_WORKLOAD, "steps": steps, "timed_runs": "median of 3", "library_calls_per_step": calls,
        "ms_per_step": round(ms, 4), "queries_per_s": round(B / (ms * 1e-3), 1),
        "in_flight": {"batches": 2, "one_batch_ms_per_step": round(ms1, 4),
                      "one_batch_queries_per_s": round(B / (ms1 * 1e-3), 1)},
        "kernels_ms_per_step": {k: round(tm, 4) for k, (n, tm) in sorted(kt.items())},
        "hbm": {"algorithmic_bytes": step_bytes, "achieved_gbs": round(achieved, 1), "peak": hbm,
                "peak_kind": kind, "frac": round(achieved / hbm, 4)},
        "cuda_graph": graph,
    }


AT_B, AT_N, AT_SEED = 128, 65536, 5
AT_WORKLOAD = ("sparse MQA decode attention alone: batch 128, 64 heads x 512 channels, top-512 "
               "FP4 entries of a 65,536-entry cache + 128 FP8 window rows per query")


def run_attention(dev, st, steps: int, warmup: int):
    """csa2_sparse_attn_decode alone at the 40-layer step's batch (one CTA per query)."""
    import numpy as np
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    B, Nn = AT_B, AT_N
    rng = np.random.default_rng(AT_SEED)
    sel = np.sort(np.stack([rng.choice(Nn, K_TOP, replace=False) for _ in range(B)]), axis=1)
    with torch.cuda.stream(st):
        planes = csa2.Planes.empty(B, Nn, dev)
        WL.fill_planes(planes, AT_SEED, 0, B, Nn, stream=st)
        q, _ = WL.attn_query_dev(AT_SEED, 0, B, dev)
        swa = WL.swa_dev(AT_SEED, 0, B, NSWA, dev, stream=st)
        topk = torch.from_numpy(sel.astype(np.int32)).to(dev)
        out = torch.empty((B, 64, 512), dtype=torch.float32, device=dev)
        lse = torch.empty((B, 64), dtype=torch.float32, device=dev)
        ws = csa2.workspace(csa2.sparse_attn_workspace_size(B, K_TOP, NSWA), dev)
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(512)

    def call():
        csa2.sparse_attn_decode(planes, B, topk, K_TOP, swa, NSWA, q, scale, out, ws, lse_out=lse, stream=st)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    assert csa2.check(ws, st)[0] == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(steps):
        call()
    b.record(st)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    csa2.timing_enable(True)
    for _ in range(min(steps, 20)):
        call()
    torch.cuda.synchronize()
    kt = csa2.kernel_times()
    csa2.timing_enable(False)
    n_k, t_k = kt["k_attn"]
    k_ms = t_k / n_k
    # the same call with the in-layer extras on: query RMSNorm + RoPE (output turned
    # back) at positions near 10^6, a sink logit per head
    w = torch.ones(512, dtype=torch.float32, device=dev)
    pos = torch.arange(1_000_000, 1_000_000 + B, dtype=torch.int64, device=dev)
    sink = torch.zeros(64, dtype=torch.float32, device=dev)
    nr = csa2.norm_rope(w, 1e-6, True, 10000.0)

    def call_ex():
        csa2.sparse_attn_decode(planes, B, topk, K_TOP, swa, NSWA, q, scale, out, ws, lse_out=lse, stream=st,
                                q_nr=nr, q_pos=pos, sink=sink)

    for _ in range(warmup):
        call_ex()
    a.record(st)
    for _ in range(steps):
        call_ex()
    b.record(st)
    torch.cuda.synchronize()
    assert csa2.check(ws, st)[0] == 0
    ms_ex = a.elapsed_time(b) / steps
    # algorithmic bytes: selected entries, window rows, q in, output out; flops: S and O
    rows = K_TOP + NSWA
    call_bytes = B * (K_TOP * MAIN_BYTES + NSWA * SWA_ROW + 64 * 512 * 2 + 64 * 512 * 4)
    call_flop = B * rows * 64 * 512 * 2 * 2
    hbm, kind = peaks()
    tp, tkind = tensor_peak()
    return {
        "workload": AT_WORKLOAD, "calls": steps, "ms_per_call": round(ms, 4),
        "ms_per_call_with_norm_rope_sink": round(ms_ex, 4),
        "kernels_ms_per_launch": {k: round(tm / n, 4) for k, (n, tm) in sorted(kt.items())},
        "k_attn": {"algorithmic_bytes": call_bytes, "hbm_gbs": round(call_bytes / (k_ms * 1e-3) / 1e9, 1),
                   "hbm_frac": round(call_bytes / (k_ms * 1e-3) / 1e9 / hbm, 4), "hbm_peak_kind": kind,
                   "flop": call_flop, "tflops": round(call_flop / (k_ms * 1e-3) / 1e12, 1),
                   "tensor_frac": round(call_flop / (k_ms * 1e-3) / 1e12 / tp, 4), "tensor_peak_kind": tkind},
    }


def run_append(dev, st, calls: int, warmup: int):
    """Per-step decode writes at batch 128: the decoder layer's append (one entry per query,
    m = 1, d_model 5120, RMSNorm + RoPE) and one window row per query."""
    import numpy as np
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    import synth
    from synth import workloads as W

    G, d, m, stride = AT_B, CW_D, 1, 4096
    ss = torch.cuda.current_stream(dev).cuda_stream
    with torch.cuda.stream(st):
        H = torch.empty((G, d), dtype=torch.int16, device=dev)
        Wkv = torch.empty((d, 512), dtype=torch.int16, device=dev)
        Wz = torch.empty((d, 512), dtype=torch.int16, device=dev)
        Wik = torch.empty((512, 128), dtype=torch.int16, device=dev)
    synth.dev_normal_bf16(CW_SEED, W.TID_H, G * d, H.data_ptr(), ss)
    synth.dev_normal_bf16(CW_SEED, W.TID_WKV, d * 512, Wkv.data_ptr(), ss, scale=1.0 / math.sqrt(d))
    synth.dev_normal_bf16(CW_SEED, W.TID_WZ, d * 512, Wz.data_ptr(), ss, scale=1.0 / math.sqrt(d))
    synth.dev_normal_bf16(CW_SEED, W.TID_WIK, 512 * 128, Wik.data_ptr(), ss, scale=1.0 / math.sqrt(512))
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        P = csa2.Planes.empty(G, stride, dev)
        slot = torch.arange(G, dtype=torch.int32, device=dev)
        entry = torch.full((G,), 4000, dtype=torch.int64, device=dev)
        pos = entry + 0
        w = torch.ones(512, dtype=torch.float32, device=dev)
        ws = csa2.workspace(csa2.cache_append_workspace_size(G, d, m), dev)
        x = torch.randn((G, 512), dtype=torch.float32, device=dev)
        ring = torch.zeros((G, NSWA, 512), dtype=torch.uint8, device=dev)
    nr = csa2.norm_rope(w, 1e-6, True, 10000.0)

    def append():
        csa2.cache_append(H, G, d, Wkv, Wz, Wik, m, P, G, slot, entry, ws, kv_nr=nr, pos=pos, stream=st)

    def window():
        csa2.swa_append(x, G, pos, G, ring, NSWA, nr=nr, stream=st)

    out = {"workload": f"decode-time writes, batch {G}: one cache entry per query (m = 1, d_model {d}, "
                       "RMSNorm + RoPE, E2M1/E4M3 + MXFP4 planes) and one E4M3 window row per query"}
    for name, fn in (("cache_append", append), ("swa_append", window)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(calls):
            fn()
        b.record(st)
        torch.cuda.synchronize()
        out[name + "_ms_per_call"] = round(a.elapsed_time(b) / calls, 4)
    assert csa2.check(ws, st)[0] == 0
    csa2.timing_enable(True)
    append()
    window()
    torch.cuda.synchronize()
    out["kernels_ms_per_launch"] = {k: round(t / n, 4) for k, (n, t) in sorted(csa2.kernel_times().items())}
    csa2.timing_enable(False)
    return out


PF_N, PF_Q, PF_SEED = 131072, 2048, 6
PF_WORKLOAD = ("prefill indexer of an encoder Full layer: 2,048 queries of one 262,144-token sequence "
               "(131,072 entries at m = 2), query i sees the entries of the 128 (i + 1) tokens before it, "
               "top-512 each")


def run_prefill_index(dev, st, calls: int, warmup: int):
    """csa2_index_topk_prefill: every query scores the visible prefix of one shared slot."""
    import numpy as np
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL

    N, Q = PF_N, PF_Q
    n_vis = ((np.arange(Q, dtype=np.int64) + 1) * (2 * N // Q) // 2).astype(np.int32)  # token 128 (i + 1), m = 2
    with torch.cuda.stream(st):
        planes = csa2.Planes.empty(1, N, dev)
        WL.fill_planes(planes, PF_SEED, 0, 1, N, stream=st)
        q, w, _, _ = WL.index_query_dev(PF_SEED, 0, Q, dev)
        nv = torch.from_numpy(n_vis).to(dev)
        topk = torch.empty((Q, K_TOP), dtype=torch.int32, device=dev)
        ws = csa2.workspace(csa2.index_topk_prefill_workspace_size(Q, N, K_TOP), dev)
    torch.cuda.synchronize()

    def call():
        csa2.index_topk_prefill(planes, 0, Q, nv, N, q, w, K_TOP, topk, ws, stream=st)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    assert csa2.check(ws, st)[0] == 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(calls):
        call()
    b.record(st)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / calls
    csa2.timing_enable(True)
    call()
    torch.cuda.synchronize()
    kt = csa2.kernel_times()
    csa2.timing_enable(False)
    scored = int(n_vis.astype(np.int64).sum())
    flop = scored * 32 * 128 * 2  # q_h . K_j for 32 heads of 128
    # the same call with MXFP4 indexer queries (csa2_quantize_index_query, as V4 quantizes
    # the indexer q): the scan needs only the hi half of each query then
    with torch.cuda.stream(st):
        q4 = torch.empty_like(q)
    csa2.quantize_index_query(q, Q * 32, q4, stream=st)

    def call4():
        csa2.index_topk_prefill(planes, 0, Q, nv, N, q4, w, K_TOP, topk, ws, stream=st)

    for _ in range(warmup):
        call4()
    torch.cuda.synchronize()
    a.record(st)
    for _ in range(calls):
        call4()
    b.record(st)
    torch.cuda.synchronize()
    ms4 = a.elapsed_time(b) / calls
    csa2.timing_enable(True)
    call4()
    torch.cuda.synchronize()
    kt4 = csa2.kernel_times()
    csa2.timing_enable(False)
    assert csa2.check(ws, st)[0] == 0
    return {
        "workload": PF_WORKLOAD, "calls": calls, "ms_per_call": round(ms, 4),
        "queries_per_s": round(Q / (ms * 1e-3), 1), "entries_scored_per_call": scored,
        "entries_scored_per_s": round(scored / (ms * 1e-3), 1),
        "score_tflops": round(flop / (ms * 1e-3) / 1e12, 1),
        "kernels_ms_per_launch": {k: round(t / n, 4) for k, (n, t) in sorted(kt.items())},
        "mxfp4_query": {"ms_per_call": round(ms4, 4), "queries_per_s": round(Q / (ms4 * 1e-3), 1),
                        "score_tflops": round(flop / (ms4 * 1e-3) / 1e12, 1),
                        "kernels_ms_per_launch": {k: round(t / n, 4) for k, (n, t) in sorted(kt4.items())}},
    }


V4_T, V4_D, V4_M, V4_MH, V4_SEED = 65536, 4096, 4, 128, 7
V4_B, V4_N = 32, 8192
V4_WORKLOAD = ("V4 compressors on a prefill chunk of T=65,536 tokens x d_model 4096: the two-path "
               "overlapping CSA compressor at m=4 (16,384 entries) and the HCA compressor at m'=128 "
               "(512 entries); HCA dense decode attention: batch 32, every one of 8,192 entries "
               "(a 1,048,576-token context at m'=128) + 128 window rows")


def run_v4(dev, st, calls: int, warmup: int):
    """The V4 compressor variants (csa2_compress_overlap, csa2_compress_hca) and the HCA
    dense attention (csa2_dense_attn_decode) on seeded device inputs."""
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    import synth
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL
    from synth import workloads as W

    T, d, m, mh = V4_T, V4_D, V4_M, V4_MH
    ss = st.cuda_stream
    sd = 1.0 / math.sqrt(d)
    H = torch.empty((T, d), dtype=torch.bfloat16, device=dev)
    synth.dev_normal_bf16(V4_SEED, W.TID_H, T * d, H.data_ptr(), ss)
    Ws = {}
    for name, tid in (("a_kv", W.TID_WA_KV), ("b_kv", W.TID_WB_KV), ("a_z", W.TID_WA_Z), ("b_z", W.TID_WB_Z),
                      ("kv", W.TID_WKV), ("z", W.TID_WZ)):
        Ws[name] = torch.empty((d, 512), dtype=torch.bfloat16, device=dev)
        synth.dev_normal_bf16(V4_SEED, tid, d * 512, Ws[name].data_ptr(), ss, scale=sd)
    Bs = {}
    for name, tid, rows in (("a", W.TID_BA, m), ("b", W.TID_BB, m), ("h", W.TID_BHCA, mh)):
        Bs[name] = torch.empty((rows, 512), dtype=torch.float32, device=dev)
        synth.dev_normal_f32(V4_SEED, tid, rows * 512, Bs[name].data_ptr(), ss, scale=W.BIAS_SD)
    out_o = torch.empty((T // m, 512), dtype=torch.float32, device=dev)
    out_h = torch.empty((T // mh, 512), dtype=torch.float32, device=dev)
    ws = csa2.workspace(csa2.compress_workspace_size(T, d), dev)
    torch.cuda.synchronize()

    def overlap():
        csa2.compress_overlap(H, T, d, Ws["a_kv"], Ws["b_kv"], Ws["a_z"], Ws["b_z"], Bs["a"], Bs["b"], m, out_o,
                              ws, stream=st)

    def hca():
        csa2.compress_hca(H, T, d, Ws["kv"], Ws["z"], Bs["h"], mh, out_h, ws, stream=st)

    def timed(fn, n):
        for _ in range(warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(st)
        for _ in range(n):
            fn()
        b.record(st)
        torch.cuda.synchronize()
        csa2.timing_enable(True)
        fn()
        torch.cuda.synchronize()
        kt = csa2.kernel_times()
        csa2.timing_enable(False)
        return a.elapsed_time(b) / n, kt

    peak, kind = tensor_peak()
    hbm, hkind = peaks()
    res = {"workload": V4_WORKLOAD}
    for name, fn, paths, pool_kernel, mm in (("compress_overlap", overlap, 2, "k_pool_overlap", m),
                                            ("compress_hca", hca, 1, "k_pool_bias", mh)):
        ms, kt = timed(fn, calls)
        assert csa2.check(ws, st)[0] == 0
        gemm_flop = 2.0 * T * d * 2 * 512  # one path: C and Z
        tc_n, tc_ms = kt.get("k_cw_tc", (0, 0.0))
        tc_avg = tc_ms / max(tc_n, 1)
        p_n, p_ms = kt.get(pool_kernel, (0, 0.0))
        pool_bytes = paths * 2 * T * 512 * 4 + (T // mm) * 512 * 4  # unpooled C, Z in; entries out
        achieved = gemm_flop / (tc_avg * 1e-3) / 1e12 if tc_n else 0.0
        res[name] = {
            "ms_per_call": round(ms, 4), "tokens_per_s": round(T / (ms * 1e-3), 1),
            "tflops_per_call": round(paths * gemm_flop / (ms * 1e-3) / 1e12, 1),
            "kernels_ms_per_launch": {k: round(t / max(c, 1), 4) for k, (c, t) in sorted(kt.items())},
            "roofline": {"kernel": "k_cw_tc (bf16 tcgen05 GEMM, unpooled C and Z out)", "bound": "tensor",
                         "achieved": round(achieved, 1), "peak": peak, "peak_kind": kind, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4) if peak else None,
                         "algorithmic_flop_per_launch": gemm_flop, "launch_ms": round(tc_avg, 4)},
            "pool": {"kernel": pool_kernel, "algorithmic_bytes": pool_bytes,
                     "hbm_gbs": round(pool_bytes / (p_ms / max(p_n, 1) * 1e-3) / 1e9, 1) if p_n else None,
                     "hbm_peak": hbm, "hbm_peak_kind": hkind},
        }
    del H, ws, out_o, out_h, Ws
    torch.cuda.empty_cache()
    # HCA dense attention: every compressed entry of a 1M-token context
    B, Nn = V4_B, V4_N
    with torch.cuda.stream(st):
        planes = csa2.Planes.empty(B, Nn, dev)
        WL.fill_planes(planes, V4_SEED, 0, B, Nn, stream=st)
        q, _ = WL.attn_query_dev(V4_SEED, 0, B, dev)
        swa = WL.swa_dev(V4_SEED, 0, B, NSWA, dev, stream=st)
        n_ent = torch.full((B,), Nn, dtype=torch.int32, device=dev)
        out = torch.empty((B, 64, 512), dtype=torch.float32, device=dev)
        lse = torch.empty((B, 64), dtype=torch.float32, device=dev)
        wsa = csa2.workspace(csa2.dense_attn_workspace_size(B, Nn, NSWA), dev)
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(512)

    def dense():
        csa2.dense_attn_decode(planes, B, n_ent, Nn, swa, NSWA, q, scale, out, wsa, lse_out=lse, stream=st)

    ms, kt = timed(dense, max(calls, 20))
    assert csa2.check(wsa, st)[0] == 0
    att_n, att_ms = kt.get("k_attn_part", kt.get("k_attn", (0, 0.0)))
    att_avg = att_ms / max(att_n, 1)
    call_bytes = B * (Nn * MAIN_BYTES + NSWA * SWA_ROW + 64 * 512 * 2)
    call_flop = B * (Nn + NSWA) * 64 * 512 * 2 * 2
    res["hca_dense_attention"] = {
        "ms_per_call": round(ms, 4), "queries_per_s": round(B / (ms * 1e-3), 1),
        "kernels_ms_per_launch": {k: round(t / max(c, 1), 4) for k, (c, t) in sorted(kt.items())},
        "k_attn": {"algorithmic_bytes": call_bytes, "flop": call_flop,
                   "hbm_gbs": round(call_bytes / (att_avg * 1e-3) / 1e9, 1) if att_n else None,
                   "tflops": round(call_flop / (att_avg * 1e-3) / 1e12, 1) if att_n else None,
                   "tensor_frac": round(call_flop / (att_avg * 1e-3) / 1e12 / peak, 4) if att_n else None,
                   "tensor_peak_kind": kind},
    }
    return res


SMALL_STEPS = 20


def run_small_decode(dev, st, wl, steps: int, warmup: int):
    """A sub-L2 decode workload (one FLAT index call + wl.n_attn attention calls sharing its
    top-k, each with its own q and window): per-step device time with L2 flushed before
    every timed step (a write of twice the L2 size) and unflushed (back to back), the HBM
    roofline of the algorithmic bytes, and the oracle timed on the same queries' work."""
    import numpy as np
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    import oracle
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL
    from synth import workloads as W

    Bq, Nq, k, n_attn = wl.B, wl.N, wl.k, wl.n_attn
    with torch.cuda.stream(st):
        planes = csa2.Planes.empty(Bq, Nq, dev)
        WL.fill_planes(planes, wl.seed, 0, Bq, Nq, stream=st)
        qd, wd, q_h, w_h = WL.index_query_dev(wl.seed, 0, Bq, dev)
        qa = [WL.attn_query_dev(wl.seed, l, Bq, dev) for l in range(n_attn)]
        swa = [WL.swa_dev(wl.seed, l, Bq, NSWA, dev, stream=st) for l in range(n_attn)]
        ne = torch.full((Bq,), Nq, dtype=torch.int32, device=dev)
        topk = torch.empty((Bq, k), dtype=torch.int32, device=dev)
        outs = [torch.empty((Bq, 64, 512), dtype=torch.float32, device=dev) for _ in range(n_attn)]
        ws_i = csa2.workspace(csa2.index_topk_workspace_size(Bq, Nq, k, BLOCK, 0), dev)
        ws_a = csa2.workspace(csa2.sparse_attn_workspace_size(Bq, k, NSWA), dev)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(512)

    def step():
        csa2.index_topk(planes, Bq, ne, Nq, qd, wd, k, csa2.TOPK_FLAT, topk, ws_i, stream=st)
        for l in range(n_attn):
            csa2.sparse_attn_decode(planes, Bq, topk, k, swa[l], NSWA, qa[l][0], scale, outs[l], ws_a, stream=st)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert csa2.check(ws_i, st)[0] == 0 and csa2.check(ws_a, st)[0] == 0
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(st):
        for a, b in ev:
            flush_buf.fill_(1)  # evicts the cache and the previous step's data from L2
            a.record(st)
            step()
            b.record(st)
    torch.cuda.synchronize()
    flushed = sorted(a.elapsed_time(b) for a, b in ev)
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(st)
    for _ in range(steps):
        step()
    b0.record(st)
    torch.cuda.synchronize()
    warm_ms = a0.elapsed_time(b0) / steps
    assert csa2.check(ws_i, st)[0] == 0 and csa2.check(ws_a, st)[0] == 0
    csa2.timing_enable(True)
    step()
    torch.cuda.synchronize()
    kt = csa2.kernel_times()
    csa2.timing_enable(False)
    med = statistics.median(flushed)
    step_bytes = Bq * (Nq * IDX_BYTES + n_attn * (k * MAIN_BYTES + NSWA * SWA_ROW))
    hbm, kind = peaks()
    achieved = step_bytes / (med * 1e-3) / 1e9

    # the oracle on the same work: query 0's scores, top-k and attention passes
    kvc, kvs = oracle.quantize_main(W.main_latents(wl.seed, 0, Bq, Nq, 0, 0, Nq))
    ixc, ixs = oracle.quantize_index(W.index_latents(wl.seed, 0, Bq, Nq, 0, 0, Nq))
    swa_h = [W.swa_rows(wl.seed, l, Bq)[0] for l in range(n_attn)]
    threads = os.cpu_count() or 1

    def oracle_query():
        sc = oracle.index_scores(ixc, ixs, q_h[0], w_h[0], nthreads=threads)
        sel = oracle.topk(sc, k)
        for l in range(n_attn):
            oracle.attention(kvc, kvs, sel, swa_h[l], qa[l][1][0], scale)

    oracle_query()  # warm
    reps, t0 = 0, time.perf_counter()
    while reps < 3 or (time.perf_counter() - t0 < 2.0 and reps < 200):
        oracle_query()
        reps += 1
    o_s = (time.perf_counter() - t0) / reps  # seconds per query
    return {
        "workload": wl.name, "B": Bq, "N_entries": Nq, "k": k, "n_swa": NSWA, "attention_passes": n_attn,
        "steps": steps, "warmup": warmup,
        "us_per_step_l2_flushed": round(med * 1e3, 2), "us_per_step_l2_flushed_mean": round(
            statistics.mean(flushed) * 1e3, 2),
        "us_per_step_unflushed": round(warm_ms * 1e3, 2),
        "queries_per_s_l2_flushed": round(Bq / (med * 1e-3), 1),
        "l2": f"flushed before each timed step by writing {2 * l2} B (2 x L2); unflushed = back to back",
        "kernels_ms_per_launch": {kk: round(t / max(n, 1), 4) for kk, (n, t) in sorted(kt.items())},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "peak_kind": kind, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": None, "algorithmic_bytes_per_step": step_bytes,
                     "of": "the whole step (all its kernels), L2 flushed"},
        "cpu_baseline": {"value": round(1.0 / o_s, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
                         "us_per_query": round(o_s * 1e6, 1),
                         "sample": f"query 0 of the workload, {reps} passes: fp64 scores over its {Nq} entries, "
                                   f"top-{k}, {n_attn} attention pass(es)"},
    }


def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p))["bf16_tflops"]), "measured bf16 (burst)"
    return 1900.0, "fallback bf16 (burst)"


def replica_seed(base: int, rank: int) -> int:
    """Seed of rank `rank`'s replica: rank 0 keeps the workload's seed, the others get
    distinct synthetic problems of the same shape (weak scaling: one batch per GPU)."""
    return base + 1000 * rank


def max_over_ranks(times, world: int, device="cpu"):
    """Each timing replaced by its maximum over the ranks: the slowest replica sets the
    job's pace.  Collective over the default process group when world > 1."""
    if world <= 1:
        return [float(t) for t in times]
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x) for x in times], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(world: int, per_rank_units: int, steps: int, ms: float) -> float:
    """Whole-job units per second: every rank processed per_rank_units per step."""
    return world * per_rank_units * steps / (ms * 1e-3)


def line_config(world: int) -> dict:
    """The workload's config object, the same in both arms' lines."""
    return {"workload": WORKLOAD, "B": B, "N_entries": N, "k": K_TOP, "block": BLOCK,
            "n_blocks_keep": KEEP, "n_swa": NSWA, "seed": SEED if world == 1 else f"{SEED} + 1000 x rank",
            "l2": "inputs larger than L2 (11.95 GB cache resident in HBM); no flush",
            "parallelism": f"replicas x{world}"}


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    import compressed_sparse_attention_nvfp4_gb300 as csa2
    from compressed_sparse_attention_nvfp4_gb300 import workload as WL
    from synth import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    csa2.lib()
    st = torch.cuda.Stream(device=dev)
    seed = replica_seed(SEED, rank)
    with torch.cuda.stream(st):
        planes = csa2.Planes.empty(B, N, dev)
        qd, wd, q_h, w_h = WL.index_query_dev(seed, 0, B, dev)
        hv = W.hot_vectors(q_h, w_h, 3.0)
        WL.fill_planes(planes, seed, 0, B, N, hot_prob=0.02, hotvecs=hv, stream=st)
        qa_d, qa_h = WL.attn_query_dev(seed, 0, B, dev)
        swa_d = WL.swa_dev(seed, 0, B, NSWA, dev, stream=st)
        ne = torch.full((B,), N, dtype=torch.int32, device=dev)
        topk = torch.empty((B, K_TOP), dtype=torch.int32, device=dev)
        pool = torch.empty((B, KEEP), dtype=torch.int32, device=dev)
        out = torch.empty((B, 64, 512), dtype=torch.float32, device=dev)
        lse = torch.empty((B, 64), dtype=torch.float32, device=dev)
        ws_i = csa2.workspace(csa2.index_topk_workspace_size(B, N, K_TOP, BLOCK, KEEP), dev)
        ws_a = csa2.workspace(csa2.sparse_attn_workspace_size(B, K_TOP, NSWA), dev)
        # a second batch's buffers: two independent batches in flight on two streams, as a
        # server keeps two micro-batches of decode requests in flight
        st2 = torch.cuda.Stream(device=dev)
        bufs = [dict(topk=topk, pool=pool, out=out, lse=lse, ws_i=ws_i, ws_a=ws_a, st=st),
                dict(topk=torch.empty_like(topk), pool=torch.empty_like(pool), out=torch.empty_like(out),
                     lse=torch.empty_like(lse), ws_i=csa2.workspace(ws_i.numel(), dev),
                     ws_a=csa2.workspace(ws_a.numel(), dev), st=st2)]
    torch.cuda.synchronize()
    scale = 1.0 / math.sqrt(512)

    def index_call(bf=None):
        bf = bf or bufs[0]
        csa2.index_topk(planes, B, ne, N, qd, wd, K_TOP, csa2.TOPK_HIER_BUILD, bf["topk"], bf["ws_i"], BLOCK,
                        KEEP, pool_out=bf["pool"], stream=bf["st"])

    def attn_call(bf=None):
        bf = bf or bufs[0]
        csa2.sparse_attn_decode(planes, B, bf["topk"], K_TOP, swa_d, NSWA, qa_d, scale, bf["out"], bf["ws_a"],
                                lse_out=bf["lse"], stream=bf["st"])

    for _ in range(args.warmup):
        for bf in bufs:
            index_call(bf)
            attn_call(bf)
    torch.cuda.synchronize()
    for bf in bufs:
        assert csa2.check(bf["ws_i"], bf["st"])[0] == 0 and csa2.check(bf["ws_a"], bf["st"])[0] == 0

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # timed region: K steps bracketed by one pair of events (nothing else recorded
    # between the kernels, so their launches overlap as in production).  Step s runs
    # batch s % 2 on stream s % 2: two independent batches in flight, so one batch's
    # latency-bound selects and attention overlap the other's HBM-bound scan
    def timed(k, in_flight):
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        st2.wait_event(a)
        for s in range(k):
            bf = bufs[s % in_flight]
            index_call(bf)
            attn_call(bf)
        j = torch.cuda.Event()
        j.record(st2)
        st.wait_event(j)
        z.record(st)
        return a, z

    with clock_sampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        clk.mark()
        start, stop = timed(args.steps, 2)
        torch.cuda.synchronize()
        clk.stop()
        barrier()
    elapsed_ms = start.elapsed_time(stop)
    clocks = clk.summary()
    # the same K steps with one batch in flight (each step waits for the one before)
    a1, z1 = timed(args.steps, 1)
    torch.cuda.synchronize()
    serial_ms = a1.elapsed_time(z1)

    # instrumented pass over the same K steps: events around each call, and the
    # library's per-kernel events (each adds a few microseconds at a kernel
    # boundary, which is why the headline value above comes from a clean pass)
    n_instr = min(args.steps, 50)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_instr)]
    csa2.timing_enable(True)
    torch.cuda.synchronize()
    for s in range(n_instr):
        ev[s][0].record(st)
        index_call()
        ev[s][1].record(st)
        attn_call()
        ev[s][2].record(st)
    torch.cuda.synchronize()
    idx_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    att_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    ktimes = csa2.kernel_times()
    csa2.timing_enable(False)

    # end to end through the same C-ABI calls with host buffers: per step the
    # query-side inputs go up from pinned memory and the output comes back.  Three
    # device input / output sets, an upload and a download stream, and step s
    # computing on stream s % 2 as in the timed region: the next steps' inputs travel
    # while step s computes, and step s's output comes back during the following ones.
    h_q = torch.from_numpy(q_h.view(np.int16)).pin_memory()
    h_w = torch.from_numpy(w_h).pin_memory()
    h_qa = torch.from_numpy(qa_h.view(np.int16)).pin_memory()
    h_swa = swa_d.cpu().pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_w, h_qa, h_swa))
    d2h = out.numel() * 4 + lse.numel() * 4
    up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    sets = []
    n_sets = 3  # three input / output sets: each step's copies have two steps' time to finish
    for i in range(n_sets):
        sets.append({"q": torch.empty_like(qd), "w": torch.empty_like(wd), "qa": torch.empty_like(qa_d),
                     "swa": torch.empty_like(swa_d), "out": torch.empty_like(out), "lse": torch.empty_like(lse),
                     "h_out": torch.empty(out.shape, dtype=torch.float32).pin_memory(),
                     "h_lse": torch.empty(lse.shape, dtype=torch.float32).pin_memory(),
                     "up": torch.cuda.Event(), "done": torch.cuda.Event(), "down": torch.cuda.Event()})
    e_start, e_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e_start.record(st)
    up_s.wait_event(e_start)
    st2.wait_event(e_start)
    for s_i in range(args.steps):
        S = sets[s_i % n_sets]
        with torch.cuda.stream(up_s):
            if s_i >= n_sets:
                up_s.wait_event(S["done"])  # the set's previous step no longer reads its inputs
            S["q"].copy_(h_q, non_blocking=True)
            S["w"].copy_(h_w, non_blocking=True)
            S["qa"].copy_(h_qa, non_blocking=True)
            S["swa"].copy_(h_swa, non_blocking=True)
            S["up"].record(up_s)
        bf = bufs[s_i % 2]  # step s computes on stream s % 2 (two batches in flight)
        cs = bf["st"]
        cs.wait_event(S["up"])
        if s_i >= n_sets:
            cs.wait_event(S["down"])  # the set's previous output has been read back
        csa2.index_topk(planes, B, ne, N, S["q"], S["w"], K_TOP, csa2.TOPK_HIER_BUILD, bf["topk"], bf["ws_i"],
                        BLOCK, KEEP, pool_out=bf["pool"], stream=cs)
        csa2.sparse_attn_decode(planes, B, bf["topk"], K_TOP, S["swa"], NSWA, S["qa"], scale, S["out"], bf["ws_a"],
                                lse_out=S["lse"], stream=cs)
        S["done"].record(cs)
        with torch.cuda.stream(down_s):
            down_s.wait_event(S["done"])
            S["h_out"].copy_(S["out"], non_blocking=True)
            S["h_lse"].copy_(S["lse"], non_blocking=True)
            S["down"].record(down_s)
    st.wait_stream(down_s)
    e_stop.record(st)
    torch.cuda.synchronize()
    e2e_ms = e_start.elapsed_time(e_stop)
    for bf in bufs:
        assert csa2.check(bf["ws_i"], bf["st"])[0] == 0 and csa2.check(bf["ws_a"], bf["st"])[0] == 0
    last = sets[(args.steps - 1) % n_sets]
    e2e_same = bool(torch.equal(last["h_out"], out.cpu()) and torch.equal(last["h_lse"], lse.cpu()))

    elapsed_ms, e2e_ms, serial_ms = max_over_ranks([elapsed_ms, e2e_ms, serial_ms], world, dev)
    if rank != 0:
        return None
    hbm, peak_kind = peaks()
    idx_bytes = B * N * IDX_BYTES  # the scan reads every entry's 68-byte indexer key once
    scan_launches, scan_ms = ktimes.get("k_scan_tc", (0, 0.0))
    scan_avg_ms = scan_ms / max(scan_launches, 1)
    achieved = idx_bytes / (scan_avg_ms * 1e-3) / 1e9 if scan_launches else 0.0
    idx_achieved = idx_bytes / (idx_ms * 1e-3) / 1e9
    fp = kernel_fingerprint()
    traffic = recorded_traffic(fp)
    # kernel launches of the K timed steps: the library's count per instrumented step x K
    launches = round(sum(n for n, _ in ktimes.values()) * args.steps / n_instr)
    value = job_rate(world, B, args.steps, elapsed_ms)
    step_bytes = B * (N * IDX_BYTES + K_TOP * MAIN_BYTES + NSWA * SWA_ROW)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": args.dtype_label, "data": "synthetic (seeded counter-based generator)",
        "config": line_config(world),
        "step_breakdown_ms": {"index_topk": round(idx_ms, 4), "sparse_attn": round(att_ms, 4)},
        "kernels_ms_per_launch": {k: round(t / max(n, 1), 4) for k, (n, t) in sorted(ktimes.items())},
        "step_hbm": {"algorithmic_bytes": step_bytes,
                     "achieved_gbs": round(step_bytes / (elapsed_ms / args.steps * 1e-3) / 1e9, 1)},
        "roofline": {"kernel": "k_scan_tc (indexer scan, block-scaled FP4 MMA)", "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": hbm, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / hbm, 4),
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "algorithmic_bytes_per_launch": idx_bytes,
                     "launch_ms": round(scan_avg_ms, 4), "sources": fp,
                     "index_call": {"achieved": round(idx_achieved, 1),
                                    "frac": round(idx_achieved / hbm, 4)}},
        "e2e": {"value": round(job_rate(world, B, args.steps, e2e_ms), 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": "overlapped with compute (three input/output sets, upload and download streams; "
                          "step s computes on stream s % 2, two batches in flight)",
                "result_equals_device_run": e2e_same},
        "gpu_launches": launches,
        "clocks": clocks,
        "in_flight": {"batches": 2, "how": "step s runs batch s % 2 on stream s % 2 (independent batches, "
                                           "separate outputs and workspaces)",
                      "one_batch_ms_per_step": round(serial_ms / args.steps, 4),
                      "one_batch_value": round(job_rate(world, B, args.steps, serial_ms), 2)},
    }
    if not args.no_small:
        from synth import workloads as W

        line["config0_single_4k"] = run_small_decode(dev, st, W.SINGLE_4K, SMALL_STEPS, 5)
        line["config1_encoder_b64"] = run_small_decode(dev, st, W.ENCODER_B64, SMALL_STEPS, 5)
    if not args.no_attn:
        line["attention_b128"] = run_attention(dev, st, 50, 3)
    if not args.no_cache_write:
        line["cache_write"] = run_cache_write(dev, st, 5, 2)
        line["decode_append"] = run_append(dev, st, 20, 3)
        line["prefill_indexer"] = run_prefill_index(dev, st, 5, 2)
        line["v4_variants"] = run_v4(dev, st, 5, 2)
    if not args.no_step40:
        del planes, ws_i, ws_a, bufs, sets
        torch.cuda.empty_cache()
        line["step_40_layers"] = run_step40(dev, st, 10, 3)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-cache-write", action="store_true",
                    help="skip the prefill cache-write measurement (its own object in the line)")
    ap.add_argument("--no-step40", action="store_true",
                    help="skip the 40-layer step measurement (its own object in the line)")
    ap.add_argument("--no-small", action="store_true",
                    help="skip the single-query 4K and batch-64 encoder workloads (their own objects)")
    ap.add_argument("--small-only", action="store_true",
                    help="profiling case: only the single-query 4K and batch-64 encoder workloads")
    ap.add_argument("--no-attn", action="store_true",
                    help="skip the batch-128 attention measurement (its own object in the line)")
    ap.add_argument("--attn-only", action="store_true",
                    help="profiling case: only the batch-128 attention, printed as its own line")
    ap.add_argument("--prefill-index-only", action="store_true",
                    help="profiling case: only the prefill indexer")
    ap.add_argument("--append-only", action="store_true",
                    help="profiling case: only the decode-time cache append and window write")
    ap.add_argument("--v4-only", action="store_true",
                    help="profiling case: only the V4 compressors and the HCA dense attention")
    ap.add_argument("--step40-only", action="store_true",
                    help="profiling case: only the 40-layer step, printed as its own line")
    ap.add_argument("--cache-write-only", action="store_true",
                    help="profiling case: only the prefill cache write, printed as its own line")
    ap.add_argument("--batch", type=int, default=32,
                    help="queries per step; values other than 32 are for small profiling cases, "
                         "not for the reported metric")
    args = ap.parse_args()
    global B
    B = args.batch
    args.warmup = max(args.warmup, 3)
    # tensor-core operands: E2M1 keys x E4M3 query halves (indexer), f16 (attention); fp32 accumulate
    args.dtype_label = "e2m1xe4m3/f16 mma, f32 acc"

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        v, cores, desc, f = oracle_reference_steps(args.steps, args.warmup)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter-based generator)",
            "config": line_config(world),
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc, "steps_per_query": f, "cpu_model": host_cpu()},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}))
        return

    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.attn_only:
        import torch

        torch.cuda.set_device(local_rank)
        import compressed_sparse_attention_nvfp4_gb300 as csa2

        csa2.lib()
        dev = torch.device("cuda", local_rank)
        st = torch.cuda.Stream(device=dev)
        if rank == 0:
            print(json.dumps({"attention_b128": run_attention(dev, st, max(1, min(args.steps, 200)),
                                                              max(1, args.warmup))}), flush=True)
        return
    if args.small_only:
        import torch

        torch.cuda.set_device(local_rank)
        import compressed_sparse_attention_nvfp4_gb300 as csa2
        from synth import workloads as W

        csa2.lib()
        dev = torch.device("cuda", local_rank)
        st = torch.cuda.Stream(device=dev)
        if rank == 0:
            n = max(1, min(args.steps, SMALL_STEPS))
            print(json.dumps({"config0_single_4k": run_small_decode(dev, st, W.SINGLE_4K, n, args.warmup),
                              "config1_encoder_b64": run_small_decode(dev, st, W.ENCODER_B64, n, args.warmup)}),
                  flush=True)
        return
    if args.step40_only:
        import torch

        torch.cuda.set_device(local_rank)
        import compressed_sparse_attention_nvfp4_gb300 as csa2

        csa2.lib()
        dev = torch.device("cuda", local_rank)
        st = torch.cuda.Stream(device=dev)
        if rank == 0:
            print(json.dumps({"step_40_layers": run_step40(dev, st, max(1, min(args.steps, 20)),
                                                           max(1, args.warmup))}), flush=True)
        return
    if args.prefill_index_only:
        import torch

        torch.cuda.set_device(local_rank)
        import compressed_sparse_attention_nvfp4_gb300 as csa2

        csa2.lib()
        dev = torch.device("cuda", local_rank)
        st = torch.cuda.Stream(device=dev)
        if rank == 0:
            print(json.dumps({"prefill_indexer": run_prefill_index(dev, st, max(1, min(args.steps, 20)),
                                                                   max(1, args.warmup))}), flush=True)
        return
    if args.append_only:
        import torch

        torch.cuda.set_device(local_rank)
        import compressed_sparse_attention_nvfp4_gb300 as csa2

        csa2.lib()
        dev = torch.device("cuda", local_rank)
        st = torch.cuda.Stream(device=dev)
        if rank == 0:
            print(json.dumps({"decode_append": run_append(dev, st, max(1, min(args.steps, 50)),
                                                          max(1, args.warmup))}), flush=True)
        return
    if args.v4_only:
        import torch

        torch.cuda.set_device(local_rank)
        import compressed_sparse_attention_nvfp4_gb300 as csa2

        csa2.lib()
        dev = torch.device("cuda", local_rank)
        st = torch.cuda.Stream(device=dev)
        if rank == 0:
            print(json.dumps({"v4_variants": run_v4(dev, st, max(1, min(args.steps, 20)), max(1, args.warmup))}),
                  flush=True)
        return
    if args.cache_write_only:
        import torch

        torch.cuda.set_device(local_rank)
        import compressed_sparse_attention_nvfp4_gb300 as csa2

        csa2.lib()
        dev = torch.device("cuda", local_rank)
        st = torch.cuda.Stream(device=dev)
        if rank == 0:
            print(json.dumps({"cache_write": run_cache_write(dev, st, max(1, min(args.steps, 20)),
                                                             max(1, args.warmup))}), flush=True)
        return
    line = run_ours(args, rank, world, local_rank)
    if line is not None:
        if world == 1 and not args.no_cpu_baseline:
            v, cores, desc = oracle_sample(2, 1)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": UNIT, "cores": cores,
                                    "kind": "oracle", "sample": desc, "cpu_model": host_cpu()}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
