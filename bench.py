"""Benchmark: MLA ragged prefill TFLOP/s on GB300 (one JSON line on stdout).

Default workload: 8 ragged causal requests, lengths uniform in [512, 4096]
(seeded), 128 heads, Q/K dim 192, V dim 128, bf16 -- the DeepSeek-R1-shaped
prefill the metric is quoted on.  A step is one pass of the hot path over
that batch: the work list comes from the plan (made once per batch, reused
by every layer) and the step is one ``mla_prefill_run``.  The chunked-prefix
path (gather -> up-projection -> non-causal chunk attention -> merge) is
timed on the 4 x (2048 new + 8192 cached) workload and reported under
``chunked_prefix``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload (there is no runnable reference implementation).
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
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from chunked_prefill_attention_ragged_gb300 import workloads as wl  # noqa: E402

METRIC = "MLA ragged prefill TFLOP/s (Dqk192/Dv128, bf16) and % of GB300 BF16 TC peak"
FLOP_PER_PAIR = 2 * (wl.DQK + wl.DV)      # QK^T (2*192) + PV (2*128) per allowed (query, key) pair and head
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0
L2_NOTE = "no flush: inputs (2.73 GB) far larger than the 129 MB L2"


# ----------------------------------------------------------------------------- accounting
def allowed_pairs(q_lens, kv_lens, causal: bool) -> int:
    """Allowed (query, key) pairs of one head, counted exactly (bottom-right causal)."""
    total = 0
    for lq, lkv in zip(q_lens, kv_lens):
        lq, lkv = int(lq), int(lkv)
        if not causal:
            total += lq * lkv
            continue
        d = lkv - lq
        # row i sees keys 0..i+d clipped to [0, lkv)
        for_rows = np.clip(np.arange(lq) + d + 1, 0, lkv)
        total += int(for_rows.sum())
    return total


def attention_flops(q_lens, kv_lens, heads: int, causal: bool) -> float:
    return float(allowed_pairs(q_lens, kv_lens, causal)) * heads * FLOP_PER_PAIR


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    out = {"bf16_tflops": FALLBACK_BF16_TFLOPS, "bf16_tflops_sustained": None, "hbm_gbs": FALLBACK_HBM_GBS,
           "source": "fallback"}
    if os.path.exists(path):
        try:
            d = json.load(open(path))

            def find(keys):
                for k in keys:
                    if k in d and isinstance(d[k], (int, float)):
                        return float(d[k])
                return None
            bf = find(["bf16_tflops", "bf16_tflops_burst"])
            bs = find(["bf16_tflops_sustained"])
            hb = find(["hbm_gbs", "hbm_GBs", "hbm_gb_s"])
            if bf:
                out["bf16_tflops"] = bf
                out["source"] = "measured"
            if bs:
                out["bf16_tflops_sustained"] = bs
            if hb:
                out["hbm_gbs"] = hb
        except Exception:
            pass
    return out


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("attn_kernel.cu", "ptx.cuh", "tmem_wide.cuh", "planner.cpp", "planner.h"):
        with open(os.path.join(ROOT, "chunked_prefill_attention_ragged_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, if it
    was taken on the current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "prefill_attention_traffic.json")
    try:
        d = json.load(open(path))
        if d.get("kernel_source_hash") == kernel_source_hash():
            return d.get("dram_bytes_per_launch_full_workload")
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.25)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=2)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, p in zip(names, parts[2:6]):
                if p.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


class NvmlClockSampler:
    """SM clock and clock-event reasons polled through NVML every ~1 ms from a thread, so
    that even a timed region of a few tens of milliseconds gets many samples.  The GPU is
    found by its PCI bus id (CUDA and NVML number devices differently).  Only reads."""
    # nvmlClocksEventReason* bits (nvml.h)
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        self.ok = False
        self.samples = []
        self._stop = threading.Event()
        try:
            import torch
            prop = torch.cuda.get_device_properties(device_index)
            bus = "%08x:%02x:%02x.0" % (prop.pci_domain_id, prop.pci_bus_id, prop.pci_device_id)
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                return
            mx = ctypes.c_uint(0)
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:   # 1 = NVML_CLOCK_SM
                return
            try:
                self.reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                self.reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons
            self.lib, self.h, self.max_mhz, self.bus = lib, h, mx.value, bus
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        import ctypes
        clk, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while not self._stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0 and \
                    self.reasons_fn(self.h, ctypes.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(0.001)

    def __enter__(self):
        if self.ok:
            self.thread = threading.Thread(target=self._run, daemon=True)
            self.thread.start()
            time.sleep(0.01)
        return self

    def __exit__(self, *a):
        if self.ok:
            time.sleep(0.005)
            self._stop.set()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return None
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(c for c, _ in self.samples), "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "NVML, polled every ~1 ms during the timed region",
                "pci_bus_id": self.bus}


# ----------------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int, device) -> float:
    """The maximum of x over all ranks (x itself when there is one rank).  Each rank runs
    its own batch (weak scaling), so the job's time is the slowest rank's."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tflops(flops_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's FLOPs over the slowest rank's step time."""
    return flops_per_rank * world / (ms_per_step * 1e-3) / 1e12


# ----------------------------------------------------------------------------- CPU oracle timing
def _oracle_job(args):
    """One (request, head) of the oracle; run in a spawned single-threaded worker."""
    q, k, v, sm_scale = args
    from oracle import attend_request
    t0 = time.perf_counter()
    attend_request(q, k, v, causal=True, sm_scale=sm_scale)
    return time.perf_counter() - t0


def time_oracle_sample(batch: wl.RaggedBatch, target_s: float = 15.0, max_workers: int | None = None):
    """Time the fp64 oracle on (request, head) pieces of the workload until about
    target_s of wall time is spent; returns (TFLOP/s, cores, sample description)."""
    import multiprocessing as mp
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"        # inherited by spawned workers: one BLAS thread each
    workers = max_workers or os.cpu_count() or 1
    qo, kv = batch.qo_indptr, batch.kv_indptr
    # (request, head) pieces in a fixed order: requests shortest first, all heads of each.
    jobs, meta = [], []
    for r in np.argsort(batch.q_lens, kind="stable"):
        r = int(r)
        for h in range(batch.num_heads):
            jobs.append((batch.q[qo[r]:qo[r + 1], h:h + 1], batch.k[kv[r]:kv[r + 1], h:h + 1],
                         batch.v[kv[r]:kv[r + 1], h:h + 1], batch.sm_scale))
            meta.append(r)
    ctx = mp.get_context("spawn")
    done = 0
    with ctx.Pool(workers) as pool:
        pool.map(_oracle_job, jobs[:workers])          # start-up and first-touch outside the clock
        t0 = time.perf_counter()
        for start in range(0, len(jobs), workers):
            pool.map(_oracle_job, jobs[start:start + workers])
            done = min(len(jobs), start + workers)
            if time.perf_counter() - t0 > target_s:
                break
        wall = time.perf_counter() - t0
    flops = sum(attention_flops([batch.q_lens[r]], [batch.kv_lens[r]], 1, True) for r in meta[:done])
    reqs = sorted(set(meta[:done]))
    return flops / wall / 1e12, workers, (f"{done} (request, head) pieces of {len(jobs)} (requests {reqs}, "
                                          f"shortest first), {workers} spawned single-thread fp64 numpy "
                                          f"workers, {wall:.1f} s")


def workload_config(b: wl.RaggedBatch, index: int, world: int, l2_note: str) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    return {
        "workload": wl.WORKLOAD_NAMES[index],
        "requests": int(b.batch),
        "q_lens": [int(x) for x in b.q_lens],
        "heads": b.num_heads, "head_dim_qk": 192, "head_dim_vo": 128, "causal": b.causal,
        "sm_scale": b.sm_scale, "window_left": b.window_left, "logits_soft_cap": b.logits_soft_cap,
        "flop_per_step": attention_flops(b.q_lens, b.kv_lens, b.num_heads, b.causal),
        "allowed_pairs_per_head": allowed_pairs(b.q_lens, b.kv_lens, b.causal),
        "l2": l2_note,
        "parallelism": f"replicas x{world} (each rank runs its own batch)",
    }


def bench_workload_row(index: int, cap: float, dev, peaks, launches: int):
    """Device time of mla_prefill_run on another workload (its own JSON row): median of
    `launches` launches after 3 warm-ups, each launch after a 256 MB L2 flush when the
    inputs fit in L2."""
    import torch
    import chunked_prefill_attention_ragged_gb300 as mla
    b = wl.make_workload(index, logits_soft_cap=cap)

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = dev_bf16(b.q), dev_bf16(b.k), dev_bf16(b.v)
    plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale,
                                window_left=b.window_left, logits_soft_cap=b.logits_soft_cap)
    o = torch.empty((b.q.shape[0], b.num_heads, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((b.q.shape[0], b.num_heads), dtype=torch.float32, device=dev)
    in_bytes = (q.numel() + k.numel() + v.numel()) * 2
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if in_bytes < (256 << 20) else None
    stream = torch.cuda.current_stream(dev)
    for _ in range(3):
        plan.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    plan.status()
    times = []
    for _ in range(launches):
        if flush is not None:
            flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        plan.run(q, k, v, o, lse)
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    plan.status()
    ms = statistics.median(times)
    flops = attention_flops(b.q_lens, b.kv_lens, b.num_heads, b.causal)
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": b.name, "heads": b.num_heads, "requests": int(b.batch), "logits_soft_cap": cap,
            "ms": round(ms, 4), "launches": launches, "flop": flops, "tflops": round(tf, 2),
            "roofline": {"kernel": "prefill_kernel", "bound": "tensor", "achieved": round(tf, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tf / peaks["bf16_tflops"], 4)},
            "plan_units": plan.num_units,
            "l2": "256 MB written before each launch" if flush is not None else "inputs larger than L2, no flush"}


# ----------------------------------------------------------------------------- our arm
def bench_ours(args, world, rank, local):
    import torch
    import chunked_prefill_attention_ragged_gb300 as mla

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks = load_peaks()
    b = wl.make_workload(args.workload)
    flops = attention_flops(b.q_lens, b.kv_lens, b.num_heads, b.causal)

    # CPU baseline first (spawned pool, before the GPU is busy), rank 0 at N=1 only.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = time_oracle_sample(b, target_s=args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = dev_bf16(b.q), dev_bf16(b.k), dev_bf16(b.v)
    stream = torch.cuda.current_stream(dev)
    # Host cost of planning (the plan call: work list, schedule, workspace upload enqueued),
    # paid once per batch and shared by every layer's run.
    plan_ms = []
    for _ in range(5):
        t0 = time.perf_counter()
        plan = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale,
                                    window_left=b.window_left, logits_soft_cap=b.logits_soft_cap)
        plan_ms.append((time.perf_counter() - t0) * 1e3)
    o = torch.empty((b.q.shape[0], b.num_heads, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((b.q.shape[0], b.num_heads), dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        plan.run(q, k, v, o, lse)
    torch.cuda.synchronize()
    plan.status()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- device-timed region: K steps, inputs resident (2.4 GB >> 129 MB L2)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    nv = NvmlClockSampler(local)
    with (nv if nv.ok else ClockSampler(local)) as clk:
        barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            plan.run(q, k, v, o, lse)
            ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    plan.status()
    total_ms = reduce_max(t_start.elapsed_time(t_end), world, dev)
    launch_ms = [a.elapsed_time(c) for a, c in ev]
    ms_per_step = total_ms / args.steps
    value = aggregate_tflops(flops, world, ms_per_step)

    # ---- end to end through the public API with host buffers
    # Every step copies its own Q/K/V from pinned host memory, plans, runs and reads O and
    # LSE back.  Steps are pipelined the way a server streams batches: two device buffer
    # sets, uploads on one stream, plan + kernel on another, downloads on a third, so step
    # i+1's upload overlaps step i's kernel and download.  The plan uploads its work list
    # from an idle stream of its own (a copy from pageable memory first waits for its
    # stream to drain).
    pin = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).pin_memory()  # noqa: E731
    hq, hk, hv = pin(b.q), pin(b.k), pin(b.v)
    nbuf = 2
    sets = []
    for _ in range(nbuf):
        sets.append({
            "q": torch.empty(hq.shape, dtype=torch.int16, device=dev),
            "k": torch.empty(hk.shape, dtype=torch.int16, device=dev),
            "v": torch.empty(hv.shape, dtype=torch.int16, device=dev),
            "o": torch.empty(o.shape, dtype=torch.bfloat16, device=dev),
            "lse": torch.empty(lse.shape, dtype=torch.float32, device=dev),
            "ho": torch.empty(o.shape, dtype=torch.int16).pin_memory(),
            "hl": torch.empty(lse.shape, dtype=torch.float32).pin_memory(),
            "inp": torch.cuda.Event(), "done": torch.cuda.Event(), "out": torch.cuda.Event(), "used": False,
        })
    s_in, s_cmp, s_out, s_plan = (torch.cuda.Stream(dev) for _ in range(4))

    def e2e_step(i):
        st = sets[i % nbuf]
        if st["used"]:
            s_in.wait_event(st["done"])          # the kernel that read this set's inputs is done
        with torch.cuda.stream(s_in):
            st["q"].copy_(hq, non_blocking=True)
            st["k"].copy_(hk, non_blocking=True)
            st["v"].copy_(hv, non_blocking=True)
            st["inp"].record(s_in)
        p = mla.mla_prefill_plan(b.qo_indptr, b.kv_indptr, b.num_heads, causal=b.causal, sm_scale=b.sm_scale,
                                 window_left=b.window_left, logits_soft_cap=b.logits_soft_cap, stream=s_plan)
        s_cmp.wait_stream(s_plan)
        s_cmp.wait_event(st["inp"])
        if st["used"]:
            s_cmp.wait_event(st["out"])          # this set's previous O/LSE have been read back
        p.run(st["q"].view(torch.bfloat16), st["k"].view(torch.bfloat16), st["v"].view(torch.bfloat16),
              st["o"], st["lse"], stream=s_cmp)
        st["done"].record(s_cmp)
        s_out.wait_event(st["done"])
        with torch.cuda.stream(s_out):
            st["ho"].copy_(st["o"].view(torch.int16), non_blocking=True)
            st["hl"].copy_(st["lse"], non_blocking=True)
            st["out"].record(s_out)
        st["used"] = True
        return p
    keep = [e2e_step(i) for i in range(2)]
    torch.cuda.synchronize()
    e_steps = max(1, min(args.steps, 10))
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(e_steps):
        keep.append(e2e_step(i))
    torch.cuda.synchronize()
    barrier()
    e2e_s = reduce_max((time.perf_counter() - t0) / e_steps, world, dev)
    for p in keep:
        if p.status() != 0:
            raise RuntimeError("e2e: device status %d" % p.status())
    del keep
    ho, hl = sets[0]["ho"], sets[0]["hl"]
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
    d2h = ho.numel() * 2 + hl.numel() * 4

    # ---- chunked-prefix path rows (workload 2), rank 0
    chunked = None
    if rank == 0 and not args.no_chunked:
        chunked = bench_chunked(args, dev, peaks)

    # ---- absorbed-weight prefill over the chunked-prefix workload's shape, rank 0
    absorbed = None
    if rank == 0 and not args.no_absorbed:
        absorbed = bench_absorbed(dev, peaks)

    # ---- the other workloads, one row each, rank 0
    rows = None
    if rank == 0 and not args.no_workloads:
        del hq, hk, hv, sets
        torch.cuda.empty_cache()
        rows = [bench_workload_row(0, 0.0, dev, peaks, 20), bench_workload_row(3, 0.0, dev, peaks, 5),
                bench_workload_row(4, 0.0, dev, peaks, 20), bench_workload_row(4, 30.0, dev, peaks, 20)]

    if rank != 0:
        return None
    avg_launch_ms = sum(launch_ms) / len(launch_ms)
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16; no dataset)",
        "config": workload_config(b, args.workload, world, L2_NOTE),
        "pct_of_bf16_peak": round(100.0 * value / world / peaks["bf16_tflops"], 2),
        "roofline": {
            "kernel": "prefill_kernel",
            "bound": "tensor",
            "achieved": round(achieved, 2),
            "peak": peaks["bf16_tflops"],
            "peak_source": f"{peaks['source']} bf16 dense (burst)",
            "unit": "TFLOP/s",
            "frac": round(achieved / peaks["bf16_tflops"], 4),
            "traffic": committed_traffic(),
            "avg_launch_ms": round(avg_launch_ms, 4),
        },
        "e2e": {"value": round(aggregate_tflops(flops, world, e2e_s * 1e3), 3), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_s * 1e3, 3),
                "includes": "every step: pinned H2D of Q/K/V, plan, run, D2H of O/LSE; steps pipelined over 2 device buffer sets (upload, compute and download streams)"},
        "cpu_baseline": cpu,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "plan_units": plan.num_units, "plan_ctas": plan.num_ctas,
        "plan": {"host_ms": round(statistics.median(plan_ms), 3), "units": plan.num_units,
                 "note": "mla_prefill_plan wall time on the host (median of 5), once per batch for all layers"},
    }
    if chunked is not None:
        line["chunked_prefix"] = chunked
    if absorbed is not None:
        line["absorbed_prefill"] = absorbed
    if rows is not None:
        line["workloads"] = rows
    return line


def absorbed_case(small: bool):
    """The absorbed-weight prefill inputs: the chunked-prefix workload's shape (4 requests of
    2048 new rows, each the last of 10240 cache positions, 128 heads, 64-slot blocks), or a
    small case (1 request of 64 rows over 2048 positions) for profiler captures."""
    if small:
        return wl.random_absorbed(1201, [64], [2048], 128, block_size=64, num_blocks=64)
    return wl.random_absorbed(1200, [2048] * 4, [10240] * 4, 128, block_size=64, num_blocks=1024)


def bench_absorbed(dev, peaks, reps: int = 3):
    """mla_absorbed_run on the chunked-prefix shape: every head attends to the 576-wide
    cache rows (prefix and new tokens) through the block table."""
    import torch
    import chunked_prefill_attention_ragged_gb300 as mla
    b = absorbed_case(False)
    plan = mla.mla_absorbed_plan(b.qo_indptr, b.kv_lens, b.num_heads, b.block_size, causal=True, sm_scale=b.sm_scale)

    def to_bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    q, cache, table = to_bf(b.q_abs), to_bf(b.cache), torch.from_numpy(b.block_table).to(dev)
    o, lse = plan.run(q, cache, table)
    plan.run(q, cache, table, o, lse)
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        plan.run(q, cache, table, o, lse)
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    if plan.status() != 0:
        raise RuntimeError("absorbed prefill reported a device problem")
    ms = statistics.median(ts)
    flop = float(plan.allowed_pairs) * b.num_heads * 2 * (576 + 512)
    tf = flop / (ms * 1e-3) / 1e12
    return {"workload": "absorbed_4x2048_over_10240_h128_bs64", "ms": round(ms, 3), "launches": reps,
            "flop": flop, "tflops": round(tf, 1), "plan_units": plan.num_units,
            "roofline": {"kernel": "absorbed_kernel", "bound": "tensor", "achieved": round(tf, 1),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tf / peaks["bf16_tflops"], 4)},
            "note": "FLOPs counted as 2 x (576 + 512) per allowed (query, key) pair and head; each CTA "
                    "computes S for its half of the 512 value columns (S work done twice)",
            "l2": "inputs (2.4 GB of queries) larger than L2, no flush"}


def bench_chunked(args, dev, peaks):
    """Per-row timings of the chunked-prefix pipeline on workload 2 (4 x (2048 + 8192 cached))."""
    import torch
    import chunked_prefill_attention_ragged_gb300 as mla
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill

    cb = wl.make_chunked_prefix()
    b = cb.new

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    q, k, v = dev_bf16(b.q), dev_bf16(b.k), dev_bf16(b.v)
    cache, w = dev_bf16(cb.cache), dev_bf16(cb.w_kvb)
    table = torch.from_numpy(cb.block_table).to(dev)
    pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                          sm_scale=b.sm_scale, device=dev)
    o = torch.empty((b.q.shape[0], b.num_heads, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((b.q.shape[0], b.num_heads), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for _ in range(2):
        pipe.run(q, k, v, cache, table, w, o, lse)
    torch.cuda.synchronize()
    pipe.check_status()
    stream = torch.cuda.current_stream(dev)
    reps = 5
    names = ["main_attention", "up_proj_paged", "chunk_attention", "gather", "up_proj", "chunk_attention_full_k",
             "chunk_attention_unfused", "merge"]
    acc = {n: [] for n in names}
    total, total_gathered = [], []
    nC = pipe.cu.shape[0]
    # The pipeline as it runs: each chunk's K/V decompressed straight from the paged cache,
    # each chunk's attention merged into (o, lse) in its epilogue.
    for _ in range(reps):
        flush.zero_()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 + 3 * nC)]
        evs[0].record(stream)
        pipe.main.run(q, k, v, o, lse)
        evs[1].record(stream)
        marks = []
        i = 2
        for c, plan in enumerate(pipe.chunks):
            t = pipe.chunk_tokens[c]
            kc, vc = pipe.k_c[:t], pipe.v_c[:t]
            pipe.decompress(c, cache, table, w, kc, vc)
            evs[i].record(stream)
            pipe.chunk_attention(c, q, o, lse)
            evs[i + 1].record(stream)
            marks.append((evs[i - 1] if c == 0 else marks[-1][2], evs[i], evs[i + 1]))
            i += 2
        torch.cuda.synchronize()
        acc["main_attention"].append(evs[0].elapsed_time(evs[1]))
        for e1, e2, e3 in marks:
            acc["up_proj_paged"].append(e1.elapsed_time(e2))
            acc["chunk_attention"].append(e2.elapsed_time(e3))
        total.append(evs[0].elapsed_time(marks[-1][2]))
    pipe.check_status()
    # The gathered variant: one gather of every chunk's latent rows, then mla_up_proj per chunk.
    gpipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                           sm_scale=b.sm_scale, device=dev, paged_up_proj=False)
    gpipe.run(q, k, v, cache, table, w, o, lse)
    torch.cuda.synchronize()
    for _ in range(reps):
        flush.zero_()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(3 + 3 * nC)]
        evs[0].record(stream)
        gpipe.main.run(q, k, v, o, lse)
        evs[1].record(stream)
        gpipe.gather_all(cache, table)
        evs[2].record(stream)
        i = 3
        for c, plan in enumerate(gpipe.chunks):
            t = gpipe.chunk_tokens[c]
            kc, vc = gpipe.k_c[:t], gpipe.v_c[:t]
            gpipe.decompress(c, cache, table, w, kc, vc)
            evs[i].record(stream)
            gpipe.chunk_attention(c, q, o, lse)
            evs[i + 1].record(stream)
            i += 2
        torch.cuda.synchronize()
        acc["gather"].append(evs[1].elapsed_time(evs[2]))
        for c in range(nC):
            acc["up_proj"].append(evs[2 + 2 * c].elapsed_time(evs[3 + 2 * c]))
            acc["chunk_attention_full_k"].append(evs[3 + 2 * c].elapsed_time(evs[4 + 2 * c]))
        total_gathered.append(evs[0].elapsed_time(evs[2 + 2 * nC]))
    gpipe.check_status()
    pipe.latent = gpipe.gather_all(cache, table)
    # The same chunk step unfused, for comparison and for the merge kernel's own row: the
    # attention writes its O/LSE, then mla_merge_state merges them into (o, lse).
    o_c = torch.empty_like(o)
    lse_c = torch.empty_like(lse)
    for _ in range(reps):
        for c, plan in enumerate(gpipe.chunks):
            t = gpipe.chunk_tokens[c]
            kc, vc = gpipe.k_c[:t], gpipe.v_c[:t]
            flush.zero_()
            e1, e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            e1.record(stream)
            plan.run(q, kc, vc, o_c, lse_c)
            e2.record(stream)
            mla.mla_merge_state(o, lse, o_c, lse_c, o, lse)
            e3.record(stream)
            torch.cuda.synchronize()
            acc["chunk_attention_unfused"].append(e1.elapsed_time(e2))
            acc["merge"].append(e2.elapsed_time(e3))
    pipe.check_status()
    del o_c, lse_c
    # The gather alone, from a cold and clean L2: 256 MB written, then a second 256 MB
    # buffer read, so no dirty line of earlier kernels is evicted inside the timed launch.
    flush_read = torch.ones(64 << 20, dtype=torch.int32, device=dev)
    iso = []
    pipe.chunk_table(table)
    for _ in range(10):
        flush.zero_()
        flush_read.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mla.mla_gather_latent(cache, pipe.table_all, pipe.cu_all_dev, pipe.starts_all_dev, pipe.total_prefix,
                              pipe.latent[:pipe.total_prefix], pipe.status)
        e1.record(stream)
        torch.cuda.synchronize()
        iso.append(e0.elapsed_time(e1))
    pipe.check_status()
    # The dequantizing gather of an fp8 cache of the same shape (648-byte entries), every
    # chunk in one launch, timed alone like the gather.
    cache8 = torch.from_numpy(wl.random_fp8_cache(np.random.default_rng(1102), cb.cache.shape[0], cb.cache.shape[1],
                                                  scale_exp=(126, 127), code_exp=(4, 8))).to(dev)
    out8 = torch.empty((pipe.total_prefix, 576), dtype=torch.bfloat16, device=dev)
    iso8 = []
    for _ in range(10):
        flush.zero_()
        flush_read.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mla.mla_gather_latent_fp8(cache8, pipe.table_all, pipe.cu_all_dev, pipe.starts_all_dev, pipe.total_prefix,
                                  out8, pipe.status)
        e1.record(stream)
        torch.cuda.synchronize()
        iso8.append(e0.elapsed_time(e1))
    pipe.check_status()
    del cache8, out8
    gather8_bytes = pipe.total_prefix * (648 + 576 * 2)
    # Cache write of the new tokens' compressed rows (slot mapping into blocks the prefix
    # does not use), timed alone like the gather.
    n_new = int(b.q.shape[0])
    free_blocks = np.setdiff1d(np.arange(cb.cache.shape[0]), cb.block_table.ravel())
    bs = cb.cache.shape[1]
    slots_h = np.concatenate([free_blocks[:(n_new + bs - 1) // bs, None] * bs + np.arange(bs)[None, :]]).ravel()
    slots = torch.from_numpy(slots_h[:n_new].astype(np.int64)).to(dev)
    new_latent = torch.randn(n_new, 576, device=dev).to(torch.bfloat16)
    cw = []
    for _ in range(10):
        flush.zero_()
        flush_read.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        mla.mla_cache_write(cache, new_latent, slots, pipe.status)
        e1.record(stream)
        torch.cuda.synchronize()
        cw.append(e0.elapsed_time(e1))
    pipe.check_status()
    cw_bytes = 2 * n_new * 576 * 2
    del flush_read
    med = {n: statistics.median(x) for n, x in acc.items()}
    T = int(pipe.chunk_tokens[0])
    rows = b.q.shape[0]
    gather_bytes = 2 * pipe.total_prefix * 576 * 2     # all chunks: read + write
    merge_bytes = rows * b.num_heads * (3 * 128 * 2 + 3 * 4)
    upf = 2.0 * T * 512 * b.num_heads * 256
    up_bytes = T * 576 * 2 + 512 * b.num_heads * 256 * 2 + T * b.num_heads * (192 + 128) * 2
    main_f = attention_flops(b.q_lens, b.q_lens, b.num_heads, True)
    chunk_f = attention_flops(b.q_lens, np.diff(pipe.cu[0]), b.num_heads, False)
    total_f = main_f + nC * (chunk_f + upf)
    hbm = peaks["hbm_gbs"]
    return {
        "workload": wl.WORKLOAD_NAMES[2],
        "chunks": nC, "chunk_tokens_per_request": cb.chunk_tokens,
        "l2": "256 MB buffer written before each repetition",
        "step_ms": round(statistics.median(total), 4),
        "step_tflops": round(total_f / (statistics.median(total) * 1e-3) / 1e12, 2),
        "main_attention": {"ms": round(med["main_attention"], 4),
                           "tflops": round(main_f / med["main_attention"] / 1e9, 2)},
        "chunk_attention": {"ms": round(med["chunk_attention"], 4),
                            "tflops": round(chunk_f / med["chunk_attention"] / 1e9, 2),
                            "merge": "fused into the attention epilogue",
                            "k": "per-head K_nope + one shared rope row per key (mla_prefill_run_shared_rope)"},
        "chunk_attention_full_k": {"ms": round(med["chunk_attention_full_k"], 4),
                                   "tflops": round(chunk_f / med["chunk_attention_full_k"] / 1e9, 2),
                                   "note": "the gathered variant: K [T, H, 192] with the rope in every head "
                                           "(mla_prefill_run_merge)"},
        "chunk_attention_unfused": {"ms": round(med["chunk_attention_unfused"], 4),
                                    "tflops": round(chunk_f / med["chunk_attention_unfused"] / 1e9, 2),
                                    "plus_merge_ms": round(med["merge"], 4)},
        "up_proj_paged": {"ms": round(med["up_proj_paged"], 4),
                          "tflops": round(upf / med["up_proj_paged"] / 1e9, 2),
                          "note": "gather + up-projection in one kernel writing K_nope, V and one rope row per "
                                  "token (mla_up_proj_paged_split), as the pipeline runs"},
        "up_proj": {"ms": round(med["up_proj"], 4), "tflops": round(upf / med["up_proj"] / 1e9, 2),
                    "gbs": round(up_bytes / med["up_proj"] / 1e6, 1),
                    "note": "mla_up_proj on gathered latent rows (the gathered variant)"},
        "step_ms_gathered_variant": round(statistics.median(total_gathered), 4),
        "gather": {"ms": round(med["gather"], 4), "gbs": round(gather_bytes / med["gather"] / 1e6, 1),
                   "frac_hbm": round(gather_bytes / med["gather"] / 1e6 / hbm, 3)},
        "gather_isolated": {"ms": round(statistics.median(iso), 4),
                            "gbs": round(gather_bytes / statistics.median(iso) / 1e6, 1),
                            "frac_hbm": round(gather_bytes / statistics.median(iso) / 1e6 / hbm, 3),
                            "l2": "256 MB written, then another 256 MB read, before each launch"},
        "gather_fp8_isolated": {"ms": round(statistics.median(iso8), 4),
                                "gbs": round(gather8_bytes / statistics.median(iso8) / 1e6, 1),
                                "frac_hbm": round(gather8_bytes / statistics.median(iso8) / 1e6 / hbm, 3),
                                "bytes": gather8_bytes,
                                "note": "mla_gather_latent_fp8: 648-byte fp8 entries read, 1152-byte bf16 rows "
                                        "written, every chunk in one launch",
                                "l2": "256 MB written, then another 256 MB read, before each launch"},
        "cache_write": {"ms": round(statistics.median(cw), 4), "tokens": n_new,
                        "gbs": round(cw_bytes / statistics.median(cw) / 1e6, 1),
                        "frac_hbm": round(cw_bytes / statistics.median(cw) / 1e6 / hbm, 3),
                        "l2": "256 MB written, then another 256 MB read, before each launch"},
        "merge": {"ms": round(med["merge"], 4), "gbs": round(merge_bytes / med["merge"] / 1e6, 1),
                  "frac_hbm": round(merge_bytes / med["merge"] / 1e6 / hbm, 3),
                  "note": "mla_merge_state alone (the unfused step); the pipeline fuses it"},
        "hbm_peak_gbs": hbm, "hbm_peak_source": peaks["source"],
    }


# ----------------------------------------------------------------------------- reference arm
def bench_reference(args, world, rank):
    """The oracle on the host cores, on the same workload and config as our arm.  Each
    step runs the oracle over (request, head) pieces of the workload for a bounded time
    (so the whole run ends within minutes); the step's wall time is measured, and the
    value is the FLOPs of the pieces done over that time."""
    if rank != 0:
        return None
    b = wl.make_workload(args.workload)
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle_sample(b, target_s=per_step)
    vals, walls, desc, cores = [], [], "", 1
    for _ in range(args.steps):
        t0 = time.perf_counter()
        v, cores, desc = time_oracle_sample(b, target_s=per_step)
        walls.append(time.perf_counter() - t0)
        vals.append(v)
    value = statistics.median(vals)
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(statistics.mean(walls) * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16; no dataset)",
        "config": workload_config(b, args.workload, world, L2_NOTE),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "note": ("the pages publish no runnable implementation; the reference arm is the fp64 oracle on host "
                 "cores.  A step is a bounded sample of the workload's (request, head) pieces (pool start-up "
                 "excluded from the value); ms_per_step is the measured wall time of such a step, not of the "
                 "whole workload"),
    }


def kernel_case(name: str, reps: int = 3):
    """A fixed case of one kernel (small ones for multi-pass captures; ``absorbed_full`` is the
    absorbed bench row's shape, for one-pass counters), launched `reps` times and nothing
    else: the command that the ncu captures under profiles/ run (``--kernel-case``)."""
    import torch
    import chunked_prefill_attention_ragged_gb300 as mla
    from chunked_prefill_attention_ragged_gb300.pipeline import ChunkedPrefill
    dev = torch.device("cuda", 0)
    cb = wl.make_chunked_prefix()
    table = torch.from_numpy(cb.block_table).to(dev)

    def dev_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    if name == "fp8_gather":
        # every chunk of the chunked-prefix workload out of an fp8 cache of the same shape
        b = cb.new
        pipe = ChunkedPrefill(b.qo_indptr, cb.layout.cu_seq_lens, cb.layout.chunk_starts, b.num_heads,
                              sm_scale=b.sm_scale, device=dev, cache_fp8=True)
        cache8 = torch.from_numpy(wl.random_fp8_cache(np.random.default_rng(1102), cb.cache.shape[0],
                                                      cb.cache.shape[1], scale_exp=(126, 127),
                                                      code_exp=(4, 8))).to(dev)
        for _ in range(reps):
            pipe.gather_all(cache8, table)
    elif name == "up_proj_paged":
        # the first 1024 prefix positions of each request: 4096 rows x 128 heads (335 MB of K/V)
        cache, w = dev_bf16(cb.cache), dev_bf16(cb.w_kvb)
        cu = torch.tensor([0, 1024, 2048, 3072, 4096], dtype=torch.int32, device=dev)
        st = torch.zeros(4, dtype=torch.int32, device=dev)
        k = torch.empty(4096, 128, 192, dtype=torch.bfloat16, device=dev)
        v = torch.empty(4096, 128, 128, dtype=torch.bfloat16, device=dev)
        for _ in range(reps):
            mla.mla_up_proj_paged(cache, table, cu, st, 4096, w, 128, k, v)
    elif name in ("absorbed", "absorbed_full"):
        # small: 1 request of 64 new rows over 2048 cache positions, 128 heads (128 units);
        # full: the absorbed bench row's shape (16384 units), for one-pass traffic counters
        b = absorbed_case(name == "absorbed")
        plan = mla.mla_absorbed_plan(b.qo_indptr, b.kv_lens, b.num_heads, b.block_size, causal=True,
                                     sm_scale=b.sm_scale)
        q, cache = dev_bf16(b.q_abs), dev_bf16(b.cache)
        tab = torch.from_numpy(b.block_table).to(dev)
        for _ in range(reps):
            plan.run(q, cache, tab)
    elif name == "up_proj_paged_split":
        # the same rows, decompressed as the pipeline does: K_nope [T, H, 128] + one rope row per token
        cache, w = dev_bf16(cb.cache), dev_bf16(cb.w_kvb)
        cu = torch.tensor([0, 1024, 2048, 3072, 4096], dtype=torch.int32, device=dev)
        st = torch.zeros(4, dtype=torch.int32, device=dev)
        k = torch.empty(4096, 128, 128, dtype=torch.bfloat16, device=dev)
        v = torch.empty(4096, 128, 128, dtype=torch.bfloat16, device=dev)
        rope = torch.empty(4096, 64, dtype=torch.bfloat16, device=dev)
        for _ in range(reps):
            mla.mla_up_proj_paged_split(cache, table, cu, st, 4096, w, 128, k, v, rope)
    else:
        raise ValueError(name)
    torch.cuda.synchronize()
    print(json.dumps({"kernel_case": name, "launches": reps, "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=1, choices=[0, 1, 3, 4])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-chunked", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the rows of the other workloads")
    ap.add_argument("--no-absorbed", action="store_true", help="skip the absorbed-weight prefill row")
    ap.add_argument("--kernel-case", choices=["fp8_gather", "up_proj_paged", "up_proj_paged_split", "absorbed",
                                              "absorbed_full"],
                    default=None,
                    help="launch one kernel on a fixed case and exit (for profiler captures)")
    args = ap.parse_args()
    if args.kernel_case:
        kernel_case(args.kernel_case)
        return
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_env()
    if args.impl == "reference":
        line = bench_reference(args, world, rank)
    else:
        line = bench_ours(args, world, rank, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
