"""Benchmark: MLA decode throughput (achieved HBM GB/s, µs per call) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one mla_decode call (stage 1 + split reduce) over the workload's
whole batch. Default workload: fp8, B=64, kv_len=8192 (16 q heads / 1 latent
KV head, 576/512 dims, page_size 1): the bandwidth-bound headline, 304 MB of
algorithmic traffic per call. Inputs are synthetic (seeded N(0,1)); two copies
rotate so no call finds the previous call's rows in L2 (each copy is larger
than the 129 MB L2). Timing: K decode calls captured in CUDA graphs, bracketed
by a barrier, a device synchronise and CUDA events; max over ranks. Under
torchrun every rank runs an independent replica (weak scaling, no collective
on the data path).

--impl reference times the float64 CPU oracle (the only reference this method
has here) on the host cores, one bounded sample of the workload per step.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import mla_inputs as mi  # noqa: E402

PROFILES = os.path.join(ROOT, "profiles")
METRIC = "MLA decode achieved HBM GB/s (KV + Q + O bytes per call / time)"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- distributed helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def replica_seed_offset(rank: int, copy: int) -> int:
    """Seed offset of input copy `copy` on `rank`: every rank holds its own independent replica."""
    return 1000 * rank + copy


def whole_job_gbs(step_bytes: int, steps: int, ws: int, ms_max: float) -> float:
    """Whole-job throughput: the bytes all ranks processed over the slowest rank's time."""
    return step_bytes * steps * ws / (ms_max * 1e-3) / 1e9


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- clocks (NVML, read only)

class ClockSampler:
    """Samples SM clock and clock-event reasons of one GPU in a thread (NVML via ctypes).

    Each sample carries the region that was marked when it was taken (mark(name)
    before a region, mark(None) after it), so a summary can cover the samples
    taken inside one timed region."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting",
               0x1: "gpu_idle", 0x10: "sync_boost", 0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.0005):
        self.period = period_s
        self.samples = []  # (region, sm_mhz, reasons)
        self.region = None
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.error = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            self.handle = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(device_index)
            ok = False
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                key = str(uuid)
                key = key if key.startswith("GPU-") else "GPU-" + key
                ok = self.nvml.nvmlDeviceGetHandleByUUID(key.encode(), ctypes.byref(self.handle)) == 0
            if not ok:
                idx = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(device_index)).split(",")[device_index])
                if self.nvml.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(self.handle)) != 0:
                    raise OSError("no NVML handle")
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
        except Exception as e:  # NVML missing: report no clocks rather than fail the benchmark
            self.nvml = None
            self.error = str(e)

    def _read(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk))
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self.handle, ctypes.byref(rs))
        return int(clk.value), int(rs.value)

    def _sample(self):
        try:
            region = self.region
            mhz, reasons = self._read()
            self.samples.append((region, mhz, reasons))
        except Exception:
            pass

    def _loop(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        if self.nvml is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()

    def mark(self, region):
        """Enter (name) or leave (None) a region; a sample is taken at each mark."""
        if self.nvml is not None:
            if region is None:
                self._sample()
            self.region = region
            if region is not None:
                self._sample()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self, region) -> dict:
        """Clocks over the samples of one region (None: every sample taken inside any region)."""
        sel = [x for x in self.samples if (x[0] == region if region is not None else x[0] is not None)]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml", "note": self.error or "no samples"}
        mhz = [x[1] for x in sel]
        mask = 0
        for x in sel:
            mask |= x[2]
        reasons = [name for bit, name in self.REASONS.items() if mask & bit and name != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_min_mhz": min(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz), "period_ms": self.period * 1e3,
                "region": region or "every timed region", "source": "nvml"}


# ---------------------------------------------------------------- helpers

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


STAGE1_KERNELS = {
    # kernel name -> (profile file stem, sources whose bytes identify the compiled kernel)
    "mla_stage1_fp8_umma_kernel": ("stage1_umma", ("stage1_umma.cu", "umma.cuh", "ptx.cuh", "internal.h")),
    "mla_stage1_kernel": ("stage1_mma", ("stage1.cu", "ptx.cuh", "internal.h")),
    "mla_stage1_a16w8_umma_kernel": ("stage1_umma_a16", ("stage1_umma_a16.cu", "umma.cuh", "ptx.cuh", "internal.h")),
    "mla_stage1_fp8_pairs_umma_kernel": ("stage1_umma_pairs",
                                         ("stage1_umma_pairs.cu", "umma.cuh", "ptx.cuh", "internal.h")),
}


def stage1_source_sha(kernel: str) -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_09_gb300", "csrc")
    for f in STAGE1_KERNELS[kernel][1]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per stage-1 launch from the committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(PROFILES, f"{STAGE1_KERNELS[kernel][0]}_{workload}.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("source_sha") != stage1_source_sha(kernel):
        return None
    return d.get("dram_bytes_per_launch")


def oracle_sample(w: mi.Workload, inp: mi.Inputs, n_seq: int, min_seconds: float = 0.0):
    """Time the float64 oracle on the first n_seq sequences (0: all), in whole passes repeated
    until min_seconds have elapsed; returns (seconds, bytes, threads, passes)."""
    import oracle
    lib = oracle.load()
    ids = list(range(min(n_seq, inp.batch) if n_seq > 0 else inp.batch))
    lens = inp.lengths()
    row_bytes = inp.kv_row_bytes
    nbytes = sum(int(lens[i]) * row_bytes for i in ids) + len(ids) * 16 * (576 + 512) * 2
    passes = 0
    t0 = time.perf_counter()
    while True:
        oracle.decode(inp.q, inp.kv, inp.kv_indptr, inp.kv_indices, inp.sm_scale, inp.mode, inp.kv_scale,
                      seq_ids=ids, lib=lib)
        passes += 1
        secs = time.perf_counter() - t0
        if secs >= min_seconds:
            return secs, nbytes * passes, oracle.threads(lib), passes


# ---------------------------------------------------------------- our arm

def parse_layout(text: str):
    """'rows' | 'rows:shuffled' | 'pages:N' | 'pages:N:shuffled' -> (kind, page_size, shuffled)."""
    parts = text.split(":")
    if parts[0] == "rows" and len(parts) <= 2 and parts[1:] in ([], ["shuffled"]):
        return "rows", 1, parts[1:] == ["shuffled"]
    if parts[0] == "pages" and len(parts) in (2, 3) and parts[1].isdigit() and int(parts[1]) >= 1 \
            and parts[2:] in ([], ["shuffled"]):
        return "pages", int(parts[1]), parts[2:] == ["shuffled"]
    raise SystemExit(f"bad --layout {text!r}: rows, rows:shuffled, pages:N or pages:N:shuffled")


def l2_bytes(dev) -> int:
    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2 ** 20)


def copies_for(bytes_per_copy: int, dev) -> int:
    """Input copies rotated call after call so that no call finds its inputs in L2:
    two when one copy exceeds L2, else enough that the copies span three L2s."""
    l2 = l2_bytes(dev)
    if bytes_per_copy > l2:
        return 2
    return max(2, -(-3 * l2 // max(bytes_per_copy, 1)))


def gpu_lead(cycles: int = 20_000_000):
    """Queue ~10 ms of GPU spinning ahead of a timed region's start event: the host
    then enqueues the region's launches while the GPU is still busy, so a host-side
    delay (a slow launch call, a driver lock held by the clock sampler) does not
    fall between the start event and the region's first kernel."""
    torch.cuda._sleep(cycles)


class GraphTimer:
    """K calls of `call(k)` (k = call index) captured in CUDA graphs of `chunk`
    calls each and replayed; CUDA events between replays on the replay stream."""

    def __init__(self, call, steps: int, chunk: int):
        self.steps = steps
        self.chunk = max(1, min(chunk, steps))
        reps, tail = divmod(steps, self.chunk)
        self.reps = reps
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        self.graphs = []
        for n in ([self.chunk] if reps else []) + ([tail] if tail else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    for k in range(n):
                        call(k)
            self.graphs.append(g)
        torch.cuda.current_stream().wait_stream(s)
        self.tail = self.graphs[-1] if tail else None
        self.main = self.graphs[0] if reps else None
        for g in self.graphs:  # one untimed replay of each graph
            g.replay()
        torch.cuda.synchronize()

    def run(self):
        """Returns (total ms, median µs per call over the full replays)."""
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(self.reps + 1)]
        e1 = torch.cuda.Event(enable_timing=True)
        gpu_lead()
        marks[0].record()
        for k in range(self.reps):
            self.main.replay()
            marks[k + 1].record()
        if self.tail is not None:
            self.tail.replay()
        e1.record()
        torch.cuda.synchronize()
        ms = marks[0].elapsed_time(e1)
        per = [marks[k].elapsed_time(marks[k + 1]) * 1e3 / self.chunk for k in range(self.reps)]
        return ms, (statistics.median(per) if per else ms * 1e3 / self.steps)


def time_stage1_graph(mla, devs, scales, outs, plan, mode, calls: int) -> float:
    """µs per stage-1 launch, timed the way the decode call runs it: consecutive
    stage-1-only launches (each with the programmatic-serialisation attribute the
    decode uses) in a CUDA graph, rotating through the input copies."""
    n = len(devs)

    def call(k):
        d = devs[k % n]
        mla.decode_stage1(d.q, d.kv, scales[k % n], d.kv_indptr, d.kv_indices, outs[k % n], plan=plan,
                          sm_scale=d.sm_scale, dtype_mode=mode)

    chunk = n * max(1, 64 // n)
    t = GraphTimer(call, max(calls, chunk), chunk)
    ms, _ = t.run()
    return ms * 1e3 / t.steps


def bench_ours(args):
    import mla_decode_attention_09_gb300 as mla
    from mla_decode_attention_09_gb300 import build as mla_build

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(ws, "nccl")
    dev = torch.device("cuda", local)
    mla_build.build()
    w = mi.get_workload(args.workload)
    nbytes = mi.workload_bytes(w)
    kind, page_size, shuffled = parse_layout(args.layout)
    q_len = args.q_len
    default_layout = kind == "rows" and not shuffled and q_len == 1
    # algorithmic bytes: KV rows read once, Q read and O written for every query token
    step_bytes = nbytes["kv"] + (nbytes["q"] + nbytes["o"]) * q_len
    peak, peak_kind = measured_peak()

    # input copies rotated call after call, none found in L2 by the next call that uses it
    # (seeded per rank: independent replicas)
    n_copies = copies_for(step_bytes, dev)

    def make(k):
        seed = w.seed + replica_seed_offset(rank, k)
        lens = mi.workload_lengths(w)
        if kind == "pages":
            return mi.make_paged_inputs(lens, page_size, w.mode, seed, permute=shuffled, device=str(dev))
        if shuffled:
            return mi.make_inputs(lens, w.mode, seed, permute=True, device=str(dev))
        return mi.make_workload(w, device=str(dev), seed_offset=replica_seed_offset(rank, k))

    devs = [make(k) for k in range(n_copies)]
    scales = [d.kv_scale_tensor(dev) for d in devs]
    opts = {"num_kv_slots": devs[0].kv.shape[0], "fp8_kernel": args.fp8_kernel}
    last_host = devs[0].kv_last_page_len.cpu() if kind == "pages" else None
    queries = None
    if q_len > 1:
        queries = []
        for k in range(n_copies):
            qh, qo = mi.make_query_tokens([q_len] * w.batch, seed=w.seed + 50 + replica_seed_offset(rank, k))
            queries.append((qh.to(dev), qo.to(dev)))
        plan = mla.plan_multi(queries[0][1].cpu(), devs[0].kv_indptr.cpu(), causal=True, page_size=page_size,
                              kv_last_page_len_host=last_host, token_pairs=args.token_pairs, **opts)
    elif kind == "pages":
        plan = mla.plan_paged(devs[0].kv_indptr.cpu(), last_host, page_size, **opts)
    else:
        plan = mla.plan(devs[0].kv_indptr.cpu(), 0, **opts)
    info = plan.info()
    outs = [torch.empty((w.batch * q_len, 16, 512), dtype=torch.bfloat16, device=dev) for _ in range(n_copies)]

    def call(k, stream=None):
        k %= n_copies
        d = devs[k]
        if queries is not None:
            mla.decode_multi(queries[k][0], d.kv, scales[k], queries[k][1], d.kv_indptr, d.kv_indices, outs[k],
                             plan=plan, kv_last_page_len=d.kv_last_page_len if kind == "pages" else None,
                             sm_scale=d.sm_scale, dtype_mode=w.mode, stream=stream, validate=False)
        elif kind == "pages":
            mla.decode_paged(d.q, d.kv, scales[k], d.kv_indptr, d.kv_indices, d.kv_last_page_len, page_size, outs[k],
                             sm_scale=d.sm_scale, dtype_mode=w.mode, plan=plan, stream=stream, validate=False)
        else:
            mla.decode(d.q, d.kv, scales[k], d.kv_indptr, d.kv_indices, outs[k], sm_scale=d.sm_scale,
                       dtype_mode=w.mode, plan=plan, stream=stream, validate=False)

    for k in range(max(args.warmup, 3)):
        call(k)
    torch.cuda.synchronize()
    status = plan.check_error()
    if status != 0:
        raise RuntimeError(f"kernel error status {status}")

    # exactly K decode calls in CUDA graphs (chunks of 64 calls, rotating the copies)
    timer = GraphTimer(call, args.steps, n_copies * max(1, 64 // n_copies))
    sampler = ClockSampler(local, period_s=args.clock_period_ms * 1e-3)
    sampler.start()
    barrier(ws)
    torch.cuda.synchronize()
    sampler.mark("timed")
    ms, median_us = timer.run()
    sampler.mark(None)
    barrier(ws)
    ms_max = max_over_ranks(ms, ws, dev)
    status = plan.check_error()
    if status != 0:
        raise RuntimeError(f"kernel error status {status}")
    ms_per_step = ms_max / args.steps
    value = whole_job_gbs(step_bytes, args.steps, ws, ms_max)
    launches_per_step = 1 + (1 if info["num_split_seqs"] > 0 else 0)

    # roofline of the dominant kernel, stage 1, timed as the call runs it (a graph of
    # consecutive stage-1 launches); other layouts than rows with one query token have no
    # stage-1-only entry point and report the whole call
    stage1_only = kind == "rows" and q_len == 1
    sampler.mark("roofline")
    if stage1_only:
        kern_us = time_stage1_graph(mla, devs, scales, outs, plan, w.mode, args.roofline_calls)
    else:
        kern_us = ms_per_step * 1e3
    sampler.mark(None)
    achieved = step_bytes / (kern_us * 1e-6) / 1e9
    if args.fp8_kernel == 1 or w.mode == mi.MODE_BF16:
        kernel = "mla_stage1_kernel"
    elif w.mode == mi.MODE_A16W8:
        kernel = "mla_stage1_a16w8_umma_kernel"
    else:
        kernel = "mla_stage1_fp8_pairs_umma_kernel" if plan.token_pairs else "mla_stage1_fp8_umma_kernel"
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic(kernel, args.workload) if default_layout else None,
                "kernel": kernel, "peak_kind": peak_kind,
                "algorithmic_bytes_per_launch": step_bytes,
                "stage1_us" if stage1_only else "call_us": round(kern_us, 2),
                "call_us": round(ms_per_step * 1e3, 2),
                "call_frac": round(value / ws / peak, 4),
                "timing": ("CUDA graph of consecutive stage-1 launches with the decode's launch attribute"
                           if stage1_only else "the whole decode call")}

    # end to end and the oracle baseline are measured on the row layout with one query token
    e2e = None
    if not args.no_e2e and default_layout:
        e2e = bench_e2e(mla, args, w, devs, scales, outs, plan, ws, dev, step_bytes)
    assert plan.check_error() == 0

    per_config = None
    if rank == 0 and default_layout and not args.no_per_config:
        sampler.mark("per_config")
        per_config = bench_per_config(mla, dev, args, peak, current=(args.workload, ms_per_step * 1e3, median_us,
                                                                     kern_us if stage1_only else None, n_copies))
        sampler.mark(None)
    sampler.stop()

    host0 = (devs[0].to("cpu") if (rank == 0 and ws == 1 and not args.no_cpu_baseline and default_layout)
             else None)
    del devs, outs
    cpu = None
    if host0 is not None:
        n_seq = args.cpu_sample_seqs if args.cpu_sample_seqs > 0 else w.batch
        secs, cbytes, threads, passes = oracle_sample(w, host0, n_seq, args.cpu_min_seconds)
        cpu = {"value": round(cbytes / secs / 1e9, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"float64 oracle on {min(n_seq, w.batch)} of {w.batch} sequences, {passes} whole "
                         f"passes ({secs:.1f} s)"}

    clocks = sampler.summary("timed")
    clocks["all_regions"] = sampler.summary(None)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 5), "us_per_call": round(ms_per_step * 1e3, 2),
        "us_per_call_median": round(median_us, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {mi.MODE_BF16: "bf16", mi.MODE_FP8: "e4m3", mi.MODE_A16W8: "f16"}[w.mode], "data": "synthetic",
        "config": {"workload": args.workload, "desc": w.describe(), "batch": w.batch, "kv_rows": nbytes["rows"],
                   "heads": 16, "qk_dim": 576, "v_dim": 512, "page_size": page_size,
                   "kv_order": "shuffled" if shuffled else ("workload" if kind == "rows" else "in order"),
                   "q_len": q_len, "causal": q_len > 1,
                   "token_pairs": bool(plan.token_pairs) and w.mode == mi.MODE_FP8 and args.fp8_kernel == 0,
                   "bytes_per_call": step_bytes,
                   "l2": (f"{n_copies} input copies rotate call after call "
                          + ("(each larger than L2)" if n_copies == 2 and step_bytes > l2_bytes(dev)
                             else "(together three times L2)")),
                   "timing": "CUDA graphs of decode calls",
                   "plan": {k: info[k] for k in ("num_ctas", "num_work_items", "num_split_seqs")},
                   "fp8_kernel": ("tcgen05" if args.fp8_kernel == 0 else "mma.sync") if w.mode == mi.MODE_FP8 else None},
        "frac_of_peak": round(value / ws / peak, 4), "peak_gbs": peak,
        "roofline": roofline, "per_config": per_config, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": launches_per_step * args.steps,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def bench_per_config(mla, dev, args, peak, current, calls: int = 1000):
    """Every workload of the five, timed like the headline: CUDA graphs of decode calls
    that rotate through enough input copies that none is found in L2, then stage 1 alone
    in a graph of consecutive stage-1 launches. `current` carries the headline's own
    measurement (workload, µs per call, median, stage-1 µs, copies), reused for that row."""
    res = {}
    for name, w in mi.WORKLOADS.items():
        nb = mi.workload_bytes(w)["total"]
        if name == current[0]:
            us, med, s1, n_copies = current[1], current[2], current[3], current[4]
        else:
            n_copies = copies_for(nb, dev)
            devs = [mi.make_workload(w, device=str(dev), seed_offset=k) for k in range(n_copies)]
            scales = [d.kv_scale_tensor(dev) for d in devs]
            plan = mla.plan(devs[0].kv_indptr.cpu(), 0, num_kv_slots=devs[0].kv.shape[0], fp8_kernel=args.fp8_kernel)
            outs = [torch.empty((w.batch, 16, 512), dtype=torch.bfloat16, device=dev) for _ in range(n_copies)]

            def call(k):
                d = devs[k % n_copies]
                mla.decode(d.q, d.kv, scales[k % n_copies], d.kv_indptr, d.kv_indices, outs[k % n_copies],
                           sm_scale=d.sm_scale, dtype_mode=w.mode, plan=plan, validate=False)

            for k in range(3):
                call(k)
            torch.cuda.synchronize()
            assert plan.check_error() == 0
            chunk = n_copies * max(1, 64 // n_copies)
            t = GraphTimer(call, max(calls, chunk), chunk)
            ms, med = t.run()
            us = ms * 1e3 / t.steps
            s1 = time_stage1_graph(mla, devs, scales, outs, plan, w.mode, max(calls, chunk))
            assert plan.check_error() == 0
            del devs, outs, plan
        res[name] = {"desc": w.describe(), "us_per_call": round(us, 2), "us_per_call_median": round(med, 2),
                     "gbs": round(nb / (us * 1e-6) / 1e9, 1), "frac": round(nb / (us * 1e-6) / 1e9 / peak, 4),
                     "stage1_us": round(s1, 2) if s1 is not None else None,
                     "stage1_frac": round(nb / (s1 * 1e-6) / 1e9 / peak, 4) if s1 else None,
                     "bytes": nb, "copies": n_copies}
    res["method"] = ("CUDA graphs of decode calls rotating through input copies (two when one copy exceeds L2, "
                     "else enough to span three L2s); stage 1 alone as a graph of consecutive stage-1 launches")
    return res


def bench_e2e(mla, args, w, devs, scales, outs, plan, ws, dev, step_bytes):
    """End to end through the public API from pinned host buffers: H2D inputs, decode, D2H output."""
    host0 = devs[0].to("cpu")
    pinned = [{"q": host0.q.pin_memory(), "kv": host0.kv.pin_memory(), "ip": host0.kv_indptr.pin_memory(),
               "ix": host0.kv_indices.pin_memory(),
               "ks": torch.tensor([host0.kv_scale], dtype=torch.float32).pin_memory()}]
    out_host = torch.empty((w.batch, 16, 512), dtype=torch.bfloat16).pin_memory()
    d = devs[0]
    h2d = sum(t.numel() * t.element_size() for t in pinned[0].values())
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        p = pinned[0]
        d.q.copy_(p["q"], non_blocking=True)
        d.kv.copy_(p["kv"], non_blocking=True)
        d.kv_indptr.copy_(p["ip"], non_blocking=True)
        d.kv_indices.copy_(p["ix"], non_blocking=True)
        scales[0].copy_(p["ks"], non_blocking=True)
        mla.decode(d.q, d.kv, scales[0], d.kv_indptr, d.kv_indices, outs[0], sm_scale=d.sm_scale,
                   dtype_mode=w.mode, plan=plan, validate=False)
        out_host.copy_(outs[0], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    gpu_lead()
    t0.record()
    for _ in range(e2e_steps):
        e2e_step()
    t1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), ws, dev) / e2e_steps
    e2e = {"value": round(step_bytes * ws / (e2e_ms * 1e-3) / 1e9, 2), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
           "note": "all inputs (q, KV cache, indices, scale) copied from pinned host memory every step"}
    return e2e


# ---------------------------------------------------------------- reference arm (the oracle on host cores)

def bench_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    w = mi.get_workload(args.workload)
    host = mi.make_workload(w)
    lib = oracle.load()
    lens = host.lengths()
    # each step: the oracle over a bounded run of one sequence's rows, sized so K steps stay within minutes
    rows = int(max(64, min(int(lens.max()), 8192 * 50 // max(args.steps, 1))))
    row_bytes = host.kv_row_bytes

    def one(step):
        b = step % w.batch
        n = min(rows, int(lens[b]))
        t0 = time.perf_counter()
        oracle.decode_range(host.q, host.kv, host.kv_indptr, host.kv_indices, host.sm_scale, b, 0, n,
                            host.mode, host.kv_scale, lib=lib)
        return time.perf_counter() - t0, n * row_bytes + 16 * (576 + 512) * 2

    for i in range(args.warmup):
        one(i)
    t_total, b_total = 0.0, 0
    for i in range(args.steps):
        secs, nb = one(i)
        t_total += secs
        b_total += nb
    value = b_total / t_total / 1e9
    threads = oracle.threads(lib)
    sample = f"float64 oracle over the first {rows} rows of one sequence per step (all 16 heads)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_total / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "desc": w.describe(), "batch": w.batch},
        "cpu_baseline": {"kind": "oracle", "cores": threads, "value": round(value, 5), "unit": UNIT,
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="fp8_b64_l8192", choices=list(mi.WORKLOADS) + list(mi.EXTRA_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-per-config", action="store_true", help="leave out the per-workload timings")
    ap.add_argument("--roofline-calls", type=int, default=1000, help="stage-1 launches timed for the roofline")
    ap.add_argument("--clock-period-ms", type=float, default=0.5, help="NVML clock sampling period")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fp8-kernel", type=int, default=0, choices=[0, 1],
                    help="fp8 stage-1 kernel: 0 tcgen05/TMA (default), 1 warp-level mma.sync")
    ap.add_argument("--cpu-sample-seqs", type=int, default=0, help="sequences in the CPU baseline's sample (0: all)")
    ap.add_argument("--cpu-min-seconds", type=float, default=10.0,
                    help="the CPU baseline repeats whole passes over its sample until this much time has passed")
    ap.add_argument("--layout", default="rows",
                    help="KV layout of the workload: rows (its own order), rows:shuffled, pages:N, pages:N:shuffled")
    ap.add_argument("--q-len", type=int, default=1, help="query tokens per sequence (causal)")
    ap.add_argument("--token-pairs", type=int, default=0, choices=[-1, 0, 1],
                    help="several query tokens, fp8 tensor-core kernel: two tokens per pass over the rows "
                         "(0 default: on, -1: one CTA per token)")
    args = ap.parse_args()
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
