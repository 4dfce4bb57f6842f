#!/usr/bin/env python3
"""Benchmark of the row-wise top-k hot path on GB300.

Metric: rows/s and achieved HBM GB/s for row-wise top-k (RTop-K) at
N = 2^20 rows, M = 256, k = 32, fp32 i.i.d. N(0, 1) (seed 0 + rank), exact mode
(max_iter = -1, eps = 0), CBSR output fp32 values + int32 indices.

One step = one rtopk_select over the whole 2^20-row batch (every step of the
path: range, bisection, fill pass, CBSR store -- one kernel launch). Inputs are
1.07 GB per rank, larger than the 129 MB L2, so no flush is needed between
steps. Timing: W untimed warm-up steps, then exactly K steps bracketed by a
barrier and torch.cuda.synchronize() on both sides, CUDA events on the
launching stream, max over ranks. Multi-GPU: every rank processes its own
2^20-row batch with no collective on the data path (weak scaling).

Usage:
  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
The reference arm times the CPU oracle (the plain C replay of the method) on
the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import glob
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "rows/s and achieved HBM GB/s (% of peak), row-wise top-k M=256 k=32 N=2^20"
N_ROWS, M_COLS, K_SEL = 1 << 20, 256, 32
WORKLOAD = ("rtopk_select exact (max_iter=-1, eps=0), N=2^20 rows x M=256 fp32 i.i.d. N(0,1) "
            "-> CBSR k=32 fp32 values + int32 indices")
PROFILE_GLOB = os.path.join(ROOT, "profiles", "*.md")


def workload_config(world: int) -> dict:
    """The `config` object of both arms' JSON lines (the same workload on each)."""
    return {"workload": WORKLOAD, "N": N_ROWS, "M": M_COLS, "k": K_SEL, "max_iter": -1, "eps": 0.0,
            "l2": f"inputs larger than L2 ({N_ROWS * M_COLS * 4 / 1e9:.2f} GB per rank; L2 129 MB)",
            "parallelism": f"rows: one {N_ROWS}-row batch per rank x {world}"}


def cpu_model() -> str:
    """The host CPU's model string (/proc/cpuinfo; Arm hosts report no model name)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "CPU part"):
        for line in info.splitlines():
            if line.startswith(key) and ":" in line:
                val = line.split(":", 1)[1].strip()
                if key == "CPU part":
                    parts = {"0xd4f": "Neoverse-V2 (Grace)", "0xd40": "Neoverse-V1", "0xd8e": "Neoverse-N3"}
                    return f"Arm {parts.get(val, 'CPU part ' + val)}"
                return val
    import platform
    return platform.processor() or platform.machine()


def algorithmic_bytes(N, M, k, s_in, s_val, s_idx):
    """Bytes the method must move: read the matrix once, write the CBSR arrays once."""
    return N * M * s_in + N * k * (s_val + s_idx)


# sources that define the timed kernel (fp32 rows of <= 2048 elements, one warp per row)
# and its launch configuration
HEADLINE_SOURCES = ("rtopk_device.cuh", "rtopk_select.cuh", "rtopk_warp.cuh", "rtopk_image16.cuh", "rtopk_lean.cuh", "rtopk_block.cuh",
                    "rtopk_dispatch.cuh", "rtopk_f32.cu", "launch_util.cu")


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in HEADLINE_SOURCES:
        p = os.path.join(ROOT, "maxk_sparse_activations_gb300", "csrc", name)
        with open(p, "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str, src_hash: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches these sources."""
    for p in glob.glob(PROFILE_GLOB):
        kv = {}
        with open(p) as f:
            for line in f:
                if line.startswith("- ") and ":" in line:
                    key, val = line[2:].split(":", 1)
                    kv[key.strip()] = val.strip().strip("`")
        if kv.get("bench_tag") == kernel_tag:
            if kv.get("source_hash") == src_hash and "traffic_bytes_per_launch" in kv:
                return int(float(kv["traffic_bytes_per_launch"])), p
            return None, p
    return None, None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------------------------------------
# clocks sampled during the timed region
# ------------------------------------------------------------------------------------------
class NvmlClockSampler:
    """SM clock, power and clock-event reasons polled through NVML (the driver's
    libnvidia-ml, loaded with ctypes) every ~2 ms on a thread: short timed
    regions (tens of ms) still get samples. Only reads; changes no setting."""
    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_uuid: str | None):
        import ctypes
        self.ct = ctypes
        if not gpu_uuid:  # NVML numbers GPUs independently of CUDA_VISIBLE_DEVICES: go by UUID only
            raise OSError("no GPU UUID")
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(gpu_uuid.encode()), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for " + gpu_uuid)
        self.reason_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(mx))  # NVML_CLOCK_SM
        self.max_mhz = float(mx.value)
        self.samples: list[tuple[float, float, float, int]] = []
        self._stop = threading.Event()
        self.thread = None

    def _one(self):
        ct = self.ct
        mhz, mw, rs = ct.c_uint(0), ct.c_uint(0), ct.c_ulonglong(0)
        self.lib.nvmlDeviceGetClockInfo(self.h, ct.c_int(1), ct.byref(mhz))
        self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(mw))
        self.reason_fn(self.h, ct.byref(rs))
        return float(mhz.value), mw.value / 1000.0, int(rs.value)

    def _loop(self):
        while not self._stop.is_set():
            t = time.time()
            mhz, w, rs = self._one()
            self.samples.append((t, mhz, w, rs))
            time.sleep(0.002)

    def start(self):
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()
        time.sleep(0.02)

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["no NVML samples"], "samples": 0,
                    "source": "nvml"}
        reasons = sorted({name for s in inside for bit, name in self.REASONS.items() if s[3] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in inside), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside), "power_w_max": max(s[2] for s in inside),
                "source": "nvml, ~2 ms polling"}


class ClockSampler:
    """nvidia-smi at 50 ms intervals: the fallback when NVML cannot be loaded."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.uuid = gpu_uuid
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._pump, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _pump(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        used = inside if inside else [r for r in rows if r[0] >= t0 - 0.5][:3]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[4]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "reasons": reasons, "samples": len(inside),
                "power_w_max": max((float(r[3]) for r in used if r[3].replace(".", "", 1).isdigit()),
                                   default=None), "source": "nvidia-smi, 50 ms"}


def make_clock_sampler(uuid: str | None):
    try:
        return NvmlClockSampler(uuid)
    except (OSError, AttributeError):
        return ClockSampler(uuid)


def rejected_clocks(c: dict) -> bool:
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "hw_power_brake_slowdown"}
    if bad & set(c.get("reasons", [])):
        return True
    if c.get("sm_mhz") and c.get("sm_max_mhz") and c["sm_mhz"] < 0.6 * c["sm_max_mhz"] \
            and not c.get("reasons"):
        return True
    return False


# ------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline field)
# ------------------------------------------------------------------------------------------
def time_oracle(x: np.ndarray, k: int, threads: int, min_seconds: float, max_reps: int, fn: str = "replay"):
    """Wall time of the oracle replay (or, fn="sort_topk", the sort definition)
    over x split into `threads` contiguous row blocks."""
    import concurrent.futures as cf
    import oracle  # test infrastructure; only the CPU-baseline leg uses it
    oracle.build()
    blocks = np.array_split(np.arange(x.shape[0]), threads)

    def work(rows):
        if rows.size:
            if fn == "replay":
                oracle.replay(x[rows[0]:rows[-1] + 1], k, -1, 0.0)
            else:
                oracle.sort_topk(x[rows[0]:rows[-1] + 1], k)

    best, reps, t_all = None, 0, time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while reps < max_reps and (reps < 1 or time.perf_counter() - t_all < min_seconds):
            t0 = time.perf_counter()
            list(ex.map(work, blocks))
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
            reps += 1
    return best, reps


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return 0
    from maxk_sparse_activations_gb300 import synth
    threads = os.cpu_count() or 1
    # calibrate on 16384 rows, then size the per-step sample so K + W steps take about a minute
    probe = synth.normal_f32(16384, M_COLS, seed=0)
    t_probe, _ = time_oracle(probe, K_SEL, threads, 0.0, 1)
    rate = probe.shape[0] / max(t_probe, 1e-9)
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    rows = int(min(N_ROWS, max(4096, rate * budget)))
    x = synth.normal_f32(N_ROWS, M_COLS, seed=0)[:rows]
    for _ in range(args.warmup):
        time_oracle(x, K_SEL, threads, 0.0, 1)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time_oracle(x, K_SEL, threads, 0.0, 1)
    dt = (time.perf_counter() - t0) / max(1, args.steps)
    value = rows / dt
    sample = f"first {rows} of the 2^20 rows per step, oracle replay (exact), {threads} threads"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(world),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": threads, "kind": "oracle",
                         "sample": sample, "sample_rows": rows, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------
# GB300 arm
# ------------------------------------------------------------------------------------------
def run_gb300(args, rank: int, world: int):
    import torch
    import torch.distributed as dist
    from maxk_sparse_activations_gb300 import _lib, api, synth

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    lib = _lib.load()
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    x_host = synth.normal_f32(N_ROWS, M_COLS, seed=rank)
    x = torch.from_numpy(x_host).to(dev)
    vals = torch.empty((N_ROWS, K_SEL), dtype=torch.float32, device=dev)
    idx = torch.empty((N_ROWS, K_SEL), dtype=torch.int32, device=dev)
    sptr = stream.cuda_stream

    def step():
        rc = lib.rtopk_select(x.data_ptr(), N_ROWS, M_COLS, K_SEL, -1, 0.0, _lib.RTOPK_F32,
                              vals.data_ptr(), idx.data_ptr(), sptr)
        if rc != 0:
            raise RuntimeError(_lib.strerror(rc))

    def timed(fn, steps):
        barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        ms = e0.elapsed_time(e1)
        if world > 1:
            t = torch.tensor([ms], device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ms = float(t.item())
        return ms

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = None
    for attempt in range(2):
        sampler = make_clock_sampler(uuid) if rank == 0 else None
        if sampler:
            sampler.start()
        w0 = time.time()
        ms = timed(step, args.steps)
        w1 = time.time()
        if sampler:
            sampler.stop()
            clocks = sampler.summary(w0, w1)
        redo = torch.tensor([1 if (clocks and rejected_clocks(clocks)) else 0], device=dev)
        if world > 1:
            dist.broadcast(redo, 0)
        if not int(redo.item()) or attempt == 1:
            break
    ms_per_step = ms / args.steps
    rows_per_s = world * N_ROWS / (ms_per_step * 1e-3)
    bytes_step = algorithmic_bytes(N_ROWS, M_COLS, K_SEL, 4, 4, 4)
    gbs = bytes_step / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    src_hash = kernel_source_hash()
    traffic, prof = profiled_traffic("rtopk_select_f32_M256_k32", src_hash)

    # ---- end to end through the public API with HOST buffers: the kernel reads
    # the pinned input and writes the pinned CBSR result over the host link
    # (NVLink-C2C), so both transfers happen inside every timed step
    x_pin = torch.from_numpy(x_host).pin_memory()
    v_pin = torch.empty((N_ROWS, K_SEL), dtype=torch.float32).pin_memory()
    i_pin = torch.empty((N_ROWS, K_SEL), dtype=torch.int32).pin_memory()

    def e2e_step():
        api.rtopk_select(x_pin, K_SEL, vals=v_pin, idx=i_pin, stream=stream)

    e2e_steps = max(3, min(args.steps, 50))
    for _ in range(2):
        e2e_step()
    ms_e2e = timed(e2e_step, e2e_steps) / e2e_steps
    e2e_ok = bool(torch.equal(i_pin, idx.cpu()) and torch.equal(v_pin, vals.cpu()))

    extra = {}
    if not args.no_extra:
        extra = secondary_measurements(torch, api, synth, dev, x, stream, world, timed)

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            threads = os.cpu_count() or 1
            t_cpu, reps = time_oracle(x_host, K_SEL, threads, 5.0, 3)
            # single-threaded replay and sort definition on bounded row samples
            n1, ns = min(N_ROWS, 1 << 16), min(N_ROWS, 1 << 14)
            t_one, _ = time_oracle(x_host[:n1], K_SEL, 1, 0.0, 1)
            t_sort, _ = time_oracle(x_host[:ns], K_SEL, 1, 0.0, 1, fn="sort_topk")
            t_sort_all, _ = time_oracle(x_host[:n1], K_SEL, threads, 0.0, 1, fn="sort_topk")
            cpu = {"value": N_ROWS / t_cpu, "unit": "rows/s", "cores": threads, "kind": "oracle",
                   "sample": f"all {N_ROWS} rows of the workload, oracle replay (exact), best of {reps}, "
                             f"{threads} threads on contiguous row blocks",
                   "cpu_model": cpu_model(),
                   "replay_single_thread_rows_per_s": n1 / t_one,
                   "replay_single_thread_sample": f"first {n1} rows, 1 thread",
                   "sort_topk_single_thread_rows_per_s": ns / t_sort,
                   "sort_topk_single_thread_sample": f"first {ns} rows, 1 thread",
                   "sort_topk_all_cores_rows_per_s": n1 / t_sort_all}
        line = {
            "metric": METRIC, "value": rows_per_s, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": workload_config(world),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "traffic": traffic,
                         "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured"
                         else "fallback", "algorithmic_bytes_per_launch": bytes_step,
                         "kernel": "rtopk_lean_kernel<float,NE=8,int32>",
                         "traffic_source": os.path.relpath(prof, ROOT) if prof else None},
            "cpu_baseline": cpu,
            "e2e": {"value": world * N_ROWS / (ms_e2e * 1e-3), "unit": "rows/s",
                    "h2d_bytes_per_step": N_ROWS * M_COLS * 4, "d2h_bytes_per_step": N_ROWS * K_SEL * 8,
                    "ms_per_step": ms_e2e, "path": "rtopk_select on pinned host buffers (zero-copy "
                    "reads/writes over the host link)", "matches_device_result": e2e_ok},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "hbm_gbs": gbs, "pct_of_nominal_8tbs": gbs / 8000.0,
            "source_hash": src_hash,
            "extra": extra,
        }
        print(json.dumps(line), flush=True)
    return 0


def secondary_measurements(torch, api, synth, dev, x, stream, world, timed):
    """Early-stop speed, the pass-count histogram, and the fused MaxK layer (bf16)."""
    out = {}
    N, M, k = N_ROWS, M_COLS, K_SEL
    vals = torch.empty((N, k), dtype=torch.float32, device=dev)
    idx = torch.empty((N, k), dtype=torch.int32, device=dev)
    reps = 50
    for m in (-1, 2, 3, 4, 5, 8):  # the early-stop settings of the MaxK-shaped configuration
        f = lambda: api.rtopk_select(x, k, m, 0.0, vals=vals, idx=idx)
        f()
        out[f"rtopk_f32_max_iter_{m}_us"] = timed(f, reps) / reps * 1e3
    # exact mode with per-row pass counts: the binary32 replay kernel (the packed
    # 16-bit search runs only when pass counts are not requested)
    iters_buf = torch.empty((N,), dtype=torch.int32, device=dev)
    st_buf = torch.zeros((1,), dtype=torch.int32, device=dev)
    f = lambda: api.rtopk_select_stats(x, k, vals=vals, idx=idx, iters=iters_buf, status=st_buf)
    f()
    out["rtopk_f32_exact_binary32_with_pass_counts_us"] = timed(f, reps) / reps * 1e3
    # context: PyTorch's own row-wise topk on the same matrix (the baseline the RTop-K
    # page reports its 7.29x exact / 11.49x max_iter=2 kernel speedups against)
    f = lambda: torch.topk(x, k, dim=1, largest=True, sorted=True)
    f()
    t_torch = timed(f, 10) / 10 * 1e3
    f = lambda: torch.topk(x, k, dim=1, largest=True, sorted=False)
    f()
    t_torch_unsorted = timed(f, 10) / 10 * 1e3
    out["torch_topk_sorted_us"] = t_torch
    out["torch_topk_unsorted_us"] = t_torch_unsorted
    out["speedup_vs_torch_topk_exact"] = t_torch / out["rtopk_f32_max_iter_-1_us"]
    out["speedup_vs_torch_topk_max_iter_2"] = t_torch / out["rtopk_f32_max_iter_2_us"]
    # bucketed approximate top-k (independent per-bucket selections): speed and
    # hit rate against the exact result on the first 2^16 rows
    from maxk_sparse_activations_gb300 import accuracy
    api.rtopk_select(x, k, vals=vals, idx=idx)
    ev = vals[: 1 << 16].cpu().numpy()
    ei = idx[: 1 << 16].cpu().numpy()
    # B = 16 / 32 keep two / one elements per bucket (no search)
    for B in (2, 4, 8, 16, 32):
        f = lambda: api.rtopk_select_bucketed(x, k, B, vals=vals, idx=idx)
        f()
        t_b = timed(f, reps) / reps * 1e3
        acc = accuracy.compare(vals[: 1 << 16].cpu().numpy(), idx[: 1 << 16].cpu().numpy(), ev, ei)
        out[f"bucketed_B{B}"] = {"us": t_b, "hit_rate_mean": acc["hit_rate_mean"],
                                 "hit_rate_worst": acc["hit_rate_worst"], "r_min_mean": acc["r_min_mean"]}
    # early-stop accuracy against exact on the MaxK-shaped 2^18-row block (the
    # pages report hit rate and max / min relative error for early stopping)
    nacc = 1 << 18
    api.rtopk_select(x, k, vals=vals, idx=idx)
    ev = vals[:nacc].cpu().numpy()
    ei = idx[:nacc].cpu().numpy()
    es = {}
    for m in (2, 3, 4, 5, 8):
        api.rtopk_select(x, k, m, 0.0, vals=vals, idx=idx)
        es[f"max_iter_{m}"] = accuracy.compare(vals[:nacc].cpu().numpy(), idx[:nacc].cpu().numpy(), ev, ei)
    out["early_stop_accuracy_vs_exact"] = es
    _, _, iters, st = api.rtopk_select_stats(x, k)
    it = iters.cpu().numpy()
    out["passes_exact"] = {"median": float(np.median(it)), "p90": float(np.percentile(it, 90)),
                           "max": int(it.max()), "frac_le_16": float(np.mean(it <= 16)),
                           "histogram": np.bincount(it, minlength=1).tolist(), "status": int(st.item())}
    xb = torch.from_numpy(synth.normal_bf16(N, M, seed=0).view(np.int16)).view(torch.bfloat16).to(dev)
    fv = torch.empty((N, k), dtype=torch.bfloat16, device=dev)
    fi = torch.empty((N, k), dtype=torch.int16, device=dev)
    fwd = lambda: api.maxk_forward(xb, k, vals=fv, idx=fi)
    fwd()
    t_f = timed(fwd, reps) / reps
    dy = torch.from_numpy(synth.normal_bf16(N, k, seed=1).view(np.int16)).view(torch.bfloat16).to(dev)
    g = torch.empty((N, M), dtype=torch.bfloat16, device=dev)
    bwd = lambda: api.maxk_backward_scatter(dy, fi, M, grad=g)
    bwd()
    t_b = timed(bwd, reps) / reps
    bytes_f = algorithmic_bytes(N, M, k, 2, 2, 2)
    bytes_b = N * k * 4 + N * M * 2
    out["maxk_forward_bf16"] = {"us": t_f * 1e3, "gbs": bytes_f / (t_f * 1e-3) / 1e9,
                                "rows_per_s": N / (t_f * 1e-3), "bytes": bytes_f}
    out["maxk_backward_scatter_bf16"] = {"us": t_b * 1e3, "gbs": bytes_b / (t_b * 1e-3) / 1e9,
                                         "bytes": bytes_b}

    # MaxK-GNN aggregation over the CBSR rows (next rows of the path): a synthetic
    # power-law graph, 2^17 nodes, mean in-degree 64, tail exponent 2.5, in-degree
    # capped at 4096 (max/mean ~ 64, as for Reddit's ~21.7k / ~490), mean weights
    n = 1 << 17
    row_ptr, col, w = synth.power_law_graph(n, n, 64.0, seed=5, alpha=2.5, max_degree=4096)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n)
    E = int(col.shape[0])
    g = {name: torch.from_numpy(a).to(dev) for name, a in
         (("rp", row_ptr), ("col", col), ("w", w), ("tp", t_ptr), ("tr", t_row), ("tw", t_w))}
    sd, si = fv[:n].contiguous(), fi[:n].contiguous()
    agg = torch.empty((n, M), dtype=torch.float32, device=dev)
    fwd_g = lambda: api.maxk_spgemm_forward(g["rp"], g["col"], g["w"], sd, si, M, out=agg)
    fwd_g()
    t_gf = timed(fwd_g, reps) / reps
    dsp = torch.empty((n, k), dtype=torch.float32, device=dev)
    bwd_g = lambda: api.maxk_sspmm_backward(g["tp"], g["tr"], g["tw"], agg, si, d_sp=dsp)
    bwd_g()
    t_gb = timed(bwd_g, reps) / reps
    bytes_gf = E * (4 + 4 + k * 4) + n * M * 4 + (n + 1) * 8
    bytes_gb = E * (4 + 4 + k * 4) + n * k * (2 + 4) + (n + 1) * 8
    out["gnn_graph"] = {"nodes": n, "edges": E, "M": M, "k": k, "max_in_degree": int(np.diff(row_ptr).max())}
    out["maxk_spgemm_forward"] = {"us": t_gf * 1e3, "gbs": bytes_gf / (t_gf * 1e-3) / 1e9,
                                  "edges_per_s": E / (t_gf * 1e-3), "bytes": bytes_gf}
    out["maxk_sspmm_backward"] = {"us": t_gb * 1e3, "gbs": bytes_gb / (t_gb * 1e-3) / 1e9,
                                  "edges_per_s": E / (t_gb * 1e-3), "bytes": bytes_gb}
    # the backward product with the MaxK scatter fused in: dense bf16 gradient
    # of the MaxK input instead of the n x k intermediate
    gx = torch.empty((n, M), dtype=torch.bfloat16, device=dev)
    bws = lambda: api.maxk_sspmm_backward_scatter(g["tp"], g["tr"], g["tw"], agg, si, M, grad=gx)
    bws()
    t_gs = timed(bws, reps) / reps
    bytes_gs = E * (4 + 4 + k * 4) + n * k * 2 + n * M * 2 + (n + 1) * 8
    # the same gradient unfused: backward product, bf16 rounding (torch), scatter
    dsp16 = torch.empty((n, k), dtype=torch.bfloat16, device=dev)
    def chain():
        api.maxk_sspmm_backward(g["tp"], g["tr"], g["tw"], agg, si, d_sp=dsp)
        dsp16.copy_(dsp)
        api.maxk_backward_scatter(dsp16, si, M, grad=gx)
    chain()
    t_ch = timed(chain, reps) / reps
    out["maxk_sspmm_backward_scatter"] = {"us": t_gs * 1e3, "gbs": bytes_gs / (t_gs * 1e-3) / 1e9,
                                          "edges_per_s": E / (t_gs * 1e-3), "bytes": bytes_gs,
                                          "unfused_chain_us": t_ch * 1e3}
    del agg, gx, dsp, dsp16, g

    # configuration 3 (shape sweep) and configuration 4 (long rows, adversarial
    # values): throughput tables, each launch timed alone with L2 flushed before it
    peak, _ = measured_peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed_cold(fn, reps):
        ms = []
        for _ in range(reps):
            flush.fill_(1)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        return statistics.median(ms)

    sweep = {}
    n3 = 1 << 18
    gen = torch.Generator(device=dev).manual_seed(0)
    for m3 in (128, 256, 512, 1024):
        x32 = torch.randn(n3, m3, device=dev, generator=gen)
        for dt, xx in (("f32", x32), ("bf16", x32.to(torch.bfloat16))):
            s_in = xx.element_size()
            for k3 in (16, 32, 64, 128, 256):
                if k3 >= m3:
                    continue
                v3 = torch.empty((n3, k3), dtype=xx.dtype, device=dev)
                i3 = torch.empty((n3, k3), dtype=torch.int32, device=dev)
                for mi in (-1, 2):
                    f = lambda: api.rtopk_select(xx, k3, mi, vals=v3, idx=i3)
                    f()
                    t = timed_cold(f, 7)
                    by = algorithmic_bytes(n3, m3, k3, s_in, s_in, 4)
                    sweep[f"{dt}_M{m3}_k{k3}_{'exact' if mi < 0 else 'max_iter_2'}"] = {
                        "us": t * 1e3, "gbs": by / (t * 1e-3) / 1e9, "frac_of_measured_hbm": by / (t * 1e-3) / 1e9 / peak,
                        "rows_per_s": n3 / (t * 1e-3)}
                del v3, i3
        del x32, xx
    out["config3_sweep_N2^18"] = sweep
    long_rows = {}
    n4 = 65536
    for m4 in (2048, 4096, 8192):
        x4 = torch.rand(n4, m4, device=dev, generator=gen) * 2 - 1
        sets = {"uniform": x4}
        xo = torch.randn(n4, m4, device=dev, generator=gen)
        hit = torch.rand(n4, m4, device=dev, generator=gen) < 0.01
        sign = torch.where(torch.rand(n4, m4, device=dev, generator=gen) < 0.5, -1e30, 1e30)
        sets["outliers_1e30"] = torch.where(hit, sign, xo)
        del xo, hit, sign
        for name, xx in sets.items():
            for k4 in (64, 256, 1024):
                v4 = torch.empty((n4, k4), dtype=torch.float32, device=dev)
                i4 = torch.empty((n4, k4), dtype=torch.int32, device=dev)
                f = lambda: api.rtopk_select(xx, k4, vals=v4, idx=i4)
                f()
                t = timed_cold(f, 5)
                by = algorithmic_bytes(n4, m4, k4, 4, 4, 4)
                long_rows[f"{name}_M{m4}_k{k4}"] = {
                    "us": t * 1e3, "gbs": by / (t * 1e-3) / 1e9, "frac_of_measured_hbm": by / (t * 1e-3) / 1e9 / peak,
                    "rows_per_s": n4 / (t * 1e-3)}
                del v4, i4
        del sets, x4
    out["config4_long_rows_N65536"] = long_rows
    del flush
    torch.cuda.empty_cache()

    # rows past the pages' 8192-element limit: one CTA cluster per row
    for Ml, Nl, kl in ((16384, 16384, 256), (65536, 4096, 256)):
        xl = torch.randn(Nl, Ml, device=dev, generator=torch.Generator(device=dev).manual_seed(3))
        vl = torch.empty((Nl, kl), dtype=torch.float32, device=dev)
        il = torch.empty((Nl, kl), dtype=torch.int32, device=dev)
        f = lambda: api.rtopk_select(xl, kl, vals=vl, idx=il)
        f()
        t_l = timed(f, 10) / 10
        by = Nl * Ml * 4 + Nl * kl * 8
        out[f"cluster_rows_M{Ml}_k{kl}"] = {"us": t_l * 1e3, "gbs": by / (t_l * 1e-3) / 1e9,
                                            "rows_per_s": Nl / (t_l * 1e-3), "N": Nl}
        del xl, vl, il
    return out


def _case_cluster():
    # rows past the pages' limit: 1024 rows of 65536 fp32 N(0,1), k = 256 (268 MB in)
    import torch
    from maxk_sparse_activations_gb300 import api
    dev = torch.device("cuda")
    x = torch.randn(1024, 65536, device=dev, generator=torch.Generator(device=dev).manual_seed(3))
    v = torch.empty((1024, 256), device=dev)
    i = torch.empty((1024, 256), dtype=torch.int32, device=dev)
    for _ in range(3):
        api.rtopk_select(x, 256, vals=v, idx=i)


def _case_fused_backward():
    # the aggregation graph of the secondary measurements (2^17 nodes, mean
    # in-degree 64, power-law tail), M = 256, k = 32: fused backward + scatter
    import torch
    from maxk_sparse_activations_gb300 import api, synth
    dev = torch.device("cuda")
    n, M, k = 1 << 17, 256, 32
    xb = torch.from_numpy(synth.normal_bf16(n, M, seed=0).view(np.int16)).view(torch.bfloat16).to(dev)
    _, fi = api.maxk_forward(xb, k)
    row_ptr, col, w = synth.power_law_graph(n, n, 64.0, seed=5, alpha=2.5, max_degree=4096)
    t_ptr, t_row, t_w = synth.transpose_graph(row_ptr, col, w, n)
    tp, tr, tw = (torch.from_numpy(a).to(dev) for a in (t_ptr, t_row, t_w))
    dout = torch.randn(n, M, device=dev)
    gx = torch.empty((n, M), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        api.maxk_sspmm_backward_scatter(tp, tr, tw, dout, fi, M, grad=gx)


def _case_maxk_forward():
    # the MaxK forward of the fused-layer workload at a quarter of its rows:
    # 2^18 x 256 bf16 N(0,1) -> CBSR k = 32 (bf16 values + int16 indices)
    import torch
    from maxk_sparse_activations_gb300 import api, synth
    dev = torch.device("cuda")
    xb = torch.from_numpy(synth.normal_bf16(1 << 18, 256, seed=0).view(np.int16)).view(torch.bfloat16).to(dev)
    for _ in range(3):
        api.maxk_forward(xb, 32)


def _case_maxk_backward():
    # the MaxK backward of the fused-layer workload at a quarter of its rows:
    # 2^18 rows, k = 32 bf16 gradients at the forward's int16 indices -> dense
    # 2^18 x 256 bf16 gradient (128 MB written)
    import torch
    from maxk_sparse_activations_gb300 import api, synth
    dev = torch.device("cuda")
    n, M, k = 1 << 18, 256, 32
    xb = torch.from_numpy(synth.normal_bf16(n, M, seed=0).view(np.int16)).view(torch.bfloat16).to(dev)
    _, fi = api.maxk_forward(xb, k)
    dy = torch.from_numpy(synth.normal_bf16(n, k, seed=1).view(np.int16)).view(torch.bfloat16).to(dev)
    g = torch.empty((n, M), dtype=torch.bfloat16, device=dev)
    for _ in range(3):
        api.maxk_backward_scatter(dy, fi, M, grad=g)


def _case_bucketed():
    # bucketed top-k, B = 4, on a quarter of the headline matrix: 2^18 x 256
    # fp32 N(0,1), k = 32 (268 MB in)
    import torch
    from maxk_sparse_activations_gb300 import api, synth
    dev = torch.device("cuda")
    x = torch.from_numpy(synth.normal_f32(1 << 18, 256, seed=0)).to(dev)
    for _ in range(3):
        api.rtopk_select_bucketed(x, 32, 4)


def _case_spgemm():
    # the MaxK-GNN forward aggregation of the bench extras: 2^17-node power-law
    # graph (mean in-degree 64, capped at 4096), CBSR k = 32 of M = 256
    import torch
    from maxk_sparse_activations_gb300 import api, synth
    dev = torch.device("cuda")
    n, M, k = 1 << 17, 256, 32
    row_ptr, col, w = synth.power_law_graph(n, n, 64.0, seed=5, alpha=2.5, max_degree=4096)
    xb = torch.from_numpy(synth.normal_bf16(n, M, seed=0).view(np.int16)).view(torch.bfloat16).to(dev)
    sd, si = api.maxk_forward(xb, k)
    rp, cl, ww = (torch.from_numpy(a).to(dev) for a in (row_ptr, col, w))
    out = torch.empty((n, M), dtype=torch.float32, device=dev)
    for _ in range(3):
        api.maxk_spgemm_forward(rp, cl, ww, sd, si, M, out=out)


def _case_long_rows():
    # exact rows of 4096 (the multi-warp 16-bit kernel, four warps per row):
    # 2^14 x 4096 fp32 N(0,1), k = 256 (268 MB in)
    import torch
    from maxk_sparse_activations_gb300 import api, synth
    dev = torch.device("cuda")
    x = torch.from_numpy(synth.normal_f32(1 << 14, 4096, seed=0)).to(dev)
    for _ in range(3):
        api.rtopk_select(x, 256)


def _case_early_stop():
    # early stop (max_iter = 2, the replay kernel) on a quarter of the headline
    # matrix: 2^18 x 256 fp32 N(0,1), k = 32 (268 MB in)
    import torch
    from maxk_sparse_activations_gb300 import api, synth
    dev = torch.device("cuda")
    x = torch.from_numpy(synth.normal_f32(1 << 18, 256, seed=0)).to(dev)
    for _ in range(3):
        api.rtopk_select(x, 32, 2)


PROFILE_CASES = {"cluster": _case_cluster, "fused-backward": _case_fused_backward, "early-stop": _case_early_stop,
                 "maxk-forward": _case_maxk_forward, "maxk-backward": _case_maxk_backward,
                 "bucketed": _case_bucketed, "long-rows": _case_long_rows, "spgemm": _case_spgemm}


def run_case(name: str) -> int:
    import torch
    PROFILE_CASES[name]()
    torch.cuda.synchronize()
    return 0


def main():
    global N_ROWS
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=N_ROWS,
                    help="rows per rank (default 2^20, the metric's workload; smaller only for profiling)")
    ap.add_argument("--case", choices=sorted(PROFILE_CASES),
                    help="run three launches of one secondary kernel on its workload and exit "
                         "(a small, self-contained target for profiler captures; prints no JSON)")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="reference arm: CPU seconds the whole run's sampled steps aim for")
    args = ap.parse_args()
    N_ROWS = args.rows
    if args.case:
        return run_case(args.case)
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # N ranks, one process per GPU, launched the way torchrun launches them
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        return subprocess.call(cmd)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch one rank per GPU")
    if world > 1:
        import torch
        import torch.distributed as dist
        if args.impl == "gb300":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    try:
        if args.impl == "reference":
            return run_reference(args, rank, world)
        return run_gb300(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
