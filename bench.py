"""Benchmark of the MoE route / dispatch / combine path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload: DeepSeek-V3-shaped decode with fp8 dispatch (T=1024 tokens from 8
virtual DP ranks, H=7168, E=256, k=8, R=8, C=128), seeded synthetic inputs
resident in HBM. One step = moe_route -> moe_dispatch (fp8) ->
moe_expert_synthetic -> moe_combine through the C ABI, with L2 flushed (a
write and a read of 2x the L2 size) before every call; each call is bracketed
by CUDA events on its stream and the flush is outside the brackets.

  value        dispatch+combine tokens/s = tokens / (dispatch + combine time),
               summed over replicas (N GPUs = N independent replicas, the
               slowest rank's time).
  ms_per_step  mean kernel time of the whole step (all four calls).
  pipelined    the four calls back to back, flushed once per step (the two
               timed loops each run K steps: gpu_launches counts both).
  e2e          the same path through the public API with pinned host buffers:
               H2D of x and logits, the four calls, D2H of out, every step;
               double-buffered so that neighbouring steps' copies overlap the
               compute (the serial figure is reported beside it).
  roofline     the combine kernel (the larger of the two kernels the metric
               names): algorithmic bytes / mean duration vs measured HBM peak.
  cpu_baseline the CPU oracle on every host core over the whole workload, and
               single-threaded on a bounded sample beside it.
  dbo          the dual-batch-overlap step on the 8192-token prefill workload.
  expert_gemm  the grouped fp8 GEMM on the tensor cores (random weights) at the
               decode shape (HBM roofline) and an 8192-token prefill shape
               (tensor roofline), and the decode step with it.

--impl reference times the CPU oracle instead (the reference arm of this
build), on every host core, over the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np

import workloads as W

METRIC = "dispatch+combine tokens/s; achieved HBM GB/s vs GB300 peak (DeepSeek-V3 shape)"
UNIT = "tokens/s"
WORKLOAD = "dsv3_fp8"
DTYPE = "e4m3+bf16 (fp32 arithmetic)"
FALLBACK_HBM_GBS = 6800.0
KERNELS_PER_STEP = 5          # route (top-k/tile, finalize), dispatch, expert, combine
CPU_SAMPLE_TOKENS = 256       # the oracle's bounded sample: 2 of the 8 source ranks


# ---------------------------------------------------------------------------
# algorithmic bytes per call (padding rows are never touched by the method)

def bytes_route(w: W.Workload) -> int:
    # logits in; topk_idx, topk_w, slot out; counts/offsets/rank_counts
    return w.T * w.E * 4 + w.T * w.k * 12 + (2 * w.E + 1 + w.R + 1) * 4


def bytes_dispatch(w: W.Workload, kept: int) -> int:
    meta = w.T * w.k * 8 + kept * 4                       # topk_idx + slot in, recv_src out
    if w.dtype == W.DTYPE_FP8_E4M3_B128:
        return w.T * w.H * 2 + kept * (w.H + 4 * (w.H // 128)) + meta
    return w.T * w.H * 2 + kept * w.H * 2 + meta


def bytes_expert(w: W.Workload, kept: int) -> int:
    if w.dtype == W.DTYPE_FP8_E4M3_B128:
        return kept * (w.H + 4 * (w.H // 128)) + kept * w.H * 2
    return kept * w.H * 2 * 2


def bytes_combine(w: W.Workload, kept: int) -> int:
    return kept * w.H * 2 + w.T * w.H * 2 + w.T * w.k * 12


# ---------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            j = json.load(fh)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


NOMINAL_HBM_GBS = 7900.0      # HBM3e data-sheet rate, for context beside the measured copy peak
FALLBACK_BF16_TFLOPS = 1900.0
FP8_PER_BF16 = 2.0            # nominal dense fp8 : bf16 tensor rate (4.5 : 2.25 PFLOP/s)


def measured_fp8_peak():
    """Dense fp8 tensor peak in TFLOP/s: the measured bf16 GEMM peak (burst and
    sustained) times the nominal fp8:bf16 ratio."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            j = json.load(fh)
        return (FP8_PER_BF16 * float(j["bf16_tflops"]), FP8_PER_BF16 * float(j["bf16_tflops_sustained"]),
                "measured bf16 x 2")
    except Exception:
        return FP8_PER_BF16 * FALLBACK_BF16_TFLOPS, FP8_PER_BF16 * 1700.0, "fallback bf16 x 2"


_X_CACHE = {}


def x_of(w: W.Workload):
    """Host token rows of a workload, drawn once per (seed, T, H)."""
    key = (w.seed, w.T, w.H)
    if key not in _X_CACHE:
        _X_CACHE[key] = W.make_x(w)
    return _X_CACHE[key]


def kernel_source_sha(files) -> str:
    """sha256[:16] of the kernels' code: the sources with comments and
    whitespace removed, so that an edit to a comment keeps a record valid."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "combine_router_top_gb300", "csrc", f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


TRAFFIC_SOURCES = {"combine": ["moe_combine.cu", "moe_internal.cuh"],
                   "dispatch": ["moe_dispatch.cu", "moe_internal.cuh"],
                   "gemm": ["moe_gemm.cu", "moe_internal.cuh"]}


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel source as it is now (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    sha = kernel_source_sha(TRAFFIC_SOURCES[kernel])
    for line in open(path):
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == kernel and f[1] == workload and f[2] == sha:
            return int(float(f[3]))
    return None


class NvmlClockSampler:
    """SM clock and clock-event reasons read through NVML (the driver's libnvidia-ml, read-only queries)
    every 2 ms on a thread, so that even a timed region of a few milliseconds holds samples."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_uuid: str, period_s: float = 0.002):
        import ctypes
        self.rows = []
        self.period = period_s
        self.nv = ctypes.CDLL("libnvidia-ml.so.1")
        if self.nv.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.nv.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle for " + gpu_uuid)
        self.reason_fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0 else None
        self.stop_flag = threading.Event()

    def _read(self):
        import ctypes
        mhz, why = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_flag.is_set():
            ok = self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(mhz)) == 0
            ok = ok and self.reason_fn(self.h, ctypes.byref(why)) == 0
            if ok:
                self.rows.append((time.time(), float(mhz.value), int(why.value)))
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag.set()
        self.thread.join(timeout=2)
        self.nv.nvmlShutdown()

    def summary(self, t0: float, t1: float) -> dict:
        inside = [r for r in self.rows if t0 <= r[0] <= t1]
        note = f"NVML every {1e3 * self.period:.0f} ms, samples inside the timed region ({1e3 * (t1 - t0):.1f} ms)"
        if not inside:
            inside = self.rows
            note = "NVML: no sample inside the timed region; all samples of the run"
        reasons = sorted({name for r in inside for bit, name in self.REASONS.items() if r[2] & bit})
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(inside), "note": note}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms (used when NVML cannot be loaded)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.rows = []
        self.proc = None
        self.err = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception as e:          # no nvidia-smi: report it, do not fail the bench
            self.err = str(e)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": f"nvidia-smi unavailable: {self.err}"}
        inside = [r for (t, r) in self.rows if t0 - 0.05 <= t <= t1 + 0.15]
        note = "samples inside the timed region"
        if not inside:
            inside = [r for (_, r) in self.rows]
            note = "timed region shorter than the sampling period: all samples of the run"
        sm = [float(r[1]) for r in inside if len(r) > 8 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if len(r) > 8 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside if len(r) > 8 for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "note": note}


def clock_sampler(gpu_id: str):
    """The NVML sampler when the driver's NVML library loads, else nvidia-smi."""
    try:
        return NvmlClockSampler(gpu_id)
    except Exception:
        return ClockSampler(gpu_id)


def gpu_id_for_smi(torch, dev: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


# ---------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)

def oracle_sample(w: W.Workload, ntok: int):
    """Seeded inputs of the first ntok tokens of workload w (same generator)."""
    return W.make_x(w, 0, ntok), W.make_logits(w, 0, ntok), W.expert_scale(w)


def time_oracle_step(O, x, lg, s, w: W.Workload) -> dict:
    fp8 = w.dtype == W.DTYPE_FP8_E4M3_B128
    t = {}
    c0 = time.perf_counter()
    idx, wt = O.route(lg, w.k)
    c = O.count(idx, w.E, w.R, w.C)
    c1 = time.perf_counter()
    if fp8:
        rq, rs, _ = O.dispatch_fp8(x, idx, c["slot"], w.E, w.C)
    else:
        rq, _ = O.dispatch_bf16(x, idx, c["slot"], w.E, w.C)
        rs = None
    c2 = time.perf_counter()
    y = O.expert_synthetic(rq, rs, c["counts"], s)
    c3 = time.perf_counter()
    O.combine(y, idx, wt, c["slot"], x.shape[0])
    c4 = time.perf_counter()
    t.update(route=c1 - c0, dispatch=c2 - c1, expert=c3 - c2, combine=c4 - c3, step=c4 - c0)
    return t


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class ThreadedOracle:
    """The oracle's own C functions, unchanged, run over disjoint ranges on every host core: route,
    dispatch and combine over contiguous token ranges, the expert stand-in over contiguous expert
    ranges, one range per thread. ctypes releases the GIL around each foreign call, so the ranges run
    in parallel. Counting runs once, serially: a pair's slot depends on every earlier token. Every
    buffer is allocated once, here, so that allocation is not timed. The oracle writes range-local
    token numbers into recv_src; each dispatch adds the range's first token back (outside the timed
    part), so the buffers equal a single-threaded run's."""

    def __init__(self, O, x, lg, s, w: W.Workload, threads: int):
        import concurrent.futures as cf
        self.O, self.L, self.w = O, O.lib(), w
        self.x = np.ascontiguousarray(x)
        self.lg = np.ascontiguousarray(lg, dtype=np.float32)
        self.s = np.ascontiguousarray(s, dtype=np.float32)
        T, H, E, k, Cap = x.shape[0], w.H, w.E, w.k, w.C
        self.T, self.fp8 = T, w.dtype == W.DTYPE_FP8_E4M3_B128
        self.threads = max(1, min(threads, T if T > 0 else 1))
        # the oracle fills its e4m3 table on first use: do that once here, on one thread
        O.e4m3_encode(np.zeros(1, np.float32))
        O.e4m3_decode(np.zeros(1, np.uint8))
        self.pool = cf.ThreadPoolExecutor(self.threads)
        self.tok = [(T * i // self.threads, T * (i + 1) // self.threads) for i in range(self.threads)]
        ne = max(1, min(self.threads, E))
        self.exp = [(E * i // ne, E * (i + 1) // ne) for i in range(ne)]
        self.idx = np.empty((T, k), np.int32)
        self.wt = np.empty((T, k), np.float32)
        self.counts = np.empty(E, np.int32)
        self.offsets = np.empty(E + 1, np.int32)
        self.slot = np.empty((T, k), np.int32)
        self.rank_counts = np.empty(w.R, np.int32)
        self.dropped = np.zeros(1, np.int32)
        self.recv = np.zeros((E, Cap, H), np.uint8 if self.fp8 else np.uint16)
        self.recv_scale = np.zeros((E, Cap, H // 128), np.float32) if self.fp8 else None
        self.recv_src = np.full((E, Cap), -1, np.int32)
        self.y = np.zeros((E, Cap, H), np.uint16)
        self.out = np.zeros((T, H), np.uint16)

    @staticmethod
    def _at(a, offset_elems: int):
        return None if a is None else a.ctypes.data + offset_elems * a.itemsize

    def _run(self, calls):
        for rc in [f.result() for f in [self.pool.submit(*c) for c in calls]]:
            if rc != 0:
                raise RuntimeError("oracle call rejected its arguments")

    def route(self):
        w, a = self.w, self._at
        self._run([(self.L.oracle_route, t1 - t0, w.E, w.k, a(self.lg, t0 * w.E), a(self.idx, t0 * w.k),
                    a(self.wt, t0 * w.k), None) for t0, t1 in self.tok])
        if self.L.oracle_count(self.T, w.E, w.k, w.R, w.C, a(self.idx, 0), a(self.counts, 0), a(self.offsets, 0),
                               a(self.slot, 0), a(self.rank_counts, 0), a(self.dropped, 0)) != 0:
            raise RuntimeError("oracle_count rejected its arguments")

    def dispatch(self):
        w, a, H = self.w, self._at, self.w.H
        if self.fp8:
            self._run([(self.L.oracle_dispatch_fp8, t1 - t0, H, w.E, w.k, w.C, a(self.x, t0 * H),
                        a(self.idx, t0 * w.k), a(self.slot, t0 * w.k), a(self.recv, 0), a(self.recv_scale, 0),
                        a(self.recv_src, 0)) for t0, t1 in self.tok])
        else:
            self._run([(self.L.oracle_dispatch_bf16, t1 - t0, H, w.E, w.k, w.C, a(self.x, t0 * H),
                        a(self.idx, t0 * w.k), a(self.slot, t0 * w.k), a(self.recv, 0), a(self.recv_src, 0))
                       for t0, t1 in self.tok])

    def fix_recv_src(self):
        for t0, t1 in self.tok[1:]:
            sl, ix = self.slot[t0:t1], self.idx[t0:t1]
            rows = (ix.astype(np.int64) * self.w.C + sl)[sl >= 0]
            self.recv_src.reshape(-1)[rows] += t0

    def expert(self):
        w, a, H = self.w, self._at, self.w.H
        self._run([(self.L.oracle_expert_synthetic, H, e1 - e0, w.C, int(self.fp8), a(self.recv, e0 * w.C * H),
                    a(self.recv_scale, e0 * w.C * (H // 128)), a(self.counts, e0), a(self.s, e0),
                    a(self.y, e0 * w.C * H)) for e0, e1 in self.exp])

    def combine(self):
        w, a, H = self.w, self._at, self.w.H
        self._run([(self.L.oracle_combine, t1 - t0, H, w.E, w.k, w.C, a(self.y, 0), a(self.idx, t0 * w.k),
                    a(self.wt, t0 * w.k), a(self.slot, t0 * w.k), a(self.out, t0 * H)) for t0, t1 in self.tok])

    def step(self) -> dict:
        c0 = time.perf_counter()
        self.route()
        c1 = time.perf_counter()
        self.dispatch()
        c2 = time.perf_counter()
        self.fix_recv_src()
        c3 = time.perf_counter()
        self.expert()
        c4 = time.perf_counter()
        self.combine()
        c5 = time.perf_counter()
        return {"route": c1 - c0, "dispatch": c2 - c1, "expert": c4 - c3, "combine": c5 - c4,
                "step": (c5 - c0) - (c3 - c2)}

    def close(self):
        self.pool.shutdown()


def cpu_baseline(w: W.Workload, budget_s: float = 10.0, max_reps: int = 20) -> dict:
    """The oracle on every host core over the whole workload (ThreadedOracle), and beside it the
    single-threaded oracle on a bounded sample of the first CPU_SAMPLE_TOKENS tokens."""
    import oracle as O
    cores = host_cores()
    x, lg, s = oracle_sample(w, w.T)
    O.lib()
    to = ThreadedOracle(O, x, lg, s, w, cores)
    to.step()                                      # warm: library load, page faults, the codec tables
    reps, tdc, tstep = 0, 0.0, 0.0
    start = time.perf_counter()
    while reps < max_reps and (reps < 2 or time.perf_counter() - start < budget_s):
        t = to.step()
        tdc += t["dispatch"] + t["combine"]
        tstep += t["step"]
        reps += 1
    to.close()
    xs, lgs, _ = oracle_sample(w, CPU_SAMPLE_TOKENS)
    time_oracle_step(O, xs, lgs, s, w)
    r1, tdc1 = 0, 0.0
    start = time.perf_counter()
    while r1 < max_reps and (r1 < 2 or time.perf_counter() - start < budget_s / 4):
        t = time_oracle_step(O, xs, lgs, s, w)
        tdc1 += t["dispatch"] + t["combine"]
        r1 += 1
    return {"value": w.T * reps / tdc, "unit": UNIT, "cores": to.threads, "kind": "oracle",
            "sample": f"all {w.T} tokens, full E/H/k/C, {reps} repetitions on {to.threads} host threads (the oracle's "
                      f"functions over disjoint token / expert ranges); value = tokens / (oracle dispatch + combine "
                      f"time); whole oracle step {1e3 * tstep / reps:.1f} ms",
            "single_thread": {"value": CPU_SAMPLE_TOKENS * r1 / tdc1, "cores": 1,
                              "sample": f"first {CPU_SAMPLE_TOKENS} of {w.T} tokens, {r1} repetitions"}}


def config_of(w: W.Workload) -> dict:
    return {"workload": f"{w.name}: T={w.T} tokens ({w.src_ranks} virtual DP ranks x {w.T // w.src_ranks}), "
                        f"H={w.H}, E={w.E}, top_k={w.k}, R={w.R} virtual EP ranks, C={w.C}, "
                        f"fp8 e4m3 block-128 dispatch, bf16 combine",
            "T": w.T, "H": w.H, "E": w.E, "top_k": w.k, "R": w.R, "C": w.C,
            "dispatch_dtype": "fp8_e4m3_b128" if w.dtype else "bf16",
            "l2": "flushed before every call (write then read of 2x L2)", "parallelism": "replicas"}


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    import oracle as O
    w = W.WORKLOADS[WORKLOAD]
    x, lg, s = oracle_sample(w, w.T)
    to = ThreadedOracle(O, x, lg, s, w, host_cores())
    for _ in range(args.warmup):
        to.step()
    tdc, tstep = 0.0, 0.0
    for _ in range(args.steps):
        t = to.step()
        tdc += t["dispatch"] + t["combine"]
        tstep += t["step"]
    to.close()
    value = w.T * args.steps / tdc
    sample = (f"each step: the oracle's whole path on all {w.T} tokens (full E/H/k/C) on {to.threads} host threads "
              f"(its functions over disjoint token / expert ranges; counting serial); "
              f"value = tokens / (dispatch + combine time)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tstep / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": to.threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# multi-GPU plumbing: N independent replicas, max over ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------

def run_ours(args, rank: int, world: int, local: int):
    import torch
    import combine_router_top_gb300 as M
    from combine_router_top_gb300 import build as B

    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if not os.path.exists(M.LIB_PATH):
        B.build()
    M.lib()
    w = W.WORKLOADS[WORKLOAD]
    fp8 = w.dtype == W.DTYPE_FP8_E4M3_B128
    p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
    x_h, lg_h, s_h = W.make_x(w), W.make_logits(w), W.expert_scale(w)
    x = torch.from_numpy(x_h.view(np.int16)).to(dev)
    lg = torch.from_numpy(lg_h).to(dev)
    s = torch.from_numpy(s_h).to(dev)
    b = M.alloc_buffers(p, dev)
    out = torch.empty((w.T, w.H), dtype=torch.int16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones_like(flush_w)       # float32: the sum reduces in place, no widening copy
    stream = torch.cuda.current_stream()

    def flush():
        flush_w.fill_(1)
        flush_r.sum()

    calls = [
        ("route", lambda: M.moe_route(p, lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"],
                                      b["rank_counts"], b["dropped"], b["workspace"], stream)),
        ("dispatch", lambda: M.moe_dispatch(p, x, b["topk_idx"], b["slot"], b["recv"], b.get("recv_scale"),
                                            b["recv_src"], stream)),
        ("expert", lambda: M.moe_expert_synthetic(p, b["recv"], b.get("recv_scale"), b["counts"], s, b["y"], stream)),
        ("combine", lambda: M.moe_combine(p, b["y"], b["topk_idx"], b["topk_w"], b["slot"], out, stream)),
    ]
    for _ in range(max(args.warmup, 3)):
        for _, fn in calls:
            flush()
            fn()
    torch.cuda.synchronize()
    kept = w.T * w.k - int(b["dropped"].item())

    K = args.steps
    ev = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
          for n, _ in calls}
    sampler = clock_sampler(gpu_id_for_smi(torch, local))
    sampler.start()
    time.sleep(0.4)
    barrier(world, dev)
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(K):
        for n, fn in calls:
            flush()
            ev[n][i][0].record(stream)
            fn()
            ev[n][i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world, dev)
    sampler.stop()
    ms = {n: statistics.fmean(a.elapsed_time(z) for a, z in ev[n]) for n, _ in calls}

    # pipelined: the four calls back to back, L2 flushed before each step only;
    # programmatic dependent launch lets each kernel launch while the previous
    # one finishes
    evp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world, dev)
    torch.cuda.synchronize()
    for i in range(K):
        flush()
        evp[i][0].record(stream)
        for _, fn in calls:
            fn()
        evp[i][1].record(stream)
    torch.cuda.synchronize()
    pipe_ms = reduce_max(statistics.fmean(a.elapsed_time(z) for a, z in evp), world, dev)
    out_ref = out.clone()

    # route + dispatch through the one fused call (two launches for a decode
    # batch instead of three), cold per call and inside the pipelined step
    def fused():
        M.moe_route_dispatch(p, lg, x, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"],
                             b["rank_counts"], b["dropped"], b["recv"], b.get("recv_scale"), b["recv_src"],
                             b["workspace"], stream)
    for _ in range(3):
        flush()
        fused()
    evf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    evfp = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    barrier(world, dev)
    torch.cuda.synchronize()
    for i in range(K):
        flush()
        evf[i][0].record(stream)
        fused()
        evf[i][1].record(stream)
    for i in range(K):
        flush()
        evfp[i][0].record(stream)
        fused()
        calls[2][1]()
        calls[3][1]()
        evfp[i][1].record(stream)
    torch.cuda.synchronize()
    fused_ms = reduce_max(statistics.fmean(a.elapsed_time(z) for a, z in evf), world, dev)
    fused_pipe_ms = reduce_max(statistics.fmean(a.elapsed_time(z) for a, z in evfp), world, dev)
    assert torch.equal(out, out_ref), "fused route+dispatch changed the step's output"

    # expert + combine with per-row readiness (one cooperative kernel) against
    # the two calls chained by PDL; L2 flushed before each pair
    epoch = [0]

    def ready_pair():
        epoch[0] += 1
        M.moe_expert_combine(p, b["recv"], b.get("recv_scale"), b["counts"], s, b["y"], b["topk_idx"],
                             b["topk_w"], b["slot"], out, b["ready_flags"], epoch[0], stream)

    def separate_pair():
        calls[2][1]()
        calls[3][1]()
    for _ in range(3):
        flush()
        ready_pair()
    evr = {n: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
           for n in ("ready", "separate", "ready_step")}
    barrier(world, dev)
    torch.cuda.synchronize()
    for i in range(K):
        for n, fn in (("ready", ready_pair), ("separate", separate_pair)):
            flush()
            evr[n][i][0].record(stream)
            fn()
            evr[n][i][1].record(stream)
        flush()
        evr["ready_step"][i][0].record(stream)
        calls[0][1]()
        calls[1][1]()
        ready_pair()
        evr["ready_step"][i][1].record(stream)
    torch.cuda.synchronize()
    ready_ms = {n: reduce_max(statistics.fmean(a.elapsed_time(z) for a, z in v), world, dev) for n, v in evr.items()}
    assert torch.equal(out, out_ref), "expert+combine with readiness flags changed the step's output"
    assert M.moe_device_status() == M.MOE_OK
    step_ms = sum(ms.values())
    dc_ms = reduce_max(ms["dispatch"] + ms["combine"], world, dev)
    step_ms_max = reduce_max(step_ms, world, dev)
    comb_ms = reduce_max(ms["combine"], world, dev)

    # end to end through the C ABI with host buffers (moe_path_host): every
    # step copies x and logits in from pinned host memory, runs the four calls
    # and copies out back to pinned host memory, all issued by one call.
    # Serial: one stream, one buffer set. Pipelined (a serving loop): three
    # streams with a buffer set each, used in turn, so that one step's copy in,
    # another's kernels and a third's copy out run at the same time (each
    # stream keeps its own step's three phases in order).
    E2E_SETS = 3
    sets = []
    for _ in range(E2E_SETS):
        sets.append({"x": torch.empty_like(x), "lg": torch.empty_like(lg), "out": torch.empty_like(out),
                     "b": M.alloc_buffers(p, dev),
                     "xp": torch.from_numpy(x_h.view(np.int16)).pin_memory(),
                     "lp": torch.from_numpy(lg_h).pin_memory(),
                     "op": torch.empty((w.T, w.H), dtype=torch.int16).pin_memory()})
    e2e_streams = [torch.cuda.Stream(device=dev) for _ in range(E2E_SETS)]
    paths = [M.HostPath(p, z["xp"], z["lp"], s, z["x"], z["lg"], z["b"], z["out"], z["op"], e2e_streams[j])
             for j, z in enumerate(sets)]
    serial_path = M.HostPath(p, sets[0]["xp"], sets[0]["lp"], s, sets[0]["x"], sets[0]["lg"], sets[0]["b"],
                             sets[0]["out"], sets[0]["op"], stream)

    def e2e_run(n, pipelined):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world, dev)
        torch.cuda.synchronize()
        e0.record(stream)
        if not pipelined:
            for i in range(n):
                serial_path()
        else:
            for st_ in e2e_streams:
                st_.wait_stream(stream)
            for i in range(n):
                paths[i % E2E_SETS]()
            for st_ in e2e_streams:
                stream.wait_stream(st_)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    for pipelined in (False, True):
        e2e_run(3, pipelined)
    ke = max(5, min(K, 50))
    e2e_serial_ms = reduce_max(e2e_run(ke, False), world, dev)
    e2e_ms = reduce_max(e2e_run(ke, True), world, dev)
    for z in sets:
        assert torch.equal(z["out"], out), "end-to-end output differs from the device-resident run"
        assert torch.equal(z["op"].to(dev), out), "copied-out result differs from the device-resident run"

    peak, peak_kind = measured_peak()
    cb = bytes_combine(w, kept)
    per_call = {}
    for n, f in [("route", lambda: bytes_route(w)), ("dispatch", lambda: bytes_dispatch(w, kept)),
                 ("expert", lambda: bytes_expert(w, kept)), ("combine", lambda: cb)]:
        by = f()
        per_call[n] = {"us": 1e3 * ms[n], "algorithmic_bytes": by, "gbs": by / (ms[n] * 1e-3) / 1e9,
                       "frac": by / (ms[n] * 1e-3) / 1e9 / peak,
                       "frac_of_nominal": by / (ms[n] * 1e-3) / 1e9 / NOMINAL_HBM_GBS}
    line = None
    if rank == 0:
        achieved = cb / (comb_ms * 1e-3) / 1e9
        line = {
            "metric": METRIC, "value": world * w.T / (dc_ms * 1e-3), "unit": UNIT, "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": step_ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": "synthetic", "config": config_of(w),
            "roofline": {"kernel": "combine_kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs",
                         "traffic": ncu_traffic("combine", WORKLOAD),
                         "algorithmic_bytes": cb, "nominal_gbs": NOMINAL_HBM_GBS,
                         "frac_of_nominal": achieved / NOMINAL_HBM_GBS},
            "e2e": {"value": world * w.T / (e2e_ms * 1e-3), "unit": UNIT,
                    "h2d_bytes_per_step": x.numel() * 2 + lg.numel() * 4, "d2h_bytes_per_step": out.numel() * 2,
                    "ms_per_step": e2e_ms,
                    "what": "every step one moe_path_host call: H2D x+logits from pinned host, route, dispatch, "
                            "expert, combine, D2H out to pinned host; three streams with a buffer set each, used "
                            "in turn, so that copies of neighbouring steps overlap the compute",
                    "serial_ms_per_step": e2e_serial_ms,
                    "serial_value": world * w.T / (e2e_serial_ms * 1e-3)},
            "gpu_launches": 2 * KERNELS_PER_STEP * K,
            "clocks": sampler.summary(t0, t1),
            "calls": per_call,
            "path_tokens_per_s": world * w.T / (step_ms_max * 1e-3),
            "route_dispatch_combine_tokens_per_s":
                world * w.T / (reduce_max(ms["route"] + ms["dispatch"] + ms["combine"], world, dev) * 1e-3),
            "pipelined": {"ms_per_step": pipe_ms, "tokens_per_s": world * w.T / (pipe_ms * 1e-3),
                          "what": "route, dispatch, expert, combine back to back (programmatic dependent "
                                  "launch), L2 flushed before each step"},
            "fused_route_dispatch": {
                "us": 1e3 * fused_ms, "separate_us": 1e3 * (ms["route"] + ms["dispatch"]),
                "pipelined_ms_per_step": fused_pipe_ms, "pipelined_tokens_per_s": world * w.T / (fused_pipe_ms * 1e-3),
                "what": "moe_route_dispatch (top-k kernel, then one kernel that forms slots and dispatches), "
                        "L2 flushed before each call; pipelined: fused call, expert, combine"},
            "expert_combine_ready": {
                "us": 1e3 * ready_ms["ready"], "separate_us": 1e3 * ready_ms["separate"],
                "step_ms": ready_ms["ready_step"], "step_tokens_per_s": world * w.T / (ready_ms["ready_step"] * 1e-3),
                "what": "moe_expert_combine (one cooperative kernel, readiness per expert row) against "
                        "moe_expert_synthetic + moe_combine chained by PDL, L2 flushed before each pair; "
                        "step: route, dispatch, moe_expert_combine"},
        }
    return line, dev


ALL_CONFIGS = ["tiny", "v2lite", "mixtral_skew", "dsv3_fp8", "dbo"]


def run_all_configs(args, dev, reps: int = 100) -> dict:
    """Route, dispatch, expert stand-in and combine of every configuration,
    each call isolated (L2 flushed before it) and event-timed on its stream,
    the mean of `reps` calls (one event interval is quantised to a fraction of
    a microsecond, so a median of few calls is off by up to half a step);
    the dual-batch configuration is timed per micro-batch (half its tokens).
    Parity of each configuration is the GPU test suite's, not this run's."""
    import torch
    import combine_router_top_gb300 as M
    peak, peak_kind = measured_peak()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones_like(flush_w)
    stream = torch.cuda.current_stream()
    rows = []
    for name in ALL_CONFIGS:
        if args.only is not None and name != args.only:
            continue
        w = W.WORKLOADS[name]
        if name == "dbo":
            w = w.with_(T=w.T // 2)
        p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
        x = torch.from_numpy(x_of(w).view(np.int16)).to(dev)
        lg = torch.from_numpy(W.make_logits(w)).to(dev)
        s = torch.from_numpy(W.expert_scale(w)).to(dev)
        b = M.alloc_buffers(p, dev)
        out = torch.empty((w.T, w.H), dtype=torch.int16, device=dev)
        calls = [
            ("route", lambda: M.moe_route(p, lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"],
                                          b["rank_counts"], b["dropped"], b["workspace"], stream)),
            ("dispatch", lambda: M.moe_dispatch(p, x, b["topk_idx"], b["slot"], b["recv"], b.get("recv_scale"),
                                                b["recv_src"], stream)),
            ("expert", lambda: M.moe_expert_synthetic(p, b["recv"], b.get("recv_scale"), b["counts"], s, b["y"],
                                                      stream)),
            ("combine", lambda: M.moe_combine(p, b["y"], b["topk_idx"], b["topk_w"], b["slot"], out, stream)),
        ]
        times = {n: [] for n, _ in calls}
        for i in range(3 + reps):
            for n, fn in calls:
                flush_w.fill_(1)
                flush_r.sum()
                a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                z.record(stream)
                if i >= 3:
                    times[n].append((a, z))
        torch.cuda.synchronize()
        kept = w.T * w.k - int(b["dropped"].item())
        by = {"route": bytes_route(w), "dispatch": bytes_dispatch(w, kept), "expert": bytes_expert(w, kept),
              "combine": bytes_combine(w, kept)}
        us = {n: 1e3 * statistics.fmean(a.elapsed_time(z) for a, z in v) for n, v in times.items()}
        row = {"workload": name if name != "dbo" else "dbo (one micro-batch)", "T": w.T, "H": w.H, "E": w.E,
               "top_k": w.k, "R": w.R, "C": w.C,
               "dispatch_dtype": "fp8_e4m3_b128" if w.dtype == W.DTYPE_FP8_E4M3_B128 else "bf16",
               "kept_pairs": kept, "dropped": w.T * w.k - kept,
               "dispatch_combine_tokens_per_s": w.T / ((us["dispatch"] + us["combine"]) * 1e-6)}
        for n in us:
            row[n] = {"us": us[n], "algorithmic_bytes": by[n], "gbs": by[n] / (us[n] * 1e-6) / 1e9,
                      "frac": by[n] / (us[n] * 1e-6) / 1e9 / peak}
        rows.append(row)
        del b, x, out
        torch.cuda.empty_cache()
    return {"peak_gbs": peak, "peak_source": f"{peak_kind} hbm_gbs", "reps": reps, "statistic": "mean",
            "l2": "flushed before every call", "configs": rows}


def run_dbo(args, dev) -> dict:
    """Dual-batch-overlap step on the 8192-token prefill workload."""
    import torch
    import combine_router_top_gb300 as M
    w = W.WORKLOADS["dbo"]
    T0, T1 = w.T // 2, w.T - w.T // 2
    pf = M.problem(w.T, w.H, w.E, w.k, w.R, w.C)
    x = torch.from_numpy(x_of(w).view(np.int16)).to(dev)
    lg = torch.from_numpy(W.make_logits(w)).to(dev)
    s = torch.from_numpy(W.expert_scale(w)).to(dev)
    bufs = [M.alloc_buffers(M.problem(T1, w.H, w.E, w.k, w.R, w.C), dev) for _ in range(2)]
    out = torch.empty((w.T, w.H), dtype=torch.int16, device=dev)
    comp, comm = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ctx = M.dbo_create()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    flush_r = torch.ones_like(flush_w)       # float32: the sum reduces in place, no widening copy
    res = {"overlap_fraction": [], "step_ms": [], "dispatch_ub1_ms": [], "combine_ub0_ms": [], "overlap_ms": [],
           "serial_ms": []}
    reps = 10
    with torch.cuda.stream(comp):
        for i in range(3 + reps):
            flush_w.fill_(1)
            flush_r.sum()
            M.dbo_step(ctx, pf, x, lg, s, bufs, out, comp, comm, record_timing=True)
            t = M.dbo_read_timing(ctx)
            if i >= 3:
                for key in ["overlap_fraction", "step_ms", "dispatch_ub1_ms", "combine_ub0_ms", "overlap_ms"]:
                    res[key].append(t[key])
        # the same work on one stream, for comparison
        for i in range(3 + reps):
            flush_w.fill_(1)
            flush_r.sum()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(comp)
            for (lo, hi), bb in zip([(0, T0), (T0, w.T)], bufs):
                p = M.problem(hi - lo, w.H, w.E, w.k, w.R, w.C)
                M.run_path(p, x[lo:hi], lg[lo:hi], s, bb, out[lo:hi], comp)
            z.record(comp)
            z.synchronize()
            if i >= 3:
                res["serial_ms"].append(a.elapsed_time(z))
    ctx.close()
    med = {k: statistics.median(v) for k, v in res.items()}
    kept1 = T1 * w.k - int(bufs[1]["dropped"].item())
    kept0 = T0 * w.k - int(bufs[0]["dropped"].item())
    wd = w.with_(T=T1)
    wc = w.with_(T=T0)
    return {"workload": f"dbo: T={w.T} split {T0}/{T1}, H={w.H}, E={w.E}, top_k={w.k}, R={w.R}, C={w.C}, bf16",
            "overlap_fraction": med["overlap_fraction"], "dbo_step_ms": med["step_ms"],
            "single_stream_ms": med["serial_ms"], "dispatch_ub1_ms": med["dispatch_ub1_ms"],
            "combine_ub0_ms": med["combine_ub0_ms"],
            "overlapped_pair_bytes": bytes_dispatch(wd, kept1) + bytes_combine(wc, kept0),
            # both kernels' algorithmic bytes over the window from the first's start to the last's end
            "window_gbs": (bytes_dispatch(wd, kept1) + bytes_combine(wc, kept0))
                          / ((med["dispatch_ub1_ms"] + med["combine_ub0_ms"] - med["overlap_ms"]) * 1e-3) / 1e9,
            "reps": reps, "l2": "flushed before every step"}


def run_dbo_layers(args, dev, layers: int = 4, busy_fmas: int = 256) -> dict:
    """The [DBO] layer schedule on the 8192-token workload: two streams eager,
    two streams replayed from a CUDA graph, and the same work on one stream."""
    import torch
    import combine_router_top_gb300 as M
    w = W.WORKLOADS["dbo"]
    T1 = w.T - w.T // 2
    pf = M.problem(w.T, w.H, w.E, w.k, w.R, w.C)
    x = torch.from_numpy(x_of(w).view(np.int16)).to(dev)
    lg = torch.from_numpy(np.stack([W.make_logits(w.with_(seed=w.seed + 31 * l)) for l in range(layers)])).to(dev)
    s = torch.from_numpy(W.expert_scale(w)).to(dev)
    bufs = [M.alloc_buffers(M.problem(T1, w.H, w.E, w.k, w.R, w.C), dev) for _ in range(2)]
    h, shared, out = (torch.empty((w.T, w.H), dtype=torch.int16, device=dev) for _ in range(3))
    a = M.dbo_layers_args(pf, layers, x, lg, s, bufs, h, shared, out, 0.75, 1.5, busy_fmas)
    comp, comm = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ctx = M.dbo_create()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    fw = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=dev)
    fr = torch.ones_like(fw)

    def timed(launch, reps=8):
        ts = []
        with torch.cuda.stream(comp):
            for i in range(2 + reps):
                fw.fill_(1)
                fr.sum()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(comp)
                launch()
                e1.record(comp)
                e1.synchronize()
                if i >= 2:
                    ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    comp.wait_stream(torch.cuda.current_stream())
    two = timed(lambda: M.dbo_layers(ctx, a, comp, comm))
    one = timed(lambda: M.dbo_layers(ctx, a, comp, comp))
    M.dbo_layers_capture(ctx, a, comp, comm)
    graph = timed(lambda: M.dbo_graph_launch(ctx, comp))
    ctx.close()
    return {"workload": f"dbo layers: {layers} layers, T={w.T} split {w.T // 2}/{T1}, H={w.H}, E={w.E}, "
                        f"top_k={w.k}, C={w.C}, bf16; A0/S stand-ins with {busy_fmas} busy FMAs per 8 elements",
            "ms_per_layer_two_streams": two / layers, "ms_per_layer_graph": graph / layers,
            "ms_per_layer_one_stream": one / layers, "speedup_vs_one_stream": one / two,
            "l2": "flushed before every run of the layers"}


def run_dbo_layers_gemm(args, dev, layers: int = 2, reps: int = 5) -> dict:
    """The [DBO] layer schedule on the 8192-token workload with the grouped bf16 GEMM as the MLP (random
    bf16 weights, 26 GB, shared by the layers; A0 and S stand-ins without busy work): two streams against
    the same work on one stream, with the GEMM on every SM or capped to leave SMs to the comm stream.
    hidden_comm_fraction = (one stream - two streams) / (the dispatch and combine kernels alone)."""
    import torch
    import combine_router_top_gb300 as M
    w = W.WORKLOADS["dbo"]
    T1 = w.T - w.T // 2
    pf = M.problem(w.T, w.H, w.E, w.k, w.R, w.C)
    x = torch.from_numpy(x_of(w).view(np.int16)).to(dev)
    lg = torch.from_numpy(np.stack([W.make_logits(w.with_(seed=w.seed + 31 * l)) for l in range(layers)])).to(dev)
    s = torch.from_numpy(W.expert_scale(w)).to(dev)
    wb = W.make_weights_bf16_device(w, dev)
    bufs = [M.alloc_buffers(M.problem(T1, w.H, w.E, w.k, w.R, w.C), dev) for _ in range(2)]
    h, shared, out = (torch.empty((w.T, w.H), dtype=torch.int16, device=dev) for _ in range(3))
    comp, comm = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ctx = M.dbo_create()

    def timed(launch):
        ts = []
        with torch.cuda.stream(comp):
            for i in range(2 + reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(comp)
                launch()
                e1.record(comp)
                e1.synchronize()
                if i >= 2:
                    ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    comp.wait_stream(torch.cuda.current_stream())
    res = {}
    for cap in [0, 128]:
        a = M.dbo_layers_args(pf, layers, x, lg, s, bufs, h, shared, out, 0.75, 1.5, 0, expert_w=wb,
                              mlp_max_blocks=cap)
        res[cap] = (timed(lambda: M.dbo_layers(ctx, a, comp, comm)), timed(lambda: M.dbo_layers(ctx, a, comp, comp)))
    a = M.dbo_layers_args(pf, layers, x, lg, s, bufs, h, shared, out, 0.75, 1.5, 0, expert_w=wb)
    M.dbo_layers_capture(ctx, a, comp, comm)
    graph = timed(lambda: M.dbo_graph_launch(ctx, comp))
    ctx.close()
    # the comm kernels alone, on the buffers the last run left (per layer: D and C of both micro-batches)
    pu = [M.problem(w.T // 2, w.H, w.E, w.k, w.R, w.C), M.problem(T1, w.H, w.E, w.k, w.R, w.C)]
    rows0 = [0, w.T // 2]

    def comm_only():
        for _ in range(layers):
            for u in range(2):
                b = bufs[u]
                M.moe_dispatch(pu[u], h[rows0[u]:], b["topk_idx"], b["slot"], b["recv"], None, b["recv_src"], comp)
                M.moe_combine(pu[u], b["y"], b["topk_idx"], b["topk_w"], b["slot"], out[rows0[u]:], comp)
    comm_ms = timed(comm_only)
    best_cap = min(res, key=lambda c: res[c][0])
    two, one = res[best_cap]
    return {"workload": f"dbo layers, grouped bf16 GEMM as the MLP: {layers} layers, T={w.T} split "
                        f"{w.T // 2}/{T1}, H={w.H}, E={w.E}, top_k={w.k}, C={w.C}, bf16 rows and weights",
            "ms_per_layer_two_streams": two / layers, "ms_per_layer_one_stream": one / layers,
            "ms_per_layer_graph": graph / layers, "speedup_vs_one_stream": one / two,
            "mlp_max_blocks": best_cap,
            "by_mlp_cap": {str(c): {"two_streams_ms_per_layer": t / layers, "one_stream_ms_per_layer": o / layers}
                           for c, (t, o) in res.items()},
            "comm_kernels_ms_per_layer": comm_ms / layers,
            "hidden_comm_fraction": max(0.0, (one - two) / comm_ms) if comm_ms > 0 else None,
            "l2": "not flushed: 26 GB of weights stream through every layer"}


def run_gemm(args, dev, reps: int = 10, experts: int = 0) -> dict:
    """The grouped fp8 GEMM on the tensor cores, fed by route + dispatch, at the
    DeepSeek-V3 decode shape (weight-streaming, bound by HBM) and at an
    8192-token prefill shape (bound by the tensor cores); plus the decode step
    with the GEMM in place of the synthetic expert. Weights (13.2 GB) and
    activations far exceed L2, so no flush is needed between calls."""
    import torch
    import combine_router_top_gb300 as M
    hbm, hbm_kind = measured_peak()
    fp8_burst, fp8_sust, fp8_kind = measured_fp8_peak()
    st = torch.cuda.current_stream()
    out = {}
    wq = ws = None
    cases = [("decode", W.WORKLOADS["dsv3_fp8"]), ("prefill", W.WORKLOADS["dbo"].with_(dtype=1))]
    if experts:                                   # a smaller case with the same shapes per expert (profiling)
        cases = [(n, w.with_(E=experts, R=min(w.R, experts))) for n, w in cases]
    for name, w in cases:
        p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, w.dtype)
        b = M.alloc_buffers(p, dev)
        x = torch.from_numpy(x_of(w).view(np.int16)).to(dev)
        lg = torch.from_numpy(W.make_logits(w)).to(dev)
        M.moe_route(p, lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"], b["rank_counts"],
                    b["dropped"], b["workspace"], st)
        M.moe_dispatch(p, x, b["topk_idx"], b["slot"], b["recv"], b["recv_scale"], b["recv_src"], st)
        if wq is None:
            wq, ws = W.make_weights_device(w, dev)
        y = torch.empty((w.E, w.C, w.H), dtype=torch.int16, device=dev)

        def gemm():
            M.moe_expert_gemm_fp8(p, b["recv"], b["recv_scale"], b["counts"], wq, ws, y, st)
        for _ in range(3):
            gemm()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a, z in ev:
            a.record(st)
            gemm()
            z.record(st)
        torch.cuda.synchronize()
        ms = statistics.fmean(a.elapsed_time(z) for a, z in ev)
        counts = b["counts"].cpu().numpy()
        kept = int(np.minimum(counts, w.C).sum())
        active = int((counts > 0).sum())
        nb = w.H // 128
        algo_bytes = active * (w.H * w.H + nb * nb * 4) + kept * (w.H + nb * 4) + kept * w.H * 2 + w.E * 4
        flops = 2.0 * kept * w.H * w.H
        gbs, tfs = algo_bytes / (ms * 1e-3) / 1e9, flops / (ms * 1e-3) / 1e12
        r = {"workload": f"{name}: T={w.T}, H={w.H}, E={w.E}, top_k={w.k}, C={w.C}, kept rows {kept}, "
                         f"{active} experts with rows, fp8 e4m3 in, bf16 out",
             "ms": ms, "algorithmic_bytes": algo_bytes, "flops": flops, "GB/s": gbs, "TFLOP/s": tfs,
             "reps": reps}
        if name == "decode":
            # the 32-expert capture, scaled to this launch by the ratio of algorithmic bytes
            # (weights dominate both; every kept row of the 32-expert decode case is full: 32 x 128)
            t32 = ncu_traffic("gemm", "dsv3_fp8_E32")
            algo32 = 32 * (w.H * w.H + nb * nb * 4) + 32 * 128 * (w.H + nb * 4) + 32 * 128 * w.H * 2 + 32 * 4
            traffic = None if t32 is None else int(t32 * algo_bytes / algo32)
            r["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                             "peak_source": f"{hbm_kind} hbm_gbs", "traffic": traffic}
            s = torch.from_numpy(W.expert_scale(w)).to(dev)
            outp = torch.empty((w.T, w.H), dtype=torch.int16, device=dev)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for i in range(reps + 3):
                if i >= 3:
                    evs[i - 3][0].record(st)
                M.moe_route(p, lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"],
                            b["rank_counts"], b["dropped"], b["workspace"], st)
                M.moe_dispatch(p, x, b["topk_idx"], b["slot"], b["recv"], b["recv_scale"], b["recv_src"], st)
                gemm()
                M.moe_combine(p, y, b["topk_idx"], b["topk_w"], b["slot"], outp, st)
                if i >= 3:
                    evs[i - 3][1].record(st)
            torch.cuda.synchronize()
            step_ms = statistics.fmean(a.elapsed_time(z) for a, z in evs)
            r["step_with_gemm"] = {"ms_per_step": step_ms, "tokens_per_s": w.T / (step_ms * 1e-3),
                                   "what": "route, dispatch, grouped GEMM, combine back to back (PDL)"}
        else:
            r["roofline"] = {"bound": "tensor", "achieved": tfs, "peak": fp8_burst, "unit": "TFLOP/s",
                             "frac": tfs / fp8_burst, "frac_of_sustained": tfs / fp8_sust,
                             "peak_source": f"{fp8_kind} (burst; sustained {fp8_sust:.0f})",
                             "traffic": None}
        r["device_status"] = M.moe_device_status()
        out[name] = r
        del b, y
    del wq, ws
    torch.cuda.empty_cache()

    # bf16 rows, bf16 weights (tcgen05 kind::f16): DeepSeek-V2-Lite decode, the
    # 8192-token prefill shape (26 GB of weights at H 7168, 256 experts) and the
    # skewed Mixtral-shaped prefill (8 experts, about 1024 rows each on average:
    # the 256-row tiles; 268 MB of weights and 67 MB of rows, more than L2);
    # the bound is whichever of HBM and the bf16 tensor peak takes longer
    bf16_burst, bf16_sust = fp8_burst / FP8_PER_BF16, fp8_sust / FP8_PER_BF16
    cases = [("decode_bf16", W.WORKLOADS["v2lite"]), ("prefill_bf16", W.WORKLOADS["dbo"]),
             ("prefill_bf16_mixtral", W.WORKLOADS["mixtral_skew"])]
    if experts:
        cases = [(n, w.with_(E=experts, R=min(w.R, experts))) for n, w in cases]
    for name, w in cases:
        p = M.problem(w.T, w.H, w.E, w.k, w.R, w.C, M.MOE_DTYPE_BF16)
        b = M.alloc_buffers(p, dev)
        x = torch.from_numpy(x_of(w).view(np.int16)).to(dev)
        lg = torch.from_numpy(W.make_logits(w)).to(dev)
        M.moe_route(p, lg, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"], b["slot"], b["rank_counts"],
                    b["dropped"], b["workspace"], st)
        M.moe_dispatch(p, x, b["topk_idx"], b["slot"], b["recv"], None, b["recv_src"], st)
        wb = W.make_weights_bf16_device(w, dev)
        y = torch.empty((w.E, w.C, w.H), dtype=torch.int16, device=dev)

        def gemm_bf16():
            M.moe_expert_gemm_bf16(p, b["recv"], b["counts"], wb, y, st)
        for _ in range(3):
            gemm_bf16()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for a, z in ev:
            a.record(st)
            gemm_bf16()
            z.record(st)
        torch.cuda.synchronize()
        ms = statistics.fmean(a.elapsed_time(z) for a, z in ev)
        counts = b["counts"].cpu().numpy()
        kept = int(np.minimum(counts, w.C).sum())
        active = int((counts > 0).sum())
        algo_bytes = active * w.H * w.H * 2 + kept * w.H * 2 * 2 + w.E * 4
        flops = 2.0 * kept * w.H * w.H
        gbs, tfs = algo_bytes / (ms * 1e-3) / 1e9, flops / (ms * 1e-3) / 1e12
        hbm_bound = algo_bytes / (hbm * 1e9) >= flops / (bf16_burst * 1e12)
        r = {"workload": f"{name}: T={w.T}, H={w.H}, E={w.E}, top_k={w.k}, C={w.C}, kept rows {kept}, "
                         f"{active} experts with rows, bf16 in, bf16 out",
             "ms": ms, "algorithmic_bytes": algo_bytes, "flops": flops, "GB/s": gbs, "TFLOP/s": tfs, "reps": reps,
             "roofline": ({"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                           "peak_source": f"{hbm_kind} hbm_gbs", "tensor_frac": tfs / bf16_burst, "traffic": None}
                          if hbm_bound else
                          {"bound": "tensor", "achieved": tfs, "peak": bf16_burst, "unit": "TFLOP/s",
                           "frac": tfs / bf16_burst, "frac_of_sustained": tfs / bf16_sust,
                           "peak_source": f"{fp8_kind.replace(' x 2', '')} bf16 (burst)", "hbm_frac": gbs / hbm,
                           "traffic": None}),
             "device_status": M.moe_device_status()}
        out[name] = r
        del b, y, wb
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-dbo", action="store_true")
    ap.add_argument("--no-gemm", action="store_true")
    ap.add_argument("--gemm-only", action="store_true", help="only the grouped GEMM measurement")
    ap.add_argument("--gemm-experts", type=int, default=0, help="with --gemm-only: E experts (profiling case)")
    ap.add_argument("--dbo-only", action="store_true", help="only the dual-batch-overlap measurements")
    ap.add_argument("--all-configs", action="store_true",
                    help="only the per-configuration timings of route, dispatch, expert and combine")
    ap.add_argument("--only", choices=ALL_CONFIGS, default=None,
                    help="with --all-configs: this configuration alone")
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.all_configs:
        import torch
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        from combine_router_top_gb300 import build as B
        import combine_router_top_gb300 as M
        if not os.path.exists(M.LIB_PATH):
            B.build()
        print(json.dumps({"all_configs": run_all_configs(args, dev)}), flush=True)
        return
    if args.gemm_only:
        import torch
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        print(json.dumps({"expert_gemm": run_gemm(args, dev, experts=args.gemm_experts)}), flush=True)
        return
    if args.dbo_only:
        import torch
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        print(json.dumps({"dbo": run_dbo(args, dev), "dbo_layers": run_dbo_layers(args, dev),
                          "dbo_layers_gemm": run_dbo_layers_gemm(args, dev)}), flush=True)
        return
    line, dev = run_ours(args, rank, world, local)
    if rank == 0:
        if world == 1 and not args.no_dbo:
            line["dbo"] = run_dbo(args, dev)
            line["dbo_layers"] = run_dbo_layers(args, dev)
            if not args.no_gemm:
                line["dbo_layers_gemm"] = run_dbo_layers_gemm(args, dev)
        if world == 1 and not args.no_gemm:
            line["expert_gemm"] = run_gemm(args, dev)
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(W.WORKLOADS[WORKLOAD])
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
