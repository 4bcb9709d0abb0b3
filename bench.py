#!/usr/bin/env python3
"""Benchmark of the partial denoising step on B300.

One step = one pass of the whole hot path over one batch: saliency select,
KV scatter, partial attention, the column-sum pass, confidence over the logit
rows, longest stable prefix.

Default workload (``--workload loop_b4_2k_128``): the block-wise decoding loop
of batch 4, L = 2048 (1024 prompt + 1024 generated positions in 32 blocks of
32, four partial steps per block, 128 steps), 32 heads x 128, hidden 4096,
vocabulary 126464, bf16.  Every step selects over the generated rows (over
all 2048 rows on the first step of each block), scatters the fresh K/V rows
of its active positions into the cache the earlier steps wrote, attends from
them and takes the column sums, scores their logit rows and commits the
longest stable prefix, advancing ``start``.  State (cache, score, start)
carries from step to step on the device; the timed region replays a CUDA
graph of K consecutive steps of the loop (``--steps K``, default the whole
loop; past step 128 the loop restarts from a fresh score and start).

The other workloads are single step shapes (``step_1k``, ``batch8_2k`` with
an active fraction and pattern, ``long_4k`` with a locked fraction,
``long_4k_schedule``, ``loop_b4_2k``) and print the same line for their shape.

Metric: active query tokens per second (sum over batch rows of the active
count / step time); the line also carries the step latency, a per-entry-point
breakdown, the roofline of the dominant entry point, the clocks seen during
the timed region, the end-to-end figure (host buffers, copies inside the
timed region) and the float64 oracle timed on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--frac F] [--pattern random|cluster] [--locked F]
Under torchrun (N > 1) every rank runs an independent replica (weak scaling);
the timed region is bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "partial-step latency (µs) & active query tokens/s; % of B300 HBM/TC roofline"
UNIT = "active query tokens/s"
CSRC = os.path.join(ROOT, "partial_attention_saliency_b300", "csrc")

ENTRY_ORDER = ["dllm_saliency_select", "dllm_kv_scatter", "dllm_partial_attention",
               "dllm_attention_colsum", "dllm_confidence", "dllm_stable_prefix"]
# with --surelock: the lock criterion between consecutive steps' logits takes
# the confidence's place (one call reads the current logits once for both),
# and the adaptive prefix threshold follows the step
SURELOCK_ORDER = ["dllm_saliency_select", "dllm_kv_scatter", "dllm_partial_attention",
                  "dllm_attention_colsum", "dllm_lock_criterion_conf", "dllm_stable_prefix",
                  "dllm_adaptive_prefix"]
LOCK_EPS, LOCK_GATE_Q = 1e-3, 0.5     # KL threshold, uncertainty percentile gate
ADAPT_LO, ADAPT_HI = 0.25, 0.5        # fraction of the active length the prefix covers
KERNELS = {  # kernels each entry point launches, and the source they come from
    "dllm_saliency_select": (["cos_rows_kernel", "compact_kernel"], "select.cu"),
    "dllm_kv_scatter": (["kv_scatter_kernel"], "kv_scatter.cu"),
    "dllm_partial_attention": (["attn_fwd_tc_kernel", "attn_split_merge_kernel"],
                               "attention_tc.cu"),
    "dllm_attention_colsum": (["attn_colsum_stream_kernel", "attn_colsum_tc_kernel"],
                              "attention_tc.cu"),
    "dllm_confidence": (["conf_stream_kernel", "conf_merge_kernel"], "confidence.cu"),
    "dllm_stable_prefix": (["stable_prefix_kernel"], "stable_prefix.cu"),
    "dllm_lock_criterion": (["lock_partial_persistent_kernel", "lock_partial_kernel",
                             "lock_merge_kernel", "lock_gate_kernel"], "lock.cu"),
    "dllm_lock_criterion_conf": (["lock_partial_persistent_kernel", "lock_partial_kernel",
                                  "lock_merge_kernel", "lock_gate_kernel"], "lock.cu"),
    "dllm_adaptive_prefix": (["adaptive_prefix_kernel"], "lock.cu"),
    "dllm_approx_attention_update": (["approx_update_tc_kernel"], "approx_update_tc.cu"),
    "dllm_attn_scores": (["attn_scores_kernel"], "sampler.cu"),
    "dllm_attn_sampler_select": (["attn_sampler_select_kernel"], "sampler.cu"),
    "dllm_slowfast_observe_device": (["slowfast_observe_kernel"], "slowfast_device.cu"),
    "dllm_slowfast_select": (["slowfast_select_kernel"], "slowfast_device.cu"),
}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of an
# entry point's main kernel, from one ncu capture of the named workload.  The
# figure is reported only while the kernel's source file still has the digest
# it was captured with; otherwise traffic is null.
TRAFFIC = {
    # (workload, entry point): {"bytes": ..., "src_sha": first 16 hex of sha256}
    ("step_1k", "dllm_confidence"): {"bytes": 133703936, "src_sha": "8852f06b7bb1aac3"},
    ("batch8_2k_f50_random", "dllm_partial_attention"): {"bytes": 386810368,
                                                          "src_sha": "e7e48f69adabdd83"},
    ("batch8_2k_f05_random", "dllm_partial_attention"): {"bytes": 284102912,
                                                          "src_sha": "e7e48f69adabdd83"},
    # steady-state loop steps, single-pass capture without cache flush (the
    # mean of a generated-rows-window step and a whole-sequence step)
    ("loop_b4_2k_128", "dllm_partial_attention"): {"bytes": 143480000,
                                                   "src_sha": "f7092d2beca757ee"},
    # the calls around the loop's step 1, single-kernel captures
    ("around_b4_2k", "dllm_approx_attention_update"): {"bytes": 160583680,
                                                       "src_sha": "d56bc4837a78c2c7"},
    ("around_b4_2k", "dllm_lock_criterion"): {"bytes": 254773760, "src_sha": "78d1876c6127b808"},
    ("around_b4_2k", "dllm_attn_sampler_select"): {"bytes": 52480, "src_sha": "dccded94e04e80a9"},
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: the whole 128-step loop, or about one second "
                         "of steps of a single-step workload)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload",
                    choices=["loop_b4_2k_128", "around_b4_2k", "step_1k", "batch8_2k", "long_4k",
                             "long_4k_schedule", "loop_b4_2k"],
                    default="loop_b4_2k_128")
    ap.add_argument("--frac", type=float, default=0.25,
                    help="batch8_2k: active fraction of the 2048 positions")
    ap.add_argument("--pattern", choices=["random", "cluster"], default="random")
    ap.add_argument("--locked", type=float, default=0.0,
                    help="long_4k: locked fraction (0 = first step of the schedule)")
    ap.add_argument("--surelock", action="store_true",
                    help="long_4k, long_4k_schedule: add the lock criterion between this and "
                         "the previous step's logits of the active rows and the adaptive prefix")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="how long the timed region is repeated (median reported; at least 5 "
                         "repetitions)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="approximate CPU time spent on the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def src_sha(fname: str) -> str:
    with open(os.path.join(CSRC, fname), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


# ----------------------------------------------------------------------------- clocks

class _NvmlC:
    """The few NVML calls the sampler needs, through the driver's own
    libnvidia-ml (ctypes), for when the Python module is not installed."""

    NVML_CLOCK_SM = 1

    def __init__(self, uuid: str):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByUUID failed")
        self._reasons = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def max_sm_mhz(self) -> int:
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, self.ct.byref(v))
        return int(v.value)

    def sample(self):
        mhz = self.ct.c_uint()
        rs = self.ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, self.ct.byref(mhz)) != 0:
            return None
        self._reasons(self.h, self.ct.byref(rs))
        return int(mhz.value), int(rs.value)


class ClockSampler:
    """Samples the SM clock and the clock-event reasons while running: NVML
    through the Python module when present, else through libnvidia-ml
    directly, else an ``nvidia-smi -lms`` child."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index: int, period_s: float = 0.005):
        self.samples = []
        self.period = period_s
        self.max_mhz = None
        self.mode = None
        self.err = None
        props = torch.cuda.get_device_properties(device_index)
        self.uuid = "GPU-" + str(props.uuid)
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        self._read = None
        try:
            import pynvml
            pynvml.nvmlInit()
            h = pynvml.nvmlDeviceGetHandleByUUID(self.uuid.encode())
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
            self._read = lambda: (pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM),
                                  int(pynvml.nvmlDeviceGetCurrentClocksEventReasons(h)))
            self.mode = "nvml"
        except Exception as e:  # noqa: BLE001
            self.err = repr(e)[:160]
            try:
                nv = _NvmlC(self.uuid)
                self.max_mhz = nv.max_sm_mhz()
                self._read = nv.sample
                self.mode = "nvml-ctypes"
            except Exception as e2:  # noqa: BLE001
                self.err += "; " + repr(e2)[:160]
                if shutil.which("nvidia-smi"):
                    self.mode = "nvidia-smi"

    def _run_nvml(self):
        while not self._stop.is_set():
            try:
                r = self._read()
                if r is not None:
                    self.samples.append(r)
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.period)

    def start(self):
        if self._read is not None:
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        elif self.mode == "nvidia-smi":
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.uuid,
                 "--query-gpu=timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)  # the child is sampling before the timed region begins
        self.t0 = time.time()

    def stop(self):
        self.t1 = time.time()
        if self._t is not None:
            self._stop.set()
            self._t.join()
        if self._proc is not None:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
                out, _ = self._proc.communicate()
            from datetime import datetime
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) != 4:
                    continue
                try:
                    ts = datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    mhz, mx = float(parts[1]), float(parts[2])
                    reasons = int(parts[3], 16)
                except ValueError:
                    continue
                self.max_mhz = mx
                if self.t0 <= ts <= self.t1:  # samples taken inside the timed region only
                    self.samples.append((mhz, reasons))

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": self.mode or "unavailable", "error": self.err}
        mhz = [m for m, _ in self.samples]
        seen = 0
        for _, r in self.samples:
            seen |= int(r)
        names = [n for bit, n in self.REASONS.items() if seen & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(mhz), "source": self.mode}


def time_regions(region, stream, est_ms: float, warm=None, min_seconds: float = 1.0,
                 min_reps: int = 5, max_reps: int = 2000):
    """Device time of a timed region, repeated: ``warm()`` once untimed (the
    graph's upload and first launch), then R times ``region()`` (which
    launches graph replays on ``stream``) bracketed by events on that stream,
    with a synchronize on both sides of each.  R is chosen so that the
    regions take about ``min_seconds`` (at least ``min_reps``).  Returns the R
    times in ms."""
    if warm is not None:
        warm()
    torch.cuda.synchronize()
    reps = max(min_reps, min(max_reps, math.ceil(min_seconds * 1e3 / max(est_ms, 1e-3))))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    out = []
    for _ in range(reps):
        a.record(stream)
        region()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b))
    return out


def read_ceiling(sizes: dict, device, reps: int = 5) -> dict:
    """Reference time of one read-bound launch per byte count: dllm_read_stream
    (one persistent CTA per SM streaming the bytes into shared memory with
    cp.async.bulk, nothing else) timed like the calls, with an external event
    on each side of every launch in a replayed CUDA graph.  Each launch reads
    its own region of a buffer three times the largest size, so consecutive
    launches find nothing in L2.  Returns {name: median us}."""
    import partial_attention_saliency_b300 as dl
    if not sizes:
        return {}
    nb = {n: max(16, int(v) // 16 * 16) for n, v in sizes.items()}
    span = max(nb.values())
    buf = torch.ones((3 * span + 4096,), dtype=torch.uint8, device=device)
    sink = torch.zeros((1,), dtype=torch.int32, device=device)
    st = torch.zeros((1,), dtype=torch.int32, device=device)
    names = list(nb)
    ev = [[(torch.cuda.Event(enable_timing=True, external=True),
            torch.cuda.Event(enable_timing=True, external=True)) for _ in names]
          for _ in range(reps)]
    cap = torch.cuda.Stream(device)
    g = torch.cuda.CUDAGraph()
    k = 0
    with torch.cuda.graph(g, stream=cap):
        for r in range(reps):
            for i, n in enumerate(names):
                off = (k % 3) * span
                k += 1
                ev[r][i][0].record()
                dl.dllm_read_stream(buf[off:off + nb[n]], nb[n], sink, dev_status=st)
                ev[r][i][1].record()
    g.replay()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    if int(st[0]) != 0:
        raise RuntimeError("dllm_read_stream: a pipeline wait ran out")
    out = {n: statistics.median(ev[r][i][0].elapsed_time(ev[r][i][1]) * 1e3
                                for r in range(reps)) for i, n in enumerate(names)}
    del buf
    return out


# ----------------------------------------------------------------------------- workloads

@dataclasses.dataclass
class Workload:
    """One benchmarked step shape.

    ``conf``: how the confidence pass reads its logit rows -- "window" (one
    logit row per window position, row r -> position win_start + r), "gather"
    (a full [B, L, V] logits buffer read through row_idx = the active
    positions), "compact" (one logit row per active row, in compaction order)
    or None (no confidence pass).
    """

    name: str
    shape: workloads.StepShape
    n_active: int
    pattern: str
    locked: float
    conf: str
    logit_rows: int
    default_steps: int
    desc: str
    schedule: int = 0  # steps of a lock schedule (masks from lock_schedule), 0 = none
    surelock: bool = False  # lock criterion and adaptive prefix after the six calls


def entries(wl: "Workload"):
    return SURELOCK_ORDER if wl.surelock else ENTRY_ORDER


def make_workload(args) -> Workload:
    wl = _make_workload(args)
    if args.surelock:
        if wl.conf != "gather":
            raise SystemExit("--surelock needs a long_4k workload (logits of every position)")
        wl = dataclasses.replace(
            wl, name=wl.name + "_surelock", surelock=True,
            desc=wl.desc + f"; the confidence comes with the lock criterion (KL < {LOCK_EPS}, "
                           f"uncertainty gate at the {round(100 * LOCK_GATE_Q)}th percentile) "
                           f"between these and the previous step's logits of the active rows, "
                           f"one call; after the prefix commit, the adaptive prefix "
                           f"({round(100 * ADAPT_LO)}-{round(100 * ADAPT_HI)}% of the active "
                           f"length)")
    return wl


def _make_workload(args) -> Workload:
    if args.workload == "step_1k":
        s = workloads.STEP_1K
        return Workload("step_1k", s, s.n_salient, "random", 0.0, "window", s.logit_rows, 10000,
                        f"partial step B{s.B} L{s.L} ({s.win_start} prompt + {s.Lw} gen) "
                        f"{s.H}x{s.d} heads, hidden {s.D}, vocab {s.V} over {s.logit_rows} "
                        f"gen rows, ~10% salient")
    if args.workload == "batch8_2k":
        s = workloads.BATCH8_2K
        n = round(args.frac * s.L)
        return Workload(f"batch8_2k_f{round(100 * args.frac):02d}_{args.pattern}", s, n,
                        args.pattern, 0.0, None, 0, 400,
                        f"partial step B{s.B} L{s.L} {s.H}x{s.d} heads, hidden {s.D}, "
                        f"{round(100 * args.frac)}% active ({args.pattern}), no logits")
    if args.workload == "long_4k_schedule":
        s = workloads.LONG_4K
        return Workload("long_4k_schedule", s, s.L, "random", 0.0, "gather", s.L, 64 * 8,
                        f"64-step schedule B{s.B} L{s.L} {s.H}x{s.d} heads, vocab {s.V}, "
                        f"locked fraction rising linearly 0 -> 90% (nested locked sets), "
                        f"logits of the active rows gathered from a [{s.L}, {s.V}] buffer",
                        schedule=64)
    if args.workload == "long_4k":
        s = workloads.LONG_4K
        n_locked = round(args.locked * s.L)
        return Workload(f"long_4k_locked{round(100 * args.locked):02d}", s, s.L - n_locked,
                        "random", args.locked, "gather", s.L, 200,
                        f"partial step B{s.B} L{s.L} {s.H}x{s.d} heads, vocab {s.V}, "
                        f"{round(100 * args.locked)}% locked, logits of the active rows "
                        f"gathered from a [{s.L}, {s.V}] buffer")
    if args.workload != "loop_b4_2k":
        raise SystemExit(f"{args.workload} is not a single-step workload")
    s = workloads.LOOP_B4_2K
    n = 134
    return Workload("loop_b4_2k", s, n, "random", 0.0, "compact", 160, 2000,
                    f"partial step B{s.B} L{s.L} ({s.win_start} prompt + {s.Lw} gen) "
                    f"{s.H}x{s.d} heads, hidden {s.D}, vocab {s.V}, {n} active per batch row, "
                    f"logits of the active rows only")


def build_set(wl: Workload, seed: int, device):
    """Inputs of one step on the device (and the host copies for e2e)."""
    s = wl.shape
    inp = workloads.make_step(dataclasses.replace(s, logit_rows=0) if wl.conf != "window" else s,
                              n_salient=0 if wl.conf == "gather" else wl.n_active,
                              pattern=wl.pattern, seed=seed, with_logits=wl.conf == "window")
    g = torch.Generator().manual_seed(seed + 7)
    if wl.conf == "gather":
        inp["logits"] = workloads.normal(g, (s.B, s.L, s.V), 2.0, s.dtype)
        if wl.surelock:
            # the previous step's logits: these plus noise whose scale, one per
            # position, spans 1e-3 .. 1, so the divergences span decades
            scale = torch.logspace(-3, 0, s.L)[torch.randperm(s.L, generator=g)]
            prev = inp["logits"].float()
            prev.add_(scale[None, :, None] * torch.randn(prev.shape, generator=g))
            inp["logits_prev"] = prev.to(s.dtype)
            del prev
    elif wl.conf == "compact":
        inp["logits"] = workloads.normal(g, (s.B, wl.logit_rows, s.V), 2.0, s.dtype)
    locked = None
    if wl.locked > 0:
        n_locked = round(wl.locked * s.Lw)
        locked = torch.zeros((s.B, s.Lw), dtype=torch.uint8)
        for b in range(s.B):
            locked[b, torch.randperm(s.Lw, generator=g)[:n_locked]] = 1
    inp["locked"] = locked
    d = {k: inp[k].to(device) for k in ("cur", "prev", "k_cache", "v_cache", "k_new", "v_new", "q")}
    d["locked"] = None if locked is None else locked.to(device)
    if wl.conf == "compact":
        # R_max = M_max logit rows; only rows < count are ever read
        buf = torch.zeros((s.B, s.Lw, s.V), dtype=s.dtype, device=device)
        buf[:, :wl.logit_rows] = inp["logits"].to(device)
        d["logits"] = buf
    elif wl.conf is not None:
        d["logits"] = inp["logits"].to(device)
    if wl.surelock:
        d["logits_prev"] = inp["logits_prev"].to(device)
    d["score"] = torch.full((s.B, s.L), float("inf"), device=device)
    d["start"] = torch.full((s.B,), s.win_start, dtype=torch.int32, device=device)
    d["host"] = inp
    return d


def lock_schedule(wl: Workload, seed: int):
    """Nested locked sets of a linear schedule: at step t of T a fraction
    0.9 t / (T - 1) of the window is locked, the positions locking in one
    seeded random order.  Returns T uint8 masks [B, Lw] (CPU)."""
    s = wl.shape
    g = torch.Generator().manual_seed(seed)
    order = [torch.randperm(s.Lw, generator=g) for _ in range(s.B)]
    masks = []
    for t in range(wl.schedule):
        n_locked = round(0.9 * t / (wl.schedule - 1) * s.Lw)
        m = torch.zeros((s.B, s.Lw), dtype=torch.uint8)
        for b in range(s.B):
            m[b, order[b][:n_locked]] = 1
        masks.append(m)
    return masks


def set_bytes(d) -> int:
    return sum(t.numel() * t.element_size() for k, t in d.items()
               if isinstance(t, torch.Tensor) and t.is_cuda)


class Buffers:
    """Outputs and workspaces of the step, allocated once."""

    def __init__(self, dl, wl: Workload, device):
        s = wl.shape
        f32, i32 = torch.float32, torch.int32
        self.M_max = s.Lw
        self.cos = torch.empty((s.B, s.Lw), dtype=f32, device=device)
        self.idx = torch.empty((s.B, s.Lw), dtype=i32, device=device)
        self.count = torch.empty((s.B,), dtype=i32, device=device)
        self.o = torch.empty((s.B, self.M_max, s.H, s.d), dtype=s.dtype, device=device)
        self.lse = torch.empty((s.B, s.H, self.M_max), dtype=f32, device=device)
        self.colsum = torch.empty((s.B, s.H, s.L), dtype=f32, device=device)
        self.argmax = torch.zeros((s.B, s.L), dtype=i32, device=device)
        self.margin = torch.zeros((s.B, s.L), dtype=f32, device=device)
        self.length = torch.empty((s.B,), dtype=i32, device=device)
        self.dev_status = torch.zeros((1,), dtype=i32, device=device)
        r_max = s.logit_rows if wl.conf == "window" else s.Lw
        cw = dl.dllm_confidence_workspace_bytes(s.B, max(r_max, 1), s.V, s.dtype)
        self.conf_ws = torch.empty((max(cw, 16),), dtype=torch.uint8, device=device)
        aw = dl.dllm_attention_workspace_bytes(s.B, s.L, s.H, s.d, self.M_max, s.dtype)
        self.attn_ws = torch.empty((max(aw, 16),), dtype=torch.uint8, device=device)
        self.attn_split = aw > 0
        if wl.surelock:
            self.kl = torch.empty((s.B, s.L), dtype=f32, device=device)
            self.unc = torch.empty((s.B, s.L), dtype=f32, device=device)
            self.lock_flags = torch.zeros((s.B, s.L), dtype=torch.uint8, device=device)
            lw = dl.dllm_lock_workspace_bytes(s.B, s.Lw, s.V, s.dtype)
            self.lock_ws = torch.empty((max(lw, 16),), dtype=torch.uint8, device=device)
            self.alen = torch.empty((s.B,), dtype=i32, device=device)
            self.atau = torch.empty((s.B,), dtype=f32, device=device)


def run_step(dl, wl: Workload, bf: Buffers, d, stream, events=None, locked=None):
    """The six calls in order (eight with the lock criterion and the adaptive
    prefix); optional events bracket each call.  ``locked`` overrides the
    set's locked mask (schedule steps).  The lock flags go to a buffer of
    their own: the set's mask or the schedule decides what is locked, so that
    every replay of the step does the same work."""
    s = wl.shape
    w = s.win_start
    ev = events
    if locked is None:
        locked = d["locked"]
    if ev: ev[0].record(stream)
    dl.dllm_saliency_select(d["cur"][:, w:], d["prev"][:, w:], s.tau, locked=locked,
                            idx_base=w, cos_out=bf.cos, idx_out=bf.idx, count_out=bf.count,
                            dev_status=bf.dev_status, stream=stream)
    if ev: ev[1].record(stream)
    dl.dllm_kv_scatter(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], bf.idx, bf.count,
                       dev_status=bf.dev_status, stream=stream)
    if ev: ev[2].record(stream)
    dl.dllm_partial_attention(d["q"], d["k_cache"], d["v_cache"], bf.count, o_out=bf.o,
                              lse_out=bf.lse, with_colsum=False, ws=bf.attn_ws,
                              dev_status=bf.dev_status, stream=stream)
    if ev: ev[3].record(stream)
    dl.dllm_attention_colsum(d["q"], d["k_cache"], bf.count, bf.lse, colsum_out=bf.colsum,
                             dev_status=bf.dev_status, stream=stream)
    if ev: ev[4].record(stream)
    if wl.conf == "window":
        dl.dllm_confidence(d["logits"], out_cols=s.L, conf_out=d["score"][:, w:],
                           argmax_out=bf.argmax[:, w:], margin_out=bf.margin[:, w:],
                           ws=bf.conf_ws, dev_status=bf.dev_status, stream=stream)
    elif wl.conf == "gather" and wl.surelock:
        dl.dllm_lock_criterion_conf(d["logits"], d["logits_prev"], LOCK_EPS, gate_q=LOCK_GATE_Q,
                                    R_max=s.Lw, row_idx=bf.idx, count=bf.count, out_idx=bf.idx,
                                    out_cols=s.L, kl_out=bf.kl, unc_out=bf.unc,
                                    conf_out=d["score"], argmax_out=bf.argmax,
                                    margin_out=bf.margin, locked_inout=bf.lock_flags,
                                    ws=bf.lock_ws, dev_status=bf.dev_status, stream=stream)
    elif wl.conf == "gather":
        dl.dllm_confidence(d["logits"], R_max=s.Lw, row_idx=bf.idx, count=bf.count,
                           out_idx=bf.idx, out_cols=s.L, conf_out=d["score"],
                           argmax_out=bf.argmax, margin_out=bf.margin, ws=bf.conf_ws,
                           dev_status=bf.dev_status, stream=stream)
    elif wl.conf == "compact":
        dl.dllm_confidence(d["logits"], R_max=s.Lw, count=bf.count, out_idx=bf.idx,
                           out_cols=s.L, conf_out=d["score"], argmax_out=bf.argmax,
                           margin_out=bf.margin, ws=bf.conf_ws, dev_status=bf.dev_status,
                           stream=stream)
    if ev: ev[5].record(stream)
    dl.dllm_stable_prefix(d["score"], d["start"], 0.9, min_commit=True, advance_start=False,
                          len_out=bf.length, dev_status=bf.dev_status, stream=stream)
    if ev: ev[6].record(stream)
    if not wl.surelock:
        return
    dl.dllm_adaptive_prefix(d["score"], d["start"], ADAPT_LO, ADAPT_HI, len_out=bf.alen,
                            tau_out=bf.atau, dev_status=bf.dev_status, stream=stream)
    if ev: ev[7].record(stream)


def launches_per_step(wl: Workload, bf: Buffers) -> int:
    # select 2, scatter 1, attention 1 (+ the split merge), column sums 2
    # (persistent kernel for small heads, key-tile-group kernel for the
    # rest), prefix 1; confidence 2 (streaming kernel, row merge)
    n = 2 + 1 + (2 if bf.attn_split else 1) + 2 + 1
    if wl.surelock:  # lock criterion with the confidence (partials, merge, gate), adaptive prefix
        n += 3 + 1
    elif wl.conf is not None:
        n += 2
    return n


def algorithmic_work(wl: Workload, counts):
    """Algorithmic bytes / flops of each entry point for one step."""
    s = wl.shape
    M = int(sum(counts))
    el = 2 if s.dtype == torch.bfloat16 else 4
    hd = s.H * s.d
    select_b = 2 * s.B * s.Lw * s.D * el + s.B * s.Lw * 8
    scatter_b = M * 2 * 2 * hd * el
    # K and V once per batch row, Q in and O out per active row, lse out
    attn_b = 2 * s.B * s.L * hd * el + 2 * M * hd * el + M * s.H * 4
    attn_f = 4.0 * M * s.L * s.d * s.H
    # K once per batch row, Q and lse per active row, colsum out
    colsum_b = s.B * s.L * hd * el + M * hd * el + M * s.H * 4 + s.B * s.H * s.L * 4
    if wl.conf == "window":
        conf_rows = s.B * s.logit_rows
    elif wl.conf is None:
        conf_rows = 0
    else:
        conf_rows = M
    conf_b = conf_rows * (s.V * el + 12)
    prefix_b = s.B * s.Lw * 4
    # both logit rows of every active row, its index twice, kl, unc and flag
    lock_b = M * (2 * s.V * el + 4 + 4 + 4 + 4 + 1)
    return {
        "dllm_lock_criterion": {"bytes": lock_b, "flops": 0.0},
        # both logit rows once, the criterion's and the confidence's outputs
        "dllm_lock_criterion_conf": {"bytes": lock_b + M * 12, "flops": 0.0},
        "dllm_adaptive_prefix": {"bytes": s.B * s.Lw * 4, "flops": 0.0},
        "dllm_saliency_select": {"bytes": select_b, "flops": 6.0 * s.B * s.Lw * s.D},
        "dllm_kv_scatter": {"bytes": scatter_b, "flops": 0.0},
        "dllm_partial_attention": {"bytes": attn_b, "flops": attn_f},
        # algorithmically the pass only adds L terms per active row; the
        # executed work recomputes Q K^T (2 M L d H flops)
        "dllm_attention_colsum": {"bytes": colsum_b, "flops": 2.0 * M * s.L * s.d * s.H,
                                  "alg_adds": float(M * s.L * s.H)},
        "dllm_confidence": {"bytes": conf_b, "flops": 0.0},
        "dllm_stable_prefix": {"bytes": prefix_b, "flops": 0.0},
    }


# ----------------------------------------------------------------------------- CPU oracle

def oracle_step(wl: Workload, h, b: int, locked_mask=None):
    """The float64 oracle over batch row ``b`` of one step (what the GPU step
    computes for that row).  Returns the row's active count."""
    import numpy as np
    import oracle
    s = wl.shape
    w = s.win_start
    sl = slice(b, b + 1)
    f = lambda k: h[k][sl].double().numpy()  # noqa: E731
    lk = h["locked"] if locked_mask is None else locked_mask
    locked = None if lk is None else lk[sl].numpy()
    cur, prev = f("cur"), f("prev")
    cos, idx, count = oracle.saliency_select(cur[:, w:], prev[:, w:], s.tau, locked, idx_base=w)
    kc, vc = oracle.kv_scatter(f("k_cache"), f("v_cache"), f("k_new"), f("v_new"), idx, count)
    o, lse, colsum = oracle.partial_attention(f("q"), kc, vc, count)
    score = np.full((1, s.L), np.inf)
    if wl.conf == "window":
        conf, _, _ = oracle.confidence(f("logits"))
        score[:, w:w + conf.shape[1]] = conf
    elif wl.conf == "gather":
        conf, _, _ = oracle.confidence(f("logits"), count=count, row_idx=idx)
        n = int(count[0])
        score[0, idx[0, :n]] = conf[0, :n]
    elif wl.conf == "compact":
        n = min(int(count[0]), wl.logit_rows)
        conf, _, _ = oracle.confidence(f("logits"), count=[n])
        score[0, idx[0, :n]] = conf[0, :n]
    oracle.stable_prefix(score, [w], 0.9, True)
    if wl.surelock:
        kl, unc = oracle.lock_kl(f("logits"), f("logits_prev"), count=count, row_idx=idx)
        oracle.lock_decision(kl, unc, count, LOCK_EPS, LOCK_GATE_Q)
        oracle.adaptive_prefix(score, [w], ADAPT_LO, ADAPT_HI)
    return int(count[0])


def blas_threads():
    """Threads numpy's BLAS runs with (all host cores unless capped)."""
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except ImportError:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return os.cpu_count() or 1


def cpu_baseline(wl: Workload, host, seconds, steps_cap=None, masks=None):
    """The float64 oracle, as it stands, on the host cores: batch rows of the
    same step (of the schedule's steps in turn) taken in turn until
    ``seconds`` have passed (or ``steps_cap`` batch rows), at least one."""
    times, rows, units = [], 0, 0
    t_begin = time.perf_counter()
    cpu_begin = time.process_time()
    while True:
        t0 = time.perf_counter()
        mask = None if masks is None else masks[(rows // wl.shape.B) % len(masks)]
        units += oracle_step(wl, host, rows % wl.shape.B, mask)
        rows += 1
        times.append(time.perf_counter() - t0)
        if steps_cap is not None and rows >= steps_cap:
            break
        if steps_cap is None and time.perf_counter() - t_begin >= seconds:
            break
    elapsed = sum(times)
    util = (time.process_time() - cpu_begin) / max(time.perf_counter() - t_begin, 1e-9)
    return {"value": units / elapsed, "unit": UNIT, "cores": blas_threads(),
            "cpu_utilisation": round(util, 2), "kind": "oracle",
            "sample": f"{rows} batch row(s) of the {wl.name} step through the float64 oracle "
                      f"({units} active rows in all), {elapsed:.1f} s on the host"}, times, units


def reference_arm(args, rank):
    """`--impl reference`: the float64 oracle timed as the reference arm."""
    if rank != 0:
        return 0
    wl = make_workload(args)
    host = build_set(wl, wl.shape.seed, torch.device("cpu"))["host"]
    masks = lock_schedule(wl, wl.shape.seed + 5) if wl.schedule else None
    # warm-up rows (at most 3), then as many of the K timed rows as fit in
    # about 90 s of oracle time, at least 3: the run stays within minutes
    _, wt, _ = cpu_baseline(wl, host, 0, steps_cap=max(1, min(args.warmup, 3)), masks=masks)
    per_row = sum(wt) / len(wt)
    k = args.steps if args.steps is not None else 10
    res, times, units = cpu_baseline(wl, host, 0,
                                     steps_cap=max(3, min(k, int(90.0 / max(per_row, 1e-6)))),
                                     masks=masks)
    timed = sum(times)
    value = units / timed
    rows_per_step = wl.shape.B
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": timed / len(times) * rows_per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.desc, "name": wl.name},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": res["cores"],
                             "kind": "oracle",
                             "sample": f"{len(times)} timed batch row(s) of the step through the "
                                       f"float64 oracle after {len(wt)} warm-up row(s)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- decoding loop

LOOP_ORDER = ENTRY_ORDER  # the six calls of a loop step, in order
LOOP_LAUNCHES_PER_STEP = 8  # cos_rows + compact, kv_scatter, attn_fwd (no workspace: no
                            # split merge), attn_colsum_stream (no row above 2 query tiles),
                            # conf_stream + conf_merge, stable_prefix


def loop_desc(sh) -> str:
    return (f"block-wise decoding loop B{sh.B} L{sh.L} ({sh.prompt} prompt + {sh.L - sh.prompt} "
            f"gen in blocks of {sh.block}, {sh.steps_per_block} steps per block, {sh.T} steps) "
            f"{sh.H}x{sh.d} heads, hidden {sh.D}, vocab {sh.V}; per step: select over the gen "
            f"rows (all {sh.L} rows every {sh.refresh}th step), kv_scatter, partial attention + "
            f"column sums, confidence of the active rows, prefix commit advancing start; active "
            f"= the block's undecoded positions + {sh.n_random} random gen positions per batch row")


def loop_step_work(sh, counts, win_start):
    """Algorithmic bytes / flops of each call of one loop step (counts: the
    active rows of each batch row)."""
    M = int(sum(counts))
    el = 2 if sh.dtype == torch.bfloat16 else 4
    hd = sh.H * sh.d
    Lw = sh.L - win_start
    return {
        "dllm_saliency_select": {"bytes": 2 * sh.B * Lw * sh.D * el + sh.B * Lw * 8,
                                 "flops": 6.0 * sh.B * Lw * sh.D},
        "dllm_kv_scatter": {"bytes": M * 2 * 2 * hd * el, "flops": 0.0},
        "dllm_partial_attention": {"bytes": 2 * sh.B * sh.L * hd * el + 2 * M * hd * el
                                   + M * sh.H * 4, "flops": 4.0 * M * sh.L * sh.d * sh.H},
        "dllm_attention_colsum": {"bytes": sh.B * sh.L * hd * el + M * hd * el + M * sh.H * 4
                                  + sh.B * sh.H * sh.L * 4,
                                  "flops": 2.0 * M * sh.L * sh.d * sh.H,
                                  "alg_adds": float(M * sh.L * sh.H)},
        "dllm_confidence": {"bytes": M * (sh.V * el + 12), "flops": 0.0},
        # the scores from start up to the first unstable position, and start
        "dllm_stable_prefix": {"bytes": sh.B * ((sh.commit + 1) * 4 + 8), "flops": 0.0},
    }


def oracle_loop_rows(sh, pools, b: int, seconds: float, steps_cap=None):
    """The float64 oracle playing the loop for batch row ``b``, step after
    step with its cache, score and start carried, until ``seconds`` have
    passed (or ``steps_cap`` steps).  Returns (per-step seconds, active rows)."""
    import numpy as np
    import oracle
    cap = workloads.loop_row_cap(sh)
    f = lambda t: t[b:b + 1].double().numpy()  # noqa: E731
    kc, vc, prev = f(pools["k_cache"]), f(pools["v_cache"]), f(pools["prev"])
    score = np.zeros((1, sh.L))
    score[:, :sh.prompt] = np.inf
    start = np.array([sh.prompt])
    times, units = [], 0
    t_begin = time.perf_counter()
    for t in range(sh.T):
        inp = workloads.loop_step_inputs(sh, pools, t, cap)
        t0 = time.perf_counter()
        w = inp["win_start"]
        _, idx, count = oracle.saliency_select(f(inp["cur"])[:, w:], prev[:, w:], sh.tau,
                                               idx_base=w)
        kc, vc = oracle.kv_scatter(kc, vc, f(inp["k_new"]), f(inp["v_new"]), idx, count)
        oracle.partial_attention(f(inp["q"]), kc, vc, count)
        conf, _, _ = oracle.confidence(f(inp["logits"]), count=count)
        n = int(count[0])
        score[0, idx[0, :n]] = conf[0, :n]
        start = start + oracle.stable_prefix(score, start, sh.tau_c, True)
        times.append(time.perf_counter() - t0)
        units += n
        if steps_cap is not None and len(times) >= steps_cap:
            break
        if steps_cap is None and time.perf_counter() - t_begin >= seconds:
            break
    return times, units


def loop_cpu_baseline(sh, pools, seconds, steps_cap=None):
    cpu0, wall0 = time.process_time(), time.perf_counter()
    times, units = oracle_loop_rows(sh, pools, 0, seconds, steps_cap)
    util = (time.process_time() - cpu0) / max(time.perf_counter() - wall0, 1e-9)
    elapsed = sum(times)
    return {"value": units / elapsed, "unit": UNIT, "cores": max(1, round(util)),
            "cpu_utilisation": round(util, 2), "blas_threads": blas_threads(), "kind": "oracle",
            "sample": f"steps 0-{len(times) - 1} of the loop for batch row 0 through the float64 "
                      f"oracle (state carried; {units} active rows), {elapsed:.1f} s of oracle "
                      f"time on the host; cores = CPU time / wall time of the sample"}, times, units


def loop_reference_arm(args, rank):
    if rank != 0:
        return 0
    sh = workloads.LOOP_128
    pools = workloads.make_loop_pools(sh)
    # warm-up steps (at most 3), then as many of the loop's first K steps as
    # fit in about 90 s of oracle time, at least 3
    wt, _ = oracle_loop_rows(sh, pools, 0, 0, steps_cap=max(1, min(args.warmup, 3)))
    per = sum(wt) / len(wt)
    k = args.steps if args.steps is not None else sh.T
    cap_steps = max(3, min(k, sh.T, int(90.0 / max(per, 1e-6))))
    res, times, units = loop_cpu_baseline(sh, pools, 0, steps_cap=cap_steps)
    value = units / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": len(times), "warmup": args.warmup,
            "ms_per_step": sum(times) / len(times) * sh.B * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": loop_desc(sh), "name": "loop_b4_2k_128"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": res["cores"],
                             "kind": "oracle",
                             "sample": f"{len(times)} timed loop steps of batch row 0 through "
                                       f"the float64 oracle after {len(wt)} warm-up step(s); "
                                       f"ms_per_step scales one row's time by the batch"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main_loop(args, rank, world, device, pg):
    import partial_attention_saliency_b300 as dl
    dl.load_library()
    sh = workloads.LOOP_128
    T = sh.T
    pools = workloads.make_loop_pools(sh)
    dpools = {k: v.to(device) for k, v in pools.items()}
    cap_rows = workloads.loop_row_cap(sh)
    counts = workloads.loop_counts(sh).tolist()  # [T][B], the planted sets
    K = args.steps if args.steps is not None else T
    W = args.warmup
    # the inputs of every step the run touches (the timed K, the warm-up W,
    # the first 8 for the end-to-end leg), each its own buffers
    n_build = min(T, max(K, W, 8))
    steps = [workloads.loop_step_inputs(sh, dpools, t, cap_rows) for t in range(n_build)]
    for st in steps:
        st.pop("planted")
    torch.cuda.synchronize()
    lp = dl.BlockDecodeLoop(sh.B, sh.L, sh.H, sh.d, sh.V, sh.dtype, sh.prompt, cap_rows, sh.tau,
                            sh.tau_c, device=device)
    stream = torch.cuda.current_stream(device)

    def run(t, events=None):
        st = steps[t]
        lp.step(st["cur"], dpools["prev"], st["q"], st["k_new"], st["v_new"], st["logits"],
                st["win_start"], events=events)

    # one eager pass over the built steps: each selects its planted set and
    # commits the block's next positions (over the whole loop start ends at L)
    lp.reset(dpools["k_cache"], dpools["v_cache"])
    for t in range(n_build):
        run(t)
        if t < 8:
            torch.cuda.synchronize()
            assert lp.count.cpu().tolist() == counts[t], (t, lp.count.cpu().tolist(), counts[t])
            assert lp.length.cpu().tolist() == [sh.commit] * sh.B, (t, lp.length.cpu().tolist())
    torch.cuda.synchronize()
    assert int(lp.dev_status[0]) == 0, "device-side check failed"
    assert lp.start.cpu().tolist() == [sh.prompt + sh.commit * n_build] * sh.B, \
        lp.start.cpu().tolist()

    # ---------------------------------------------------------------- device-timed
    # The K timed steps (the loop's steps 0 .. K-1, restarting the loop from a
    # fresh score and start after step T-1) are one CUDA graph; the graph's
    # first node resets score and start.  It is replayed once untimed, then
    # the K-step region is timed repeatedly for about a second (events on the
    # stream around each replay) and the median is reported.
    cap = torch.cuda.Stream(device)
    g_warm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=cap):
        for i in range(W):
            if i % T == 0:
                lp.reset_positions()
            run(i % T)
    g_timed = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_timed, stream=cap):
        for i in range(K):
            if i % T == 0:
                lp.reset_positions()
            run(i % T)
    S = min(K, T)
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(7)]
          for _ in range(S)]
    g_events = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_events, stream=cap):
        lp.reset_positions()
        for i in range(S):
            run(i, ev[i])
    clocks = ClockSampler(torch.cuda.current_device())
    g_warm.replay()
    torch.cuda.synchronize()
    if pg: pg.barrier()
    torch.cuda.synchronize()
    clocks.start()
    reps = time_regions(g_timed.replay, stream, est_ms=0.15 * K, warm=g_timed.replay,
                        min_seconds=args.min_seconds)
    clocks.stop()
    if pg: pg.barrier()
    g_events.replay()
    torch.cuda.synchronize()
    assert int(lp.dev_status[0]) == 0, "device-side check failed"
    elapsed_ms = statistics.median(reps)
    active_total = sum(sum(counts[i % T]) for i in range(K))
    elapsed_ms, active_total = reduce_over_ranks(pg, elapsed_ms, active_total, device)
    value = active_total / (elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / K

    # ---------------------------------------------------------------- per call
    pk = peaks()
    per_ms = {n: 0.0 for n in LOOP_ORDER}
    work = {n: {"bytes": 0.0, "flops": 0.0} for n in LOOP_ORDER}
    for i in range(S):
        w = loop_step_work(sh, counts[i], workloads.loop_window(sh, i))
        for j, n in enumerate(LOOP_ORDER):
            per_ms[n] += ev[i][j].elapsed_time(ev[i][j + 1])
            work[n]["bytes"] += w[n]["bytes"]
            work[n]["flops"] += w[n]["flops"]
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    kernels = {}
    total_ms = sum(per_ms.values())
    for n in LOOP_ORDER:
        t_s = per_ms[n] / 1e3
        gbs = work[n]["bytes"] / t_s / 1e9
        tfs = work[n]["flops"] / t_s / 1e12
        ai = work[n]["flops"] / max(work[n]["bytes"], 1)
        bound = "tensor" if n == "dllm_partial_attention" and ai > ridge else "hbm"
        kernels[n] = {"us": per_ms[n] / S * 1e3, "share": per_ms[n] / total_ms,
                      "alg_bytes": work[n]["bytes"] / S, "alg_flops": work[n]["flops"] / S,
                      "GB/s": gbs, "TFLOP/s": tfs, "bound": bound,
                      "frac": (tfs / pk["bf16_tflops"]) if bound == "tensor"
                      else gbs / pk["hbm_gbs"], "kernels": KERNELS[n][0]}
    # the single-launch read reference at each memory-bound call's byte count
    ceil = read_ceiling({n: kernels[n]["alg_bytes"] for n in LOOP_ORDER
                         if kernels[n]["bound"] == "hbm" and kernels[n]["alg_bytes"] >= 1 << 20},
                        device)
    for n, us in ceil.items():
        kernels[n]["read_ceiling_us"] = us
        kernels[n]["frac_of_read_ceiling"] = us / kernels[n]["us"]
    dom = max(kernels, key=lambda n: kernels[n]["us"])
    dk = kernels[dom]
    if dk["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": dk["TFLOP/s"], "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": dk["TFLOP/s"] / pk["bf16_tflops"]}
    else:
        roof = {"bound": "hbm", "achieved": dk["GB/s"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": dk["GB/s"] / pk["hbm_gbs"]}
        if dom in ceil:
            roof["read_ceiling"] = {
                "us": ceil[dom], "GB/s": dk["alg_bytes"] / ceil[dom] / 1e3,
                "frac_of_peak": dk["alg_bytes"] / ceil[dom] / 1e3 / pk["hbm_gbs"],
                "frac": ceil[dom] / dk["us"],
                "what": "dllm_read_stream over the same bytes: one launch that only streams "
                        "them into shared memory, timed the same way"}
    tr = TRAFFIC.get(("loop_b4_2k_128", dom))
    traffic = None
    if tr is not None and tr["src_sha"] == src_sha(KERNELS[dom][1]):
        traffic = tr["bytes"]
    roof.update({"traffic": traffic, "kernel": dom, "kernels": KERNELS[dom][0],
                 "peak_source": pk["source"] + " (burst)",
                 "alg_per_launch": dk["alg_flops"] if roof["unit"] == "TFLOP/s"
                 else dk["alg_bytes"],
                 "timing": "CUDA events around the call on the launching stream, averaged "
                           f"over steps 0-{S - 1} of a replay of the loop graph with an event "
                           "between every two calls"})

    # ---------------------------------------------------------------- end to end
    e2e = loop_e2e(lp, sh, steps, pools, dpools, counts, cap_rows, run, stream, pg, device)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": ms_per_step, "latency_us_per_step": ms_per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": loop_desc(sh), "name": "loop_b4_2k_128", "batch": sh.B,
                       "seq_len": sh.L, "prompt": sh.prompt, "block": sh.block,
                       "loop_steps": T, "heads": sh.H, "head_dim": sh.d, "hidden": sh.D,
                       "vocab": sh.V,
                       "active_rows_per_step": active_total / K / max(world, 1),
                       "l2": "inputs larger than L2: every step reads its own hidden states "
                             "(64 MB), logit rows (~136 MB) and fresh rows, and the 134 MB "
                             "K/V cache",
                       "parallelism": "replicas (one independent loop per GPU)"},
            "roofline": roof, "kernels": kernels, "clocks": clocks.summary(),
            "gpu_launches": LOOP_LAUNCHES_PER_STEP * K,
            "timing": f"median of {len(reps)} timed regions (one replay each of a CUDA graph of "
                      f"the {K} steps), after one untimed replay; region times "
                      f"{min(reps):.3f}-{max(reps):.3f} ms",
            "us_per_step_with_call_events": total_ms / S * 1e3, "e2e": e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb, _, _ = loop_cpu_baseline(sh, pools, args.cpu_seconds)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def loop_e2e(lp, sh, steps, pools, dpools, counts, cap_rows, run, stream, pg, device,
             host_steps: int = 8):
    """The loop through the public API with host buffers: each step copies its
    inputs from pinned host memory (the window's hidden states, the fresh
    query/key/value rows and the logit rows of the rows that can be active)
    and reads its results back (indices, counts, outputs, log-sum-exps,
    column sums, scores, argmax, prefix length and start).  Runs the loop's
    first ``host_steps`` steps over and over, restarting score and start."""
    E = host_steps
    host = []
    for t in range(E):
        inp = workloads.loop_step_inputs(sh, pools, t, cap_rows)
        w = inp["win_start"]
        host.append({"cur": inp["cur"][:, w:].contiguous().pin_memory(),
                     "q": inp["q"][:, :cap_rows].contiguous().pin_memory(),
                     "k_new": inp["k_new"][:, :cap_rows].contiguous().pin_memory(),
                     "v_new": inp["v_new"][:, :cap_rows].contiguous().pin_memory(),
                     "logits": inp["logits"].pin_memory(), "w": w})
    Lw_max = sh.L
    out = {"idx": torch.empty((sh.B * Lw_max,), dtype=torch.int32).pin_memory(),
           "count": torch.empty((sh.B,), dtype=torch.int32).pin_memory(),
           "o": torch.empty((sh.B, cap_rows, sh.H, sh.d), dtype=sh.dtype).pin_memory(),
           "lse": torch.empty((sh.B, sh.H, cap_rows), dtype=torch.float32).pin_memory(),
           "colsum": torch.empty((sh.B, sh.H, sh.L), dtype=torch.float32).pin_memory(),
           "score": torch.empty((sh.B, sh.L), dtype=torch.float32).pin_memory(),
           "argmax": torch.empty((sh.B, sh.L), dtype=torch.int32).pin_memory(),
           "length": torch.empty((sh.B,), dtype=torch.int32).pin_memory(),
           "start": torch.empty((sh.B,), dtype=torch.int32).pin_memory()}
    h2d, d2h = [], []

    def one(t):
        hs, ds = host[t], steps[t]
        w = hs["w"]
        Lw = sh.L - w
        # one contiguous copy per batch row (the window and the first rows of
        # each batch row are contiguous; the batch rows are not)
        for b in range(sh.B):
            ds["cur"][b, w:].copy_(hs["cur"][b], non_blocking=True)
            for k in ("k_new", "v_new"):
                ds[k][b, :cap_rows].copy_(hs[k][b], non_blocking=True)
        ds["q"].copy_(hs["q"], non_blocking=True)
        ds["logits"].copy_(hs["logits"], non_blocking=True)
        run(t)
        out["idx"][:sh.B * Lw].copy_(lp.idx(Lw).view(-1), non_blocking=True)
        out["count"].copy_(lp.count, non_blocking=True)
        out["o"].copy_(lp.o, non_blocking=True)
        out["lse"].copy_(lp.lse, non_blocking=True)
        for k, src in (("colsum", lp.colsum), ("score", lp.score), ("argmax", lp.argmax),
                       ("length", lp.length), ("start", lp.start)):
            out[k].copy_(src, non_blocking=True)
        h2d.append(sum(hs[k].numel() * hs[k].element_size()
                       for k in ("cur", "q", "k_new", "v_new", "logits")))
        d2h.append(sh.B * Lw * 4 + sum(out[k].numel() * out[k].element_size()
                                       for k in ("count", "o", "lse", "colsum", "score",
                                                 "argmax", "length", "start")))

    lp.reset_positions()
    for t in range(E):
        one(t)
    torch.cuda.synchronize()
    h2d.clear()
    d2h.clear()
    n_steps = 4 * E
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if pg: pg.barrier()
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(n_steps):
        if i % E == 0:
            lp.reset_positions()
        one(i % E)
    b.record(stream)
    torch.cuda.synchronize()
    assert int(lp.dev_status[0]) == 0
    ms = a.elapsed_time(b)
    active = sum(sum(counts[i % E]) for i in range(n_steps))
    ms, active = reduce_over_ranks(pg, ms, active, device)
    return {"value": active / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": sum(h2d) / len(h2d), "d2h_bytes_per_step": sum(d2h) / len(d2h),
            "steps": n_steps, "ms_per_step": ms / n_steps,
            "sample": f"the loop's steps 0-{E - 1} from pinned host buffers, {n_steps // E} times"}


# ----------------------------------------------------------------------------- around the step

FP32_SIMT_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12  # SMs x FP32 lanes x 2 (FMA) x max clock


def main_around(args, rank, world, device, pg):
    """The calls that run around the step, each timed alone (a graph of 20
    calls, median of 15 replays), on the state of the 128-step loop's step 1
    (batch 4, L 2048, the step's active rows): DyLLM's stable-row update
    (every position not active this step is a stable row, the active ones
    the salient columns; tensor cores, HBM-bound by its arithmetic
    intensity of about 77 flop/B), Attn-Sampler's total attention and order,
    SlowFast's device controller and token selection, SureLock's lock
    criterion (this step's logit rows against another step's).  Prints one
    line whose value is the step's active rows per second through these
    calls together, with the per-call breakdown."""
    import partial_attention_saliency_b300 as dl
    dl.load_library()
    sh = workloads.LOOP_128
    pools = workloads.make_loop_pools(sh)
    dp = {k: v.to(device) for k, v in pools.items()}
    cap = workloads.loop_row_cap(sh)
    lp = dl.BlockDecodeLoop(sh.B, sh.L, sh.H, sh.d, sh.V, sh.dtype, sh.prompt, cap, sh.tau,
                            sh.tau_c, device=device)
    lp.reset(dp["k_cache"], dp["v_cache"])
    st0, st1 = (workloads.loop_step_inputs(sh, dp, t, cap) for t in range(2))
    for st in (st0, st1):
        lp.step(st["cur"], dp["prev"], st["q"], st["k_new"], st["v_new"], st["logits"],
                st["win_start"])
    torch.cuda.synchronize()
    counts = lp.count.cpu().tolist()
    M = sum(counts)
    Lw = sh.L - st1["win_start"]
    idx = lp.idx(Lw)
    B, L, H, d, V = sh.B, sh.L, sh.H, sh.d, sh.V
    g = torch.Generator(device=device).manual_seed(9)
    rnd = lambda *shape: torch.randn(shape, generator=g, device=device).to(sh.dtype)  # noqa: E731
    q_prev, v_prev, o = rnd(B, L, H, d), rnd(B, L, H, d), rnd(B, L, H, d)
    lse_prev = torch.randn((B, H, L), generator=g, device=device) + 8.0
    stable = torch.ones((B, L), dtype=torch.bool, device=device)
    for b in range(B):
        stable[b, idx[b, :counts[b]].long()] = False
    stable_idx = torch.full((B, L), -1, dtype=torch.int32, device=device)
    stable_count = stable.sum(1).to(torch.int32)
    for b in range(B):
        pos = torch.nonzero(stable[b]).flatten().to(torch.int32)
        stable_idx[b, :pos.numel()] = pos
    N = int(stable_count.sum())
    masked = (~torch.isinf(lp.score)).to(torch.uint8)
    sf = dl.SlowFastDevice(B, 3, 2.0, device=device)
    plen = torch.full((B,), 8, dtype=torch.int32, device=device)
    logits_prev = st0["logits"]
    lock_ws = torch.empty((max(dl.dllm_lock_workspace_bytes(B, Lw, V, sh.dtype), 16),),
                          dtype=torch.uint8, device=device)
    kl = torch.empty((B, L), device=device)
    unc = torch.empty((B, L), device=device)
    flags = torch.zeros((B, L), dtype=torch.uint8, device=device)
    score = torch.empty((B, L), device=device)
    status = torch.zeros((1,), dtype=torch.int32, device=device)
    el = 2
    calls = {
        "dllm_approx_attention_update": (
            lambda: dl.dllm_approx_attention_update(q_prev, lse_prev, lp.k_cache, v_prev,
                                                    st1["v_new"], idx, lp.count, stable_idx,
                                                    stable_count, o, dev_status=status),
            H * (N * (3 * d * el + 4) + M * 3 * d * el), 4.0 * d * N * M / B * H, "hbm"),
        "dllm_attn_scores": (lambda: dl.dllm_attn_scores(lp.colsum, score_inout=score),
                             B * H * L * 4 + B * L * 4, 0.0, "hbm"),
        "dllm_attn_sampler_select": (
            lambda: dl.dllm_attn_sampler_select(score, candidates=masked, tau=0.0, gamma=0.5,
                                                k_max=8), B * L * 9 + B * 4, 0.0, "latency"),
        "dllm_slowfast_observe_device": (lambda: sf.observe(lp.start, plen), B * 40, 0.0,
                                         "latency"),
        "dllm_slowfast_select": (
            lambda: dl.dllm_slowfast_select(lp.score, lp.start, sf.phase, sf.region_end, 0.9,
                                            64, 4, masked=masked), B * L * 9, 0.0, "latency"),
        "dllm_lock_criterion": (
            lambda: dl.dllm_lock_criterion(st1["logits"], logits_prev, 1e-3, gate_q=0.5,
                                           R_max=Lw, count=lp.count, out_idx=idx, out_cols=L,
                                           kl_out=kl, unc_out=unc, locked_inout=flags, ws=lock_ws,
                                           dev_status=status),
            M * (2 * V * el + 17), 0.0, "hbm"),
    }
    pk = peaks()
    kernels, total_ms = {}, 0.0
    cap_stream = torch.cuda.Stream(device)
    for name, (fn, byts, flops, bound) in calls.items():
        fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap_stream):
            for _ in range(20):
                fn()
        ms = statistics.median(time_regions(gr.replay, torch.cuda.current_stream(device),
                                            est_ms=1.0, warm=gr.replay, min_seconds=0.2,
                                            min_reps=15)) / 20
        total_ms += ms
        k = {"us": ms * 1e3, "alg_bytes": byts, "GB/s": byts / (ms / 1e3) / 1e9, "bound": bound}
        if bound == "alu":
            k.update({"alg_flops": flops, "TFLOP/s": flops / (ms / 1e3) / 1e12,
                      "peak_TFLOP/s": FP32_SIMT_PEAK_TFLOPS,
                      "frac": flops / (ms / 1e3) / 1e12 / FP32_SIMT_PEAK_TFLOPS})
        elif bound == "hbm":
            k["frac"] = k["GB/s"] / pk["hbm_gbs"]
            if flops:
                k.update({"alg_flops": flops, "TFLOP/s": flops / (ms / 1e3) / 1e12,
                          "tensor_frac": flops / (ms / 1e3) / 1e12 / pk["bf16_tflops"]})
        kernels[name] = k
    torch.cuda.synchronize()
    assert int(status[0]) == 0, "device-side check failed"
    dom = max(kernels, key=lambda n: kernels[n]["us"])
    dk = kernels[dom]
    if dk["bound"] == "alu":
        roof = {"bound": "alu", "achieved": dk["TFLOP/s"], "peak": FP32_SIMT_PEAK_TFLOPS,
                "unit": "TFLOP/s", "frac": dk["frac"], "traffic": None, "kernel": dom,
                "peak_source": "derived: 148 SMs x 128 FP32 lanes x 2 flops x 2032 MHz"}
    else:
        roof = {"bound": "hbm", "achieved": dk["GB/s"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": dk["frac"], "traffic": None, "kernel": dom,
                "peak_source": pk["source"] + " (burst)"}
    for n, k in kernels.items():  # ncu DRAM traffic of each call's main kernel, while current
        tr = TRAFFIC.get(("around_b4_2k", n))
        if tr is not None and n in KERNELS and tr["src_sha"] == src_sha(KERNELS[n][1]):
            k["traffic"] = tr["bytes"]
            if n == dom:
                roof["traffic"] = tr["bytes"]
    roof["kernels"] = KERNELS.get(dom, ([], ""))[0]
    line = {"metric": METRIC, "value": M / (total_ms / 1e3), "unit": UNIT, "n_gpus": world,
            "steps": 1, "warmup": args.warmup, "ms_per_step": total_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "the calls around one step of the batch-4 L 2048 loop (step "
                                   f"1: {M} active rows, {N} stable rows), each timed alone",
                       "name": "around_b4_2k", "active_rows": M, "stable_rows": N},
            "roofline": roof, "kernels": kernels,
            "timing": "each call: median of 15 replays of a graph of 20 calls / 20"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- main

def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        if args.workload == "loop_b4_2k_128":
            return loop_reference_arm(args, rank)
        return reference_arm(args, rank)

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist

    if args.workload == "loop_b4_2k_128":
        return main_loop(args, rank, world, device, pg)
    if args.workload == "around_b4_2k":
        return main_around(args, rank, world, device, pg)

    import partial_attention_saliency_b300 as dl
    dl.load_library()

    wl = make_workload(args)
    s = wl.shape
    sets = [build_set(wl, s.seed + 1000 * (rank * 16 + 0), device)]
    # rotate input sets so that every step's inputs come from HBM, not L2
    n_sets = min(4, max(2, math.ceil(512e6 / set_bytes(sets[0]))))
    for i in range(1, n_sets):
        sets.append(build_set(wl, s.seed + 1000 * (rank * 16 + i), device))
    bf = Buffers(dl, wl, device)
    stream = torch.cuda.current_stream(device)
    masks_host = lock_schedule(wl, s.seed + 5) if wl.schedule else None
    masks = None if masks_host is None else [m.to(device) for m in masks_host]
    period = wl.schedule if wl.schedule else n_sets  # steps after which the inputs repeat
    lk = lambda i: None if masks is None else masks[i % wl.schedule]  # noqa: E731
    counts_per_step = []  # active rows of step i % period
    for i in range(period):
        run_step(dl, wl, bf, sets[i % n_sets], stream, locked=lk(i))
        torch.cuda.synchronize()
        counts_per_step.append(bf.count.cpu().tolist())
    assert int(bf.dev_status[0]) == 0, "device-side check failed"
    mean_counts = [sum(c[b] for c in counts_per_step) / period for b in range(s.B)]

    # ---------------------------------------------------------------- device-timed
    # A graph of S steps is replayed K / S times back to back: no host launch
    # gaps in the timed region, and consecutive kernels keep their
    # programmatic-launch overlap.  The graph is replayed once untimed (upload,
    # first launch); the K-step region is then timed repeatedly for about a
    # second and the median region is reported.  A second graph of the same S steps with
    # an external timing event between every two calls (events between calls
    # remove that overlap, so its per-call times are conservative) is then
    # replayed for the per-call breakdown.
    K = args.steps if args.steps is not None else wl.default_steps
    S = wl.schedule if wl.schedule else min(K, 250)
    K = max(S, (K // S) * S)
    cap = torch.cuda.Stream(device)
    g_warm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=cap):
        for i in range(args.warmup):
            run_step(dl, wl, bf, sets[i % n_sets], torch.cuda.current_stream(), locked=lk(i))
    g_timed = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_timed, stream=cap):
        for i in range(S):
            run_step(dl, wl, bf, sets[i % n_sets], torch.cuda.current_stream(), locked=lk(i))
    order = entries(wl)
    nev = len(order) + 1
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(nev)]
          for _ in range(S)]
    g_events = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_events, stream=cap):
        for i in range(S):
            run_step(dl, wl, bf, sets[i % n_sets], torch.cuda.current_stream(), ev[i],
                     locked=lk(i))
    clocks = ClockSampler(torch.cuda.current_device())
    g_warm.replay()
    torch.cuda.synchronize()
    if pg: pg.barrier()
    torch.cuda.synchronize()
    clocks.start()
    reps = time_regions(lambda: [g_timed.replay() for _ in range(K // S)], stream,
                        est_ms=0.1 * K, warm=g_timed.replay, min_seconds=args.min_seconds)
    clocks.stop()
    if pg: pg.barrier()
    g_events.replay()
    g_events.replay()
    torch.cuda.synchronize()
    assert int(bf.dev_status[0]) == 0, "device-side check failed"
    elapsed_ms = statistics.median(reps)
    per_entry = {n: 0.0 for n in order}
    for i in range(S):
        for j, n in enumerate(order):
            per_entry[n] += ev[i][j].elapsed_time(ev[i][j + 1])
    events_step_ms = sum(per_entry.values()) / S
    active_total = sum(sum(counts_per_step[i % period]) for i in range(S)) * (K // S)
    elapsed_ms, active_total = reduce_over_ranks(pg, elapsed_ms, active_total, device)
    value = active_total / (elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / K

    # ---------------------------------------------------------------- per entry point
    pk = peaks()
    work = algorithmic_work(wl, mean_counts)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    kernels = {}
    for n in order:
        if n == "dllm_confidence" and wl.conf is None:
            continue
        avg_ms = per_entry[n] / S
        w = work[n]
        gbs = w["bytes"] / (avg_ms / 1e3) / 1e9
        tfs = w["flops"] / (avg_ms / 1e3) / 1e12
        ai = w["flops"] / max(w["bytes"], 1)
        bound = "tensor" if w["flops"] > 0 and ai > ridge and n == "dllm_partial_attention" \
            else "hbm"
        kernels[n] = {"us": avg_ms * 1e3, "share": per_entry[n] / sum(per_entry.values()),
                      "alg_bytes": w["bytes"], "alg_flops": w["flops"], "GB/s": gbs,
                      "TFLOP/s": tfs, "bound": bound,
                      "frac": (tfs / pk["bf16_tflops"]) if bound == "tensor"
                      else gbs / pk["hbm_gbs"],
                      "kernels": KERNELS[n][0]}
    dom = max(kernels, key=lambda n: kernels[n]["us"])
    dk = kernels[dom]
    if dk["bound"] == "tensor":
        roof = {"bound": "tensor", "achieved": dk["TFLOP/s"], "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": dk["TFLOP/s"] / pk["bf16_tflops"],
                "frac_of_sustained": dk["TFLOP/s"] / pk["bf16_tflops_sustained"]}
    else:
        roof = {"bound": "hbm", "achieved": dk["GB/s"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": dk["GB/s"] / pk["hbm_gbs"]}
    tr = TRAFFIC.get((wl.name, dom))
    traffic = None
    if tr is not None and tr["src_sha"] == src_sha(KERNELS[dom][1]):
        traffic = tr["bytes"]
    roof.update({"traffic": traffic, "kernel": dom, "kernels": KERNELS[dom][0],
                 "peak_source": pk["source"] + " (burst)",
                 "alg_per_launch": work[dom]["flops"] if roof["unit"] == "TFLOP/s"
                 else work[dom]["bytes"],
                 "timing": "CUDA events around the call on the launching stream, averaged "
                           f"over the {S} steps of a replay of the step graph with an event "
                           "between every two calls"})

    # ---------------------------------------------------------------- end to end
    e2e = e2e_run(dl, wl, bf, sets, n_sets, stream, args, pg, device, K, lk, counts_per_step)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step,
            "latency_us_per_step": ms_per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.desc, "name": wl.name, "batch": s.B, "seq_len": s.L,
                       "heads": s.H, "head_dim": s.d, "hidden": s.D, "vocab": s.V,
                       "active_rows_per_step": sum(mean_counts),
                       "l2": f"{n_sets} rotating input sets of {set_bytes(sets[0]) / 1e6:.0f} MB "
                             f"each (> 126 MB L2)",
                       "parallelism": "replicas (one independent step per GPU)"},
            "roofline": roof, "kernels": kernels, "clocks": clocks.summary(),
            "gpu_launches": launches_per_step(wl, bf) * K,
            "timing": f"median of {len(reps)} timed regions of {K} steps ({K // S} replays "
                      f"of a {S}-step CUDA graph), after one untimed replay; region times "
                      f"{min(reps):.3f}-{max(reps):.3f} ms",
            "us_per_step_with_call_events": events_step_ms * 1e3, "e2e": e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb, _, _ = cpu_baseline(wl, sets[0]["host"], args.cpu_seconds, masks=masks_host)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def reduce_over_ranks(pg, elapsed_ms: float, units: float, device):
    """Whole-job figures of a replicated run: the slowest rank's time and the
    units all ranks processed (each rank steps its own batch rows)."""
    if pg is None:
        return elapsed_ms, units
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    u = torch.tensor([float(units)], dtype=torch.float64, device=device)
    pg.all_reduce(u, op=pg.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def e2e_run(dl, wl, bf, sets, n_sets, stream, args, pg, device, K_dev, lk, counts_per_step):
    """Same metric through the public API with pinned host buffers: H2D of the
    step's fresh inputs and D2H of its results inside the timed region."""
    host_in = ["cur", "k_new", "v_new", "q"] + (["logits"] if wl.conf is not None else [])
    pinned = [{k: sets[i]["host"][k].pin_memory() for k in host_in} for i in range(n_sets)]
    out_host = {
        "idx": torch.empty_like(bf.idx, device="cpu").pin_memory(),
        "count": torch.empty_like(bf.count, device="cpu").pin_memory(),
        "o": torch.empty_like(bf.o, device="cpu").pin_memory(),
        "lse": torch.empty_like(bf.lse, device="cpu").pin_memory(),
        "colsum": torch.empty_like(bf.colsum, device="cpu").pin_memory(),
        "score": torch.empty((wl.shape.B, wl.shape.L), dtype=torch.float32).pin_memory(),
        "argmax": torch.empty_like(bf.argmax, device="cpu").pin_memory(),
        "length": torch.empty_like(bf.length, device="cpu").pin_memory(),
    }
    out_dev = [("idx", bf.idx), ("count", bf.count), ("o", bf.o), ("lse", bf.lse),
               ("colsum", bf.colsum), ("score", None), ("argmax", bf.argmax),
               ("length", bf.length)]
    if wl.surelock:  # the previous step's logits stay on the device
        for k, t in (("lock_flags", bf.lock_flags), ("alen", bf.alen)):
            out_host[k] = torch.empty_like(t, device="cpu").pin_memory()
            out_dev.append((k, t))
    h2d = sum(t.numel() * t.element_size() for t in pinned[0].values())
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())

    def one(i):
        d = sets[i % n_sets]
        for k in host_in:
            dst = d[k][:, :pinned[i % n_sets][k].shape[1]] if k == "logits" else d[k]
            dst.copy_(pinned[i % n_sets][k], non_blocking=True)
        run_step(dl, wl, bf, d, stream, locked=lk(i))
        for k, src in out_dev:
            out_host[k].copy_(d["score"] if src is None else src, non_blocking=True)

    for i in range(max(args.warmup, 3)):
        one(i)
    K = max(min(K_dev // 40, 500), 10)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if pg: pg.barrier()
    a.record(stream)
    for i in range(K):
        one(i)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    active = sum(sum(counts_per_step[i % len(counts_per_step)]) for i in range(K))
    ms, active = reduce_over_ranks(pg, ms, active, device)
    return {"value": active / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K, "ms_per_step": ms / K}


if __name__ == "__main__":
    sys.exit(main())
