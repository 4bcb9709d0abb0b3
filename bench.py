#!/usr/bin/env python3
"""Benchmark of the partial denoising step on B300.

One step = one pass of the whole hot path over one batch: saliency select,
KV scatter, partial attention with column sums, confidence over the window's
logit rows, longest stable prefix.  Default workload: batch 1, L = 1024
(512 prompt + 512 generated), 32 heads x 128, hidden 4096, vocabulary 126464
logits over the generated rows, ~10% of positions salient, bf16.

Metric: active query tokens per second (sum over batch rows of the active
count / step time); the line also carries the step latency, a per-entry-point
breakdown, the roofline of the dominant entry point, the clocks seen during
the timed region, the end-to-end figure (host buffers, copies inside the
timed region) and the float64 oracle timed on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica (weak scaling);
the timed region is bracketed by barriers and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "partial-step latency (µs) & active query tokens/s; % of B300 HBM/TC roofline"
UNIT = "active query tokens/s"
N_SETS = 4  # rotating input sets: 4 x ~175 MB keeps every step's inputs out of L2 (126 MB)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
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


class ClockSampler:
    """Polls NVML (SM clock, clock-event reasons) from a thread while running."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples = []
        self.period = period_s
        self.ok = False
        self.max_mhz = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.ok = True
        except Exception as e:  # noqa: BLE001
            self.err = repr(e)[:200]
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        nv = self.nv
        while not self._stop.is_set():
            try:
                mhz = nv.nvmlDeviceGetClockInfo(self.h, nv.NVML_CLOCK_SM)
                reasons = nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                self.samples.append((mhz, reasons))
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()

    def stop(self):
        if self._t is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "source": "nvml unavailable" if not self.ok else "nvml",
                    "error": getattr(self, "err", None)}
        mhz = [m for m, _ in self.samples]
        seen = 0
        for _, r in self.samples:
            seen |= int(r)
        names = [n for bit, n in self.REASONS.items() if seen & bit and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz, "reasons": names,
                "samples": len(mhz), "source": "nvml"}


# ----------------------------------------------------------------------------- workload

def workload_desc(s, n_active):
    return {"workload": f"partial step B{s.B} L{s.L} ({s.win_start} prompt + {s.Lw} gen) "
                        f"{s.H}x{s.d} heads, hidden {s.D}, vocab {s.V} over {s.logit_rows} gen rows, "
                        f"~{round(100 * n_active / s.L)}% salient",
            "batch": s.B, "seq_len": s.L, "heads": s.H, "head_dim": s.d, "hidden": s.D,
            "vocab": s.V, "logit_rows": s.logit_rows, "active_rows": n_active,
            "l2": f"{N_SETS} rotating input sets (~{N_SETS * 175} MB) > 126 MB L2",
            "parallelism": "replicas (one independent step per GPU)"}


def algorithmic_work(s, counts):
    """Algorithmic bytes / flops of each entry point for one step."""
    M = int(sum(counts))
    el = 2 if s.dtype == torch.bfloat16 else 4
    hd = s.H * s.d
    select_b = 2 * s.B * s.Lw * s.D * el + s.B * s.Lw * 8
    scatter_b = M * 2 * 2 * hd * el
    attn_b = 2 * s.B * s.L * hd * el + 2 * M * hd * el + M * s.H * 4 + s.B * s.H * s.L * 4
    attn_f = 4.0 * M * s.L * s.d * s.H
    conf_b = s.B * s.logit_rows * (s.V * el + 12)
    prefix_b = s.B * s.Lw * 4
    return {
        "dllm_saliency_select": {"bytes": select_b, "flops": 6.0 * s.B * s.Lw * s.D},
        "dllm_kv_scatter": {"bytes": scatter_b, "flops": 0.0},
        "dllm_partial_attention": {"bytes": attn_b, "flops": attn_f,
                                   "colsum_executed_flops": 2.0 * M * s.L * s.d * s.H},
        "dllm_confidence": {"bytes": conf_b, "flops": 0.0},
        "dllm_stable_prefix": {"bytes": prefix_b, "flops": 0.0},
    }


KERNELS = {  # kernels each entry point launches (for the ncu launch-list summary)
    "dllm_saliency_select": ["cos_rows_kernel", "compact_kernel"],
    "dllm_kv_scatter": ["kv_scatter_kernel"],
    "dllm_partial_attention": ["attention kernels (forward + column sums)"],
    "dllm_confidence": ["conf_partial_kernel", "conf_merge_kernel"],
    "dllm_stable_prefix": ["stable_prefix_kernel"],
}


def build_sets(s, device):
    sets = []
    for i in range(N_SETS):
        inp = workloads.make_step(s, seed=s.seed + 1000 * i)
        d = {k: inp[k].to(device) for k in ("cur", "prev", "k_cache", "v_cache", "k_new", "v_new",
                                            "q", "logits")}
        d["score"] = torch.full((s.B, s.L), float("inf"), device=device)
        d["start"] = torch.full((s.B,), s.win_start, dtype=torch.int32, device=device)
        d["host"] = inp
        sets.append(d)
    return sets


def run_step(dl, step, d, stream, events=None):
    """The five entry points in order; optional events bracket each call."""
    w = step.win_start
    ev = events
    if ev: ev[0].record(stream)
    dl.dllm_saliency_select(d["cur"][:, w:], d["prev"][:, w:], step.tau, idx_base=w,
                            cos_out=step.cos, idx_out=step.idx, count_out=step.count,
                            dev_status=step.dev_status, stream=stream)
    if ev: ev[1].record(stream)
    dl.dllm_kv_scatter(d["k_cache"], d["v_cache"], d["k_new"], d["v_new"], step.idx, step.count,
                       dev_status=step.dev_status, stream=stream)
    if ev: ev[2].record(stream)
    dl.dllm_partial_attention(d["q"], d["k_cache"], d["v_cache"], step.count, o_out=step.o,
                              lse_out=step.lse, colsum_out=step.colsum, ws=step.attn_ws,
                              dev_status=step.dev_status, stream=stream)
    if ev: ev[3].record(stream)
    dl.dllm_confidence(d["logits"], out_cols=step.L, conf_out=d["score"][:, w:],
                       argmax_out=step.argmax[:, w:], margin_out=step.margin[:, w:],
                       ws=step.conf_ws, dev_status=step.dev_status, stream=stream)
    if ev: ev[4].record(stream)
    dl.dllm_stable_prefix(d["score"], d["start"], step.tau_c, min_commit=True,
                          advance_start=False, len_out=step.length, dev_status=step.dev_status,
                          stream=stream)
    if ev: ev[5].record(stream)


ENTRY_ORDER = ["dllm_saliency_select", "dllm_kv_scatter", "dllm_partial_attention",
               "dllm_confidence", "dllm_stable_prefix"]
LAUNCHES_PER_STEP = 2 + 1 + 2 + 2 + 1


def cpu_baseline(s, seconds, steps_cap=None):
    """The float64 oracle, as it stands, on the host cores over full steps."""
    import numpy as np
    import oracle
    inp = workloads.make_step(s)
    d = {k: inp[k].double().numpy() for k in ("cur", "prev", "k_cache", "v_cache", "k_new",
                                               "v_new", "q", "logits")}
    times, active = [], 0
    t_begin = time.perf_counter()
    cpu_begin = time.process_time()
    while True:
        t0 = time.perf_counter()
        out = oracle.step(d["cur"], d["prev"], d["k_cache"], d["v_cache"], d["k_new"],
                          d["v_new"], d["q"], d["logits"], tau=s.tau, win_start=s.win_start,
                          score=np.full((s.B, s.L), np.inf), start=[s.win_start] * s.B,
                          tau_c=0.9)
        times.append(time.perf_counter() - t0)
        active = int(out["count"].sum())
        if steps_cap is not None and len(times) >= steps_cap:
            break
        if steps_cap is None and time.perf_counter() - t_begin >= seconds:
            break
    util = (time.process_time() - cpu_begin) / max(time.perf_counter() - t_begin, 1e-9)
    per_step = sum(times) / len(times)
    return {"value": active / per_step, "unit": UNIT, "cores": blas_threads(),
            "cpu_utilisation": round(util, 2), "kind": "oracle",
            "sample": f"{len(times)} full float64 oracle steps of the same workload "
                      f"({active} active rows each), {sum(times):.1f} s on the host",
            "s_per_step": per_step}, times, active


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


def reference_arm(args, rank):
    """`--impl reference`: the float64 oracle timed as the reference arm."""
    s = workloads.STEP_1K
    if rank != 0:
        return 0
    res, times, active = cpu_baseline(s, 0, steps_cap=args.warmup + args.steps)
    timed = times[args.warmup:]
    per = sum(timed) / len(timed)
    value = active / per
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_desc(s, active),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": res["cores"],
                             "kind": "oracle",
                             "sample": f"{len(timed)} timed full float64 oracle steps after "
                                       f"{args.warmup} warm-up steps"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
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

    import partial_attention_saliency_b300 as dl
    dl.load_library()

    s = workloads.STEP_1K
    sets = build_sets(s, device)
    step = dl.PartialStep(s.B, s.L, s.H, s.d, s.D, s.V, s.dtype, s.win_start, s.logit_rows,
                          s.tau, device=device)
    stream = torch.cuda.current_stream(device)
    counts_per_set = []
    for d in sets:
        run_step(dl, step, d, stream)
        torch.cuda.synchronize()
        counts_per_set.append(step.count.cpu().tolist())
    assert int(step.dev_status[0]) == 0, "device-side check failed"

    # ---------------------------------------------------------------- device-timed
    # W warm-up steps and the K timed steps are each captured as one CUDA graph
    # (no host launch gaps inside the timed region); external timing events
    # between the entry points of every timed step give the per-kernel times.
    K = args.steps
    cap = torch.cuda.Stream(device)
    g_warm = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_warm, stream=cap):
        for i in range(args.warmup):
            run_step(dl, step, sets[i % N_SETS], torch.cuda.current_stream())
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(6)]
          for _ in range(K)]
    g_timed = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_timed, stream=cap):
        for i in range(K):
            run_step(dl, step, sets[i % N_SETS], torch.cuda.current_stream(), ev[i])
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    g_warm.replay()
    torch.cuda.synchronize()
    if pg: pg.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start.record(stream)
    g_timed.replay()
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    if pg: pg.barrier()
    assert int(step.dev_status[0]) == 0, "device-side check failed"
    elapsed_ms = t_start.elapsed_time(t_end)
    per_entry = {n: 0.0 for n in ENTRY_ORDER}
    for i in range(K):
        for j, n in enumerate(ENTRY_ORDER):
            per_entry[n] += ev[i][j].elapsed_time(ev[i][j + 1])
    active_total = sum(sum(counts_per_set[i % N_SETS]) for i in range(K))
    if pg:
        t = torch.tensor([elapsed_ms], device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        elapsed_ms = float(t.item())
        a = torch.tensor([float(active_total)], device=device)
        pg.all_reduce(a, op=pg.ReduceOp.SUM)
        active_total = a.item()
    value = active_total / (elapsed_ms / 1e3)
    ms_per_step = elapsed_ms / K

    # ---------------------------------------------------------------- per entry point
    pk = peaks()
    work = algorithmic_work(s, counts_per_set[0])
    kernels = {}
    for n in ENTRY_ORDER:
        avg_ms = per_entry[n] / K
        w = work[n]
        gbs = w["bytes"] / (avg_ms / 1e3) / 1e9
        tfs = w["flops"] / (avg_ms / 1e3) / 1e12
        kernels[n] = {"us": avg_ms * 1e3, "share": per_entry[n] / sum(per_entry.values()),
                      "alg_bytes": w["bytes"], "alg_flops": w["flops"], "GB/s": gbs,
                      "TFLOP/s": tfs, "hbm_frac": gbs / pk["hbm_gbs"],
                      "kernels": KERNELS[n]}
    dom = max(ENTRY_ORDER, key=lambda n: per_entry[n])
    dk = kernels[dom]
    ai = work[dom]["flops"] / max(work[dom]["bytes"], 1)
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if work[dom]["flops"] > 0 and ai > ridge:
        roof = {"bound": "tensor", "achieved": dk["TFLOP/s"], "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": dk["TFLOP/s"] / pk["bf16_tflops"]}
    else:
        roof = {"bound": "hbm", "achieved": dk["GB/s"], "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": dk["GB/s"] / pk["hbm_gbs"]}
    roof.update({"traffic": None, "kernel": dom, "peak_source": pk["source"] + " (burst)",
                 "alg_per_launch": work[dom]["bytes"] if roof["unit"] == "GB/s" else work[dom]["flops"]})

    # ---------------------------------------------------------------- end to end
    e2e = e2e_run(dl, s, step, sets, stream, args, pg, device)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_per_step,
            "latency_us_per_step": ms_per_step * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_desc(s, sum(counts_per_set[0])),
            "roofline": roof, "kernels": kernels, "clocks": clocks.summary(),
            "gpu_launches": LAUNCHES_PER_STEP * K, "timing": "K steps replayed as one CUDA graph", "e2e": e2e}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cb, _, _ = cpu_baseline(s, args.cpu_seconds)
        cb.pop("s_per_step", None)
        line["cpu_baseline"] = cb
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()
    return 0


def e2e_run(dl, s, step, sets, stream, args, pg, device):
    """Same metric through the public API with pinned host buffers: H2D of the
    step's fresh inputs and D2H of its results inside the timed region."""
    host_in = ["cur", "k_new", "v_new", "q", "logits"]
    pinned = [{k: sets[i]["host"][k].pin_memory() for k in host_in} for i in range(N_SETS)]
    out_host = {
        "idx": torch.empty_like(step.idx, device="cpu").pin_memory(),
        "count": torch.empty_like(step.count, device="cpu").pin_memory(),
        "o": torch.empty_like(step.o, device="cpu").pin_memory(),
        "lse": torch.empty_like(step.lse, device="cpu").pin_memory(),
        "colsum": torch.empty_like(step.colsum, device="cpu").pin_memory(),
        "score": torch.empty((s.B, s.L), dtype=torch.float32).pin_memory(),
        "argmax": torch.empty_like(step.argmax, device="cpu").pin_memory(),
        "length": torch.empty_like(step.length, device="cpu").pin_memory(),
    }
    h2d = sum(t.numel() * t.element_size() for t in pinned[0].values())
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())

    def one(i):
        d = sets[i % N_SETS]
        for k in host_in:
            d[k].copy_(pinned[i % N_SETS][k], non_blocking=True)
        run_step(dl, step, d, stream)
        for k, src in (("idx", step.idx), ("count", step.count), ("o", step.o),
                       ("lse", step.lse), ("colsum", step.colsum), ("score", d["score"]),
                       ("argmax", step.argmax), ("length", step.length)):
            out_host[k].copy_(src, non_blocking=True)

    for i in range(max(args.warmup, 3)):
        one(i)
    K = max(args.steps // 4, 10)
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
    if pg:
        t = torch.tensor([ms], device=device)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        ms = float(t.item())
    active = int(step.count.sum().item()) * (pg.get_world_size() if pg else 1)
    return {"value": active * K / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": K, "ms_per_step": ms / K}


if __name__ == "__main__":
    sys.exit(main())
