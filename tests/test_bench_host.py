"""Host logic of bench.py: workloads, algorithmic work per call, launch
counts and the lock schedule (no GPU needed)."""
import os
import sys
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _args(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.parse()
    finally:
        sys.argv = old


def _wl(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.make_workload(bench.parse())
    finally:
        sys.argv = old


def test_default_workload_is_the_128_step_loop():
    args = _args()
    assert args.workload == "loop_b4_2k_128" and args.steps is None
    sh = bench.workloads.LOOP_128
    assert (sh.B, sh.L, sh.prompt, sh.block, sh.T, sh.H, sh.d, sh.D, sh.V) == \
        (4, 2048, 1024, 32, 128, 32, 128, 4096, 126464)
    with pytest.raises(SystemExit):
        bench.make_workload(args)  # not a single-step workload


def test_the_1k_step_workload():
    wl = _wl("--workload", "step_1k")
    assert wl.name == "step_1k" and wl.conf == "window" and wl.n_active == 102
    s = wl.shape
    assert (s.B, s.L, s.H, s.d, s.D, s.V, s.win_start, s.logit_rows) == \
        (1, 1024, 32, 128, 4096, 126464, 512, 512)


def test_algorithmic_work_of_a_loop_step():
    # hand-derived: batch 4, 120 active rows each, generated-rows window (1024)
    sh = bench.workloads.LOOP_128
    w = bench.loop_step_work(sh, [120] * 4, 1024)
    M = 480
    assert w["dllm_saliency_select"]["bytes"] == 2 * 4 * 1024 * 4096 * 2 + 4 * 1024 * 8
    assert w["dllm_kv_scatter"]["bytes"] == M * 2 * 2 * 4096 * 2
    assert w["dllm_partial_attention"]["bytes"] == 2 * 4 * 2048 * 4096 * 2 + 2 * M * 4096 * 2 + M * 32 * 4
    assert w["dllm_partial_attention"]["flops"] == 4 * M * 2048 * 128 * 32
    assert w["dllm_confidence"]["bytes"] == M * (126464 * 2 + 12)
    # the whole-sequence window of every 4th step doubles the select's reads
    assert bench.loop_step_work(sh, [120] * 4, 0)["dllm_saliency_select"]["bytes"] == \
        2 * (2 * 4 * 1024 * 4096 * 2 + 4 * 1024 * 8)


def test_oracle_loop_baseline_on_the_small_loop():
    sh = bench.workloads.LOOP_SMALL
    pools = bench.workloads.make_loop_pools(sh)
    times, units = bench.oracle_loop_rows(sh, pools, 0, 0, steps_cap=sh.T)
    assert len(times) == sh.T
    assert units == int(bench.workloads.loop_counts(sh)[:, 0].sum())


def test_algorithmic_work_of_the_1k_step():
    # hand-derived for 102 active rows, bf16, window of 512 generated rows
    w = bench.algorithmic_work(_wl("--workload", "step_1k"), [102])
    assert w["dllm_saliency_select"]["bytes"] == 2 * 512 * 4096 * 2 + 512 * 8
    assert w["dllm_kv_scatter"]["bytes"] == 102 * 2 * 2 * 4096 * 2
    assert w["dllm_partial_attention"]["bytes"] == 2 * 1024 * 4096 * 2 + 2 * 102 * 4096 * 2 + 102 * 32 * 4
    assert w["dllm_partial_attention"]["flops"] == 4 * 102 * 1024 * 128 * 32  # 1.71 GFLOP
    assert w["dllm_confidence"]["bytes"] == 512 * (126464 * 2 + 12)          # 129.5 MB
    assert w["dllm_stable_prefix"]["bytes"] == 512 * 4


def test_workload_names_and_options():
    assert _wl("--workload", "batch8_2k", "--frac", "0.5", "--pattern", "cluster").name == \
        "batch8_2k_f50_cluster"
    assert _wl("--workload", "long_4k", "--locked", "0.9").name == "long_4k_locked90"
    wl = _wl("--workload", "long_4k_schedule", "--surelock")
    assert wl.name == "long_4k_schedule_surelock" and wl.surelock and wl.schedule == 64
    # the lock criterion with the confidence takes the confidence's place
    order = bench.entries(wl)
    assert order == bench.SURELOCK_ORDER and "dllm_confidence" not in order
    assert order.index("dllm_lock_criterion_conf") < order.index("dllm_stable_prefix") \
        < order.index("dllm_adaptive_prefix") == len(order) - 1
    assert bench.entries(_wl("--workload", "step_1k")) == bench.ENTRY_ORDER
    with pytest.raises(SystemExit):
        _wl("--workload", "step_1k", "--surelock")  # needs logits of every position


def test_launch_counts():
    wl = _wl("--workload", "step_1k")
    assert bench.launches_per_step(wl, types.SimpleNamespace(attn_split=False)) == 9
    assert bench.launches_per_step(wl, types.SimpleNamespace(attn_split=True)) == 10
    nolog = _wl("--workload", "batch8_2k")
    assert bench.launches_per_step(nolog, types.SimpleNamespace(attn_split=True)) == 8
    sl = _wl("--workload", "long_4k", "--surelock")
    assert bench.launches_per_step(sl, types.SimpleNamespace(attn_split=False)) == 11


def test_lock_schedule_is_nested_and_linear():
    wl = _wl("--workload", "long_4k_schedule")
    masks = bench.lock_schedule(wl, 5)
    assert len(masks) == 64
    Lw = wl.shape.Lw
    assert int(masks[0].sum()) == 0 and int(masks[-1].sum()) == round(0.9 * Lw)
    for a, b in zip(masks, masks[1:]):
        assert torch.all(b >= a)  # a locked position stays locked
    assert int(masks[32].sum()) == round(0.9 * 32 / 63 * Lw)
