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


def _wl(*argv):
    old = sys.argv
    sys.argv = ["bench.py", *argv]
    try:
        return bench.make_workload(bench.parse())
    finally:
        sys.argv = old


def test_default_workload_is_the_1k_step():
    wl = _wl()
    assert wl.name == "step_1k" and wl.conf == "window" and wl.n_active == 102
    s = wl.shape
    assert (s.B, s.L, s.H, s.d, s.D, s.V, s.win_start, s.logit_rows) == \
        (1, 1024, 32, 128, 4096, 126464, 512, 512)


def test_algorithmic_work_of_the_1k_step():
    # hand-derived for 102 active rows, bf16, window of 512 generated rows
    w = bench.algorithmic_work(_wl(), [102])
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
    assert bench.entries(wl) == bench.ENTRY_ORDER + bench.SURELOCK_ORDER
    assert bench.entries(_wl()) == bench.ENTRY_ORDER
    with pytest.raises(SystemExit):
        _wl("--workload", "step_1k", "--surelock")  # needs logits of every position


def test_launch_counts():
    wl = _wl()
    assert bench.launches_per_step(wl, types.SimpleNamespace(attn_split=False)) == 8
    assert bench.launches_per_step(wl, types.SimpleNamespace(attn_split=True)) == 9
    nolog = _wl("--workload", "batch8_2k")
    assert bench.launches_per_step(nolog, types.SimpleNamespace(attn_split=True)) == 7
    sl = _wl("--workload", "long_4k", "--surelock")
    assert bench.launches_per_step(sl, types.SimpleNamespace(attn_split=False)) == 12


def test_lock_schedule_is_nested_and_linear():
    wl = _wl("--workload", "long_4k_schedule")
    masks = bench.lock_schedule(wl, 5)
    assert len(masks) == 64
    Lw = wl.shape.Lw
    assert int(masks[0].sum()) == 0 and int(masks[-1].sum()) == round(0.9 * Lw)
    for a, b in zip(masks, masks[1:]):
        assert torch.all(b >= a)  # a locked position stays locked
    assert int(masks[32].sum()) == round(0.9 * 32 / 63 * Lw)
