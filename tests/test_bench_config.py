"""Host-side configuration of bench.py's workloads (no GPU).

The benchmark lines run each workload with the plan the workload states: the
GQA cascade over 148 CTAs with alpha = beta = 1, the tiny cascade without a
plan, a smaller case of a workload keeping its prefix groups whole."""
import workloads

import bench


def test_gqa_workload_plans_over_148_ctas():
    cfg = bench.workload_cfg("gqa_cascade_lb")
    assert cfg["num_ctas"] == 148 and cfg["alpha"] == 1.0 and cfg["beta"] == 1.0
    assert cfg["prefix_lens"] == [8192] * 4 and cfg["prefix_groups"] == [64] * 4


def test_tiny_workload_runs_without_a_plan():
    cfg = bench.workload_cfg("tiny_cascade")
    assert cfg["num_ctas"] == 0
    assert bench.host_plan(None, [32] * 4, cfg["num_ctas"], cfg) is None


def test_smaller_case_keeps_whole_prefix_groups():
    cfg = bench.workload_cfg("gqa_cascade_lb", batch=100)
    # 64 requests share the first prefix, the next 36 the second
    assert cfg["batch"] == 100
    assert cfg["prefix_lens"] == [8192, 8192] and cfg["prefix_groups"] == [64, 36]
    cfg = bench.workload_cfg("cascade_long_prompt", batch=32)
    assert cfg["batch"] == 32 and cfg["prefix_groups"] == [32]


def test_effective_bytes_count_a_shared_prefix_once():
    p = workloads.workload("tiny_cascade")
    B, Hq, D = p["q"].shape
    kv_token = 2 * p["num_kv_heads"] * D * 2  # fp16 K and V, all heads
    want = (256 + 4 * 32) * kv_token + 2 * B * Hq * D * 2 + B * Hq * 4
    assert workloads.effective_bytes(p) == want
