"""prefix_attention_state and cascade_decode on the GPU against the oracle.

The cascade's result must equal plain attention over prefix u suffix (the
oracle computes that definition directly, not the cascade)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, dev, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


def _prefix(p):
    d = to_device(p)
    ws = workspace_for(pkc, p)
    o, lse = pkc.prefix_attention_state(d["q"], d["k_prefix"], d["v_prefix"],
                                        p["prefix_kv_indptr"], p["prefix_req_indptr"],
                                        p["sm_scale"], ws)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    return o, lse


def _cascade(p, num_ctas=None, alpha=1.0, beta=1.0):
    d = to_device(p)
    plan_buf = None
    if num_ctas:
        plan_buf = pkc.plan(p["cache_seqlens"], num_ctas, alpha=alpha, beta=beta)
    ws = workspace_for(pkc, p, num_ctas=num_ctas or 0)
    if plan_buf is not None:
        pkc.plan_upload(plan_buf, ws)
    o, lse = pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                p["prefix_req_indptr"], d["k_cache"], d["v_cache"],
                                d["block_table"], d["cache_seqlens"], p["sm_scale"], ws,
                                plan_buf=plan_buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    return o, lse


PREFIX_CASES = [
    # (hq, hkv, dtype, prefix_lens, groups, batch)
    (32, 32, "f16", [256], [4], 4),
    (32, 32, "f16", [1], [3], 3),                 # one prefix token
    (32, 8, "bf16", [300, 77], [40, 30], 70),     # ragged tails, 2 groups, 2 row tiles
    (8, 1, "bf16", [1000], [20], 25),             # g = 8, requests outside the group
    (16, 8, "f16", [129, 0, 512], [5, 2, 9], 16), # an empty prefix
]


@pytest.mark.parametrize("case", range(len(PREFIX_CASES)))
def test_prefix_state_small(case):
    hq, hkv, dtype, pl, groups, batch = PREFIX_CASES[case]
    p = workloads.make_problem(batch=batch, hq=hq, hkv=hkv, d=128, dtype=dtype, prefix_lens=pl,
                               prefix_groups=groups, suffix=("const", 0), page_size=16,
                               seed=20 + case)
    o, lse = _prefix(p)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, suffix=False))
    # the prefix state is float32 output: same tolerance as the final output
    compare(o, lse, ref_o, ref_lse)


def test_prefix_peaky():
    p = workloads.make_problem(batch=9, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[700],
                               prefix_groups=[9], suffix=("const", 0), page_size=16, seed=5,
                               q_scale=8.0)
    o, lse = _prefix(p)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, suffix=False))
    compare(o, lse, ref_o, ref_lse)


@pytest.mark.parametrize("num_ctas", [None, 148])
def test_cascade_tiny_workload_full(num_ctas):
    p = workloads.workload("tiny_cascade", poison=True)
    o, lse = _cascade(p, num_ctas)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


CASCADE_CASES = [
    # (hq, hkv, dtype, prefix_lens, groups, suffix lens, page_size)
    (32, 32, "f16", [256], [4], [32, 0, 1, 33], 16),
    (32, 8, "bf16", [1000, 300], [6, 5], [0, 5, 900, 17, 16, 2, 3000, 1, 0, 64, 65], 16),
    (16, 4, "f16", [130], [12], list(range(0, 120, 10)), 32),
]


@pytest.mark.parametrize("case", range(len(CASCADE_CASES)))
@pytest.mark.parametrize("num_ctas", [None, 5, 148])
def test_cascade_small(case, num_ctas):
    hq, hkv, dtype, pl, groups, lens, ps = CASCADE_CASES[case]
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype,
                               prefix_lens=pl, prefix_groups=groups, suffix=("list", lens),
                               page_size=ps, seed=30 + case, poison=True, extra_pages=3)
    o, lse = _cascade(p, num_ctas)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


def test_cascade_long_prompt_workload_every_row():
    """Batch 128, 32 heads, 32768-token shared prefix + 256-token suffixes,
    planned over 148 CTAs: all 4096 (request, head) rows against the oracle."""
    p = workloads.workload("cascade_long_prompt")
    o, lse = _cascade(p, 148)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


def test_gqa_cascade_lb_workload_every_row():
    """The load-balanced GQA cascade (batch 256, 4 prefixes x 8192 tokens,
    lognormal suffixes, 37 split requests): all 8192 rows, so every chunk of
    every split request reaches the comparison."""
    w = workloads.WORKLOADS["gqa_cascade_lb"]
    p = workloads.workload("gqa_cascade_lb")
    o, lse = _cascade(p, w["num_ctas"], w["alpha"], w["beta"])
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


def test_gqa_cascade_3level_workload_every_row():
    """The three-level workload as the benchmark runs it: its prefix (8 and 2
    row tiles per K/V tile) gets SMs of its own next to the decode."""
    w = workloads.WORKLOADS["gqa_cascade_3level"]
    p = workloads.workload("gqa_cascade_3level")
    d = to_device(p)
    C = w["num_ctas"]
    buf = pkc.plan(p["cache_seqlens"], C)
    ws = workspace_for(pkc, p, num_ctas=C)
    pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode_multilevel(
        d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], w["prefix_ranges"], d["k_cache"],
        d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    pb, db = pkc.last_launch_blocks()
    assert pb + db <= torch.cuda.get_device_properties(0).multi_processor_count
    a = oracle_args(p)
    a.pop("prefix_req_indptr")
    ref_o, ref_lse = oracle.attention_rows(p["q"], prefix_req_ranges=w["prefix_ranges"], **a)
    compare(o, lse, ref_o, ref_lse)


def test_gqa_cascade_paged_prefix_workload_every_row():
    """gqa_cascade_lb with its four 8192-token prefixes kept in the page pool
    (NaN past their ends) and read in place, as the benchmark line runs it."""
    w = workloads.WORKLOADS["gqa_cascade_lb"]
    p = workloads.workload("gqa_cascade_lb")
    kc, vc, pages, page_indptr = workloads.pool_prefixes(p, 5, poison=True)
    d = to_device(p)
    ind = p["prefix_req_indptr"]
    ranges = [(int(ind[j]), int(ind[j + 1])) for j in range(len(ind) - 1)]
    C = w["num_ctas"]
    buf = pkc.plan(p["cache_seqlens"], C)
    ws = workspace_for(pkc, p, num_ctas=C)
    pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode_paged_prefix(
        d["q"], dev(pages), page_indptr, p["prefix_kv_indptr"], ranges, dev(kc), dev(vc),
        d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


def test_workspace_reused_across_calls_and_problems():
    # The split-request arrival counters live in the workspace and must be
    # back at zero after every call: run three different problems through
    # one workspace, each checked against the oracle.
    probs = [
        workloads.make_problem(batch=9, hq=16, hkv=4, d=128, dtype="bf16", prefix_lens=[300],
                               prefix_groups=[9], suffix=("list", [700, 0, 5, 1300, 64, 65, 2, 900, 33]),
                               page_size=16, seed=61, poison=True),
        workloads.make_problem(batch=5, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[128, 256],
                               prefix_groups=[2, 3], suffix=("list", [4000, 3, 0, 2500, 17]),
                               page_size=16, seed=62, poison=True),
    ]
    B, Hq = 9, 32
    ws = torch.empty(pkc.workspace_size(B, Hq, 11, 64), dtype=torch.uint8, device="cuda")
    pkc.workspace_init(ws)
    for p in probs + [probs[0]]:
        d = to_device(p)
        plan_buf = pkc.plan(p["cache_seqlens"], 11)
        pkc.plan_upload(plan_buf, ws)
        o, lse = pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                    p["prefix_req_indptr"], d["k_cache"], d["v_cache"],
                                    d["block_table"], d["cache_seqlens"], p["sm_scale"], ws,
                                    plan_buf=plan_buf)
        torch.cuda.synchronize()
        assert pkc.device_status(ws) == pkc.PKC_OK
        ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
        compare(o, lse, ref_o, ref_lse)


def test_noncascade_decode_of_the_long_prompt_shape():
    """The pages' non-cascade baseline: the long-prompt problem (32768-token
    shared prefix, 256-token suffixes, 32 heads, fp16) at batch 6, decoded
    by pkc_paged_decode_state alone with every block table listing the shared
    prefix's pages and then the request's own.  It must give the cascade's
    answer: attention over prefix u suffix, every row against the oracle."""
    cfg = dict(workloads.WORKLOADS["cascade_long_prompt"], batch=6, prefix_groups=[6])
    p = workloads.make_problem(**cfg)
    n = workloads.noncascade_problem(p, 4)
    d = to_device(n)
    C = 148
    buf = pkc.plan(n["cache_seqlens"], C)
    ws = workspace_for(pkc, n, num_ctas=C, prefix_splits=0)
    pkc.plan_upload(buf, ws)
    o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["cache_seqlens"], n["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


@pytest.mark.parametrize("contraction", ["separate", "fused"])
def test_cascade_plan_never_uploaded_is_reported(contraction):
    """A planned cascade on a workspace that never received the plan (its
    plan words are zeros here): every kernel that reads the plan (decode,
    contraction, and the prefix kernel when it merges) checks the device
    plan's header against the call's host plan and reports PKC_ERR_PLAN.
    Once the plan is uploaded the same call matches the oracle."""
    p = workloads.make_problem(batch=12, hq=16, hkv=4, d=128, dtype="bf16", prefix_lens=[300],
                               prefix_groups=[12], suffix=("uniform", 1, 200), page_size=16,
                               seed=41)
    d = to_device(p)
    plan_buf = pkc.plan(p["cache_seqlens"], 8)
    nbytes = pkc.workspace_size(12, 16, 8, 64)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    args = (d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], p["prefix_req_indptr"],
            d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws)
    pkc.set_contraction(contraction)
    try:
        pkc.cascade_decode(*args, plan_buf=plan_buf)
        assert pkc.device_status(ws) == 7  # PKC_ERR_PLAN
        pkc.plan_upload(plan_buf, ws)
        o, lse = pkc.cascade_decode(*args, plan_buf=plan_buf)
        torch.cuda.synchronize()
        assert pkc.device_status(ws) == pkc.PKC_OK
    finally:
        pkc.set_contraction("separate")
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)
