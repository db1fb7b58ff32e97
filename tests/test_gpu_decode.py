"""paged_decode_state on the GPU against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


def _run(p, num_ctas=None):
    d = to_device(p)
    plan_buf = None
    if num_ctas:
        plan_buf = pkc.plan(p["cache_seqlens"], num_ctas)
    ws = workspace_for(pkc, p, num_ctas=num_ctas or 0, prefix_splits=0)
    if plan_buf is not None:
        pkc.plan_upload(plan_buf, ws)
    o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["cache_seqlens"], p["sm_scale"], ws, plan_buf=plan_buf)
    torch.cuda.synchronize()
    status = pkc.device_status(ws)
    return o, lse, status


CASES = [
    # (hq, hkv, dtype, page_size, lengths)
    (32, 32, "f16", 16, [1, 15, 16, 17, 100, 0, 513]),
    (32, 8, "bf16", 16, [3, 250, 16, 0, 1000, 7]),
    (8, 4, "f16", 32, [30, 32, 70]),            # the worked example's lengths
    (16, 2, "bf16", 7, [6, 7, 8, 49, 50, 333]),  # page size not a power of two
    (4, 4, "bf16", 1, [1, 5, 0]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("num_ctas", [None, 3, 40])
def test_decode_small(case, num_ctas):
    hq, hkv, dtype, ps, lens = CASES[case]
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype,
                               prefix_lens=[], prefix_groups=[], suffix=("list", lens),
                               page_size=ps, seed=10 + case, extra_pages=5, poison=True)
    o, lse, status = _run(p, num_ctas)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_decode_gqa_group_sizes(g):
    lens = [200, 37, 1]
    p = workloads.make_problem(batch=3, hq=8 * g, hkv=8, d=128, dtype="bf16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", lens), page_size=16, seed=g,
                               poison=True)
    o, lse, status = _run(p, 5)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_decode_peaky_softmax():
    # q scaled x8: sharp softmax, so a wrong weight shows up in O
    p = workloads.make_problem(batch=6, hq=32, hkv=8, d=128, dtype="f16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [300, 1, 64, 65, 900, 17]),
                               page_size=16, seed=77, q_scale=8.0, poison=True)
    o, lse, status = _run(p, 7)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_decode_paged_decode_workload_every_row():
    """Batch 64, 32 heads, fp16, lengths U{512..4096}: every row against the
    oracle, planned over 148 CTAs and without a plan."""
    p = workloads.workload("paged_decode")
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    for num_ctas in (148, None):
        o, lse, status = _run(p, num_ctas)
        assert status == pkc.PKC_OK
        compare(o, lse, ref_o, ref_lse)


def test_decode_all_empty():
    p = workloads.make_problem(batch=3, hq=4, hkv=4, d=128, dtype="f16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [0, 0, 0]), page_size=16,
                               seed=1, extra_pages=1)
    for nc in (None, 2):
        o, lse, status = _run(p, nc)
        assert status == pkc.PKC_OK
        assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_decode_bad_page_id_is_reported_not_faulted():
    p = workloads.make_problem(batch=2, hq=4, hkv=4, d=128, dtype="f16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [40, 20]), page_size=16, seed=2)
    p["block_table"] = p["block_table"].copy()
    p["block_table"][0, 1] = -1          # inside the used range of request 0
    p["block_table"][1, 0] = 10 ** 6     # out of range
    o, lse, status = _run(p, None)
    assert status == 4  # PKC_ERR_BLOCK_TABLE
    # the status word was cleared by the read
    ws = workspace_for(pkc, p, prefix_splits=0)
    assert pkc.device_status(ws) == pkc.PKC_OK


def test_decode_plan_that_does_not_match_lengths_is_reported():
    p = workloads.make_problem(batch=3, hq=4, hkv=4, d=128, dtype="f16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [40, 20, 5]), page_size=16,
                               seed=3)
    d = to_device(p)
    plan_buf = pkc.plan([40, 25, 5], 4)  # request 1 claims 25 tokens, cache has 20
    ws = workspace_for(pkc, p, num_ctas=4, prefix_splits=0)
    pkc.plan_upload(plan_buf, ws)
    pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                           d["cache_seqlens"], p["sm_scale"], ws, plan_buf=plan_buf)
    assert pkc.device_status(ws) == 7


@pytest.mark.parametrize("hq", [4, 8])  # G = 1: CUDA-core decode; G = 2: tensor-core decode
def test_decode_plan_never_uploaded_is_reported(hq):
    """A planned call on a workspace that never received the plan (no
    pkc_plan_upload; its plan words are zeros here): the decode and the
    contraction compare the device plan's header with the call's host plan
    and report PKC_ERR_PLAN instead of following the words.  Once the plan
    is uploaded the same call is exact."""
    p = workloads.make_problem(batch=3, hq=hq, hkv=4, d=128, dtype="f16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [40, 20, 5]), page_size=16,
                               seed=3)
    d = to_device(p)
    plan_buf = pkc.plan([40, 20, 5], 4)
    ws = torch.zeros(pkc.workspace_size(3, hq, 4, 0), dtype=torch.uint8, device="cuda")
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws)
    pkc.paged_decode_state(*args, plan_buf=plan_buf)
    assert pkc.device_status(ws) == 7  # PKC_ERR_PLAN
    pkc.plan_upload(plan_buf, ws)
    o, lse = pkc.paged_decode_state(*args, plan_buf=plan_buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)
