"""Multi-level cascade on the GPU: prefix groups as overlapping request ranges
(a prompt for every request, then prompts of request groups, then each
request's paged cache) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


def _problem(prefix_lens, ranges, lens, hq=32, hkv=8, dtype="bf16", seed=31):
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype,
                               prefix_lens=prefix_lens, prefix_groups=[1] * len(prefix_lens),
                               suffix=("list", lens), page_size=16, seed=seed, poison=True)
    p["ranges"] = ranges
    return p


def _run(p, num_ctas, prefix_splits=64):
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], num_ctas) if num_ctas else None
    ws = workspace_for(pkc, p, num_ctas=num_ctas or 0, prefix_splits=prefix_splits)
    if buf is not None:
        pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode_multilevel(
        d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], p["ranges"], d["k_cache"],
        d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    return o, lse, pkc.device_status(ws)


def _reference(p):
    a = oracle_args(p)
    a.pop("prefix_req_indptr")
    return oracle.attention_rows(p["q"], prefix_req_ranges=p["ranges"], **a)


@pytest.mark.parametrize("num_ctas", [None, 7])
def test_three_levels(num_ctas):
    # level 0: 300 tokens for all 12 requests; level 1: 200 tokens for 0-5,
    # 130 tokens (a ragged last tile) for 6-11; then ragged caches
    p = _problem([300, 200, 130], [(0, 12), (0, 6), (6, 12)],
                 [5, 0, 17, 300, 1, 64, 33, 129, 2, 16, 90, 7])
    o, lse, status = _run(p, num_ctas)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = _reference(p)
    compare(o, lse, ref_o, ref_lse)


def test_partial_overlaps_empty_group_and_uncovered_request():
    # groups overlap partly; group 2 has no tokens; request 11 is in no group
    p = _problem([260, 90, 0, 140], [(0, 11), (2, 7), (3, 9), (5, 11)],
                 [9, 40, 0, 3, 77, 16, 1, 250, 31, 8, 64, 12], hq=16, hkv=4, dtype="f16")
    o, lse, status = _run(p, 5)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = _reference(p)
    compare(o, lse, ref_o, ref_lse)


def test_disjoint_ranges_match_the_two_level_call():
    p = workloads.make_problem(batch=8, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[384, 200],
                               prefix_groups=[5, 3], suffix=("list", [3, 90, 16, 0, 41, 7, 300, 2]),
                               page_size=16, seed=9)
    d = to_device(p)
    ws = workspace_for(pkc, p, num_ctas=4)
    buf = pkc.plan(p["cache_seqlens"], 4)
    pkc.plan_upload(buf, ws)
    o2, lse2 = pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                  p["prefix_req_indptr"], d["k_cache"], d["v_cache"], d["block_table"],
                                  d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    ind = p["prefix_req_indptr"]
    om, lsem = pkc.cascade_decode_multilevel(
        d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], [(ind[0], ind[1]), (ind[1], ind[2])],
        d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    assert torch.equal(o2, om) and torch.equal(lse2, lsem)


def test_too_few_partial_slots_for_overlapping_groups_is_refused():
    p = _problem([130, 130, 130], [(0, 4), (0, 4), (0, 4)], [3, 5, 7, 9], hq=8, hkv=8)
    with pytest.raises(pkc.PkcError):
        _run(p, None, prefix_splits=2)  # three groups share every request: three slots needed
    o, lse, status = _run(p, None, prefix_splits=3)  # exactly enough: one block per group piece
    assert status == pkc.PKC_OK
    ref_o, ref_lse = _reference(p)
    compare(o, lse, ref_o, ref_lse)
