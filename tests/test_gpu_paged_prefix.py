"""Cascade with the shared prefixes kept in the page pool (read in place
through a page list) against the oracle over the same tokens held
contiguously."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, dev, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


def _pooled(prefix_lens, ranges, lens, ps, hq=32, hkv=8, dtype="bf16", seed=41):
    """A problem whose prefixes also live in pages of the cache pool: the
    suffix pages come first, the prefix pages are appended in a seeded order,
    and every slot past a prefix's end in its last page is NaN."""
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype,
                               prefix_lens=prefix_lens, prefix_groups=[1] * len(prefix_lens),
                               suffix=("list", lens), page_size=ps, seed=seed, poison=True)
    kc, vc, pages, page_indptr = workloads.pool_prefixes(p, seed)
    return p, dict(k_cache=kc, v_cache=vc, pages=pages, page_indptr=page_indptr, ranges=ranges)


def _run(p, pool, num_ctas):
    d = to_device(p)
    kc, vc = dev(pool["k_cache"]), dev(pool["v_cache"])
    buf = pkc.plan(p["cache_seqlens"], num_ctas) if num_ctas else None
    ws = workspace_for(pkc, p, num_ctas=num_ctas or 0)
    if buf is not None:
        pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode_paged_prefix(
        d["q"], dev(pool["pages"]), pool["page_indptr"], p["prefix_kv_indptr"], pool["ranges"], kc, vc,
        d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    return o, lse, pkc.device_status(ws)


def _reference(p, ranges):
    a = oracle_args(p)
    a.pop("prefix_req_indptr")
    return oracle.attention_rows(p["q"], prefix_req_ranges=ranges, **a)


@pytest.mark.parametrize("ps", [16, 32, 8])
def test_paged_prefix_two_levels(ps):
    # a shared 300-token prompt for all, then 200 / 77 tokens for two groups
    p, pool = _pooled([300, 200, 77], [(0, 10), (0, 6), (6, 10)],
                      [5, 0, 17, 40, 1, 64, 33, 130, 2, 16], ps)
    o, lse, status = _run(p, pool, 6)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = _reference(p, pool["ranges"])
    compare(o, lse, ref_o, ref_lse)


def test_paged_prefix_mha_fp16_matches_contiguous_call():
    p, pool = _pooled([520], [(0, 6)], [9, 40, 0, 3, 77, 16], 16, hq=16, hkv=16, dtype="f16", seed=42)
    o, lse, status = _run(p, pool, None)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = _reference(p, pool["ranges"])
    compare(o, lse, ref_o, ref_lse)
    # the contiguous two-level call on the same tokens agrees to rounding
    d = to_device(p)
    ws = workspace_for(pkc, p)
    o2, lse2 = pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                  [0, 6], d["k_cache"], d["v_cache"], d["block_table"],
                                  d["cache_seqlens"], p["sm_scale"], ws)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(o.float() - o2.float())).item() <= 2e-3


def test_paged_prefix_bad_page_is_reported():
    p, pool = _pooled([64, 64], [(0, 2), (2, 4)], [3, 5, 7, 9], 16, hq=8, hkv=8)
    pool["pages"] = pool["pages"].copy()
    pool["pages"][1] = 10 ** 6
    _, _, status = _run(p, pool, None)
    assert status == 4  # PKC_ERR_BLOCK_TABLE, reported, no fault
