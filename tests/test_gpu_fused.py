"""The contraction fused into the attention kernels against the standalone
contraction kernel.

Fused, the kernel that writes the last source of a (request,
KV head) pair -- a chunk's partial state, a cascade's suffix state or a
prefix piece -- merges the pair's sources itself.  One routine merges a
row's sources in the same order either way, so the two must agree bit for
bit, whichever kernel happens to arrive last; both are also checked against
the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, dev, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


@pytest.fixture
def contraction():
    yield pkc.set_contraction
    pkc.set_contraction("separate")


def _cascade(p, num_ctas, ws=None):
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], num_ctas) if num_ctas else None
    ws = workspace_for(pkc, p, num_ctas=num_ctas or 0) if ws is None else ws
    if buf is not None:
        pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                p["prefix_req_indptr"], d["k_cache"], d["v_cache"], d["block_table"],
                                d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    return o, lse


def _decode(p, num_ctas, fp8=False):
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], num_ctas)
    ws = workspace_for(pkc, p, num_ctas=num_ctas, prefix_splits=0)
    pkc.plan_upload(buf, ws)
    if fp8:
        o, lse = pkc.paged_decode_state_fp8(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                            d["cache_seqlens"], p["sm_scale"], ws, k_scale=p["k_scale"],
                                            v_scale=p["v_scale"], plan_buf=buf)
    else:
        o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                        d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    return o, lse


def _both(contraction, run):
    contraction("separate")
    a = run()
    contraction("fused")
    b = run()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]), "fused and standalone contraction differ"
    return b


CASCADES = [
    # (hq, hkv, dtype, prefix_lens, groups, suffix lens, page_size, num_ctas)
    (32, 32, "f16", [256], [4], [32, 0, 1, 33], 16, None),
    (32, 32, "f16", [256], [4], [32, 0, 1, 33], 16, 148),
    (32, 8, "bf16", [1000, 300], [6, 5], [0, 5, 900, 17, 16, 2, 3000, 1, 0, 64, 65], 16, 5),
    (32, 8, "bf16", [1000, 300], [6, 3], [0, 5, 900, 17, 16, 2, 3000, 1, 0, 64, 65], 16, 148),  # 2 outside
    (16, 4, "f16", [130], [12], list(range(0, 120, 10)), 32, 7),
    (64, 8, "bf16", [4100], [40], [3 * (i % 11) for i in range(40)], 16, 64),   # g = 8, 3 row tiles
    (8, 8, "f16", [0, 700], [3, 4], [0, 0, 50, 600, 1, 0, 9], 16, 11),           # an empty prefix
]


@pytest.mark.parametrize("case", range(len(CASCADES)))
def test_fused_cascade_equals_standalone_and_oracle(contraction, case):
    hq, hkv, dtype, pl, groups, lens, ps, nc = CASCADES[case]
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype, prefix_lens=pl,
                               prefix_groups=groups, suffix=("list", lens), page_size=ps,
                               seed=90 + case, poison=True, extra_pages=3)
    o, lse = _both(contraction, lambda: _cascade(p, nc))
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


DECODES = [
    # (hq, hkv, dtype, lens, num_ctas)
    (32, 8, "bf16", [900, 0, 33, 4000, 17, 250, 0, 1], 148),
    (32, 32, "f16", [5, 1200, 64, 2, 0, 3000], 37),
    (16, 2, "f16", [700, 3, 2100, 64, 16], 9),
    (64, 8, "bf16", [129, 4096, 1], 148),
]


@pytest.mark.parametrize("case", range(len(DECODES)))
def test_fused_planned_decode_equals_standalone_and_oracle(contraction, case):
    hq, hkv, dtype, lens, nc = DECODES[case]
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype, prefix_lens=[],
                               prefix_groups=[], suffix=("list", lens), page_size=16, seed=110 + case,
                               poison=True, extra_pages=2)
    o, lse = _both(contraction, lambda: _decode(p, nc))
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_fused_fp8_decode_equals_standalone(contraction):
    p = workloads.make_problem(batch=6, hq=32, hkv=8, d=128, dtype="f16", kv_dtype="e4m3", k_scale=0.5,
                               v_scale=1.25, prefix_lens=[], prefix_groups=[],
                               suffix=("list", [3, 250, 16, 0, 1000, 7]), page_size=16, seed=120,
                               extra_pages=3, poison=True)
    o, lse = _both(contraction, lambda: _decode(p, 40, fp8=True))
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_fused_multilevel_and_paged_prefix_equal_standalone(contraction):
    p = workloads.make_problem(batch=10, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[300, 200, 500],
                               prefix_groups=[1, 1, 1], suffix=("list", [0, 40, 300, 7, 16, 900, 1, 2, 64, 0]),
                               page_size=16, seed=121, poison=True)
    ranges = [(0, 10), (0, 4), (4, 9)]
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], 13)
    ws = workspace_for(pkc, p, num_ctas=13)
    pkc.plan_upload(buf, ws)

    def multilevel():
        o, lse = pkc.cascade_decode_multilevel(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                               ranges, d["k_cache"], d["v_cache"], d["block_table"],
                                               d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
        torch.cuda.synchronize()
        assert pkc.device_status(ws) == pkc.PKC_OK
        return o, lse

    o, lse = _both(contraction, multilevel)
    a = oracle_args(p)
    a.pop("prefix_req_indptr")
    ref_o, ref_lse = oracle.attention_rows(p["q"], prefix_req_ranges=ranges, **a)
    compare(o, lse, ref_o, ref_lse)

    q = workloads.make_problem(batch=7, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[300, 77],
                               prefix_groups=[4, 3], suffix=("list", [5, 0, 700, 16, 33, 2, 1]),
                               page_size=16, seed=122, poison=True)
    kc, vc, pages, page_indptr = workloads.pool_prefixes(q, 3, poison=True)
    dq = to_device(q)
    ind = q["prefix_req_indptr"]
    rr = [(int(ind[j]), int(ind[j + 1])) for j in range(len(ind) - 1)]
    wq = workspace_for(pkc, q, num_ctas=17)
    bq = pkc.plan(q["cache_seqlens"], 17)
    pkc.plan_upload(bq, wq)
    kcd, vcd, pgd = dev(kc), dev(vc), dev(pages)

    def paged():
        o, lse = pkc.cascade_decode_paged_prefix(dq["q"], pgd, page_indptr, q["prefix_kv_indptr"], rr, kcd, vcd,
                                                 dq["block_table"], dq["cache_seqlens"], q["sm_scale"], wq,
                                                 plan_buf=bq)
        torch.cuda.synchronize()
        assert pkc.device_status(wq) == pkc.PKC_OK
        return o, lse

    o, lse = _both(contraction, paged)
    ref_o, ref_lse = oracle.attention_rows(q["q"], **oracle_args(q))
    compare(o, lse, ref_o, ref_lse)


def test_fused_headline_workload_equals_standalone(contraction):
    """The load-balanced GQA cascade at full size (batch 256, 37 split
    requests, prefix on its own SMs next to the decode): fused and standalone
    contraction give the same bits."""
    w = workloads.WORKLOADS["gqa_cascade_lb"]
    p = workloads.workload("gqa_cascade_lb")
    _both(contraction, lambda: _cascade(p, w["num_ctas"]))


def test_fused_counters_start_from_zero_every_call(contraction):
    """Each fused call zeroes its counters, so a workspace serves calls of
    different shapes back to back, and a repeated call gives the same bits."""
    contraction("fused")
    a = workloads.make_problem(batch=9, hq=16, hkv=4, d=128, dtype="bf16", prefix_lens=[300], prefix_groups=[9],
                               suffix=("list", [700, 0, 5, 1300, 64, 65, 2, 900, 33]), page_size=16, seed=61,
                               poison=True)
    b = workloads.make_problem(batch=5, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[128, 256],
                               prefix_groups=[2, 3], suffix=("list", [4000, 3, 0, 2500, 17]), page_size=16,
                               seed=62, poison=True)
    ws = torch.empty(pkc.workspace_size(9, 32, 11, 64), dtype=torch.uint8, device="cuda")
    pkc.workspace_init(ws)
    first = _cascade(a, 11, ws)
    for p in (b, a, b):
        o, lse = _cascade(p, 11, ws)
        ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
        compare(o, lse, ref_o, ref_lse)
    again = _cascade(a, 11, ws)
    assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])
