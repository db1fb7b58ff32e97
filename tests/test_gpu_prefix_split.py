"""The prefix stage over fewer thread blocks than SMs.

In a planned cascade call the prefix runs next to the suffix decode.  When
its K/V tiles are shared by two or more 128-row query tiles it is bound by
the tensor pipe and gets SMs of its own (pkc_set_prefix_ctas, automatic): a
quarter of them next to a dynamically scheduled decode on the rest, or the
SMs a static plan leaves free; a caller may also cap its blocks.  The block
count changes how the flattened KV tiles are cut into pieces, so the states
must match the oracle for every count, and a call must give the same bits
timed (stage events, stages in order), untimed (the decode launched as the
prefix kernel's programmatic dependent, next to it) and replayed from a CUDA
graph."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, dev, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu

# the plan's CTAs (2 row tiles per KV head and a suffix much longer than the
# prefix's work: the automatic rule splits the SMs)
PLAN_CTAS = 148


@pytest.fixture
def prefix_ctas():
    yield pkc.set_prefix_ctas
    pkc.set_prefix_ctas(0)
    pkc.set_decode_schedule("dynamic")


@pytest.fixture(scope="module")
def gqa():
    # GQA 32/8: 64 requests x 4 heads = 256 rows per KV head on one
    # 1000-token prefix (8 KV tiles, the last ragged); lognormal suffixes
    w = dict(workloads.WORKLOADS["gqa_cascade_lb"])
    p = workloads.make_problem(**dict(w, batch=64, prefix_lens=[1000], prefix_groups=[64],
                                      suffix=("lognormal", 6.5, 1.0, 16, 4096), seed=91, poison=True))
    ref = oracle.attention_rows(p["q"], **oracle_args(p))
    return p, to_device(p), ref


def _cascade(p, d, buf, ws, o=None, lse=None):
    return pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                              p["prefix_req_indptr"], d["k_cache"], d["v_cache"], d["block_table"],
                              d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf, o=o, lse=lse)


@pytest.mark.parametrize("schedule,ctas", [("dynamic", PLAN_CTAS), ("static", 112)])
@pytest.mark.parametrize("n", [1, 5, 40, 0])
def test_prefix_block_counts_match_oracle(prefix_ctas, gqa, n, schedule, ctas):
    p, d, (ref_o, ref_lse) = gqa
    prefix_ctas(n)
    pkc.set_decode_schedule(schedule)
    buf = pkc.plan(p["cache_seqlens"], ctas)
    ws = workspace_for(pkc, p, num_ctas=ctas)
    pkc.plan_upload(buf, ws)
    o, lse = _cascade(p, d, buf, ws)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    compare(o, lse, ref_o, ref_lse)
    # the split the library chose: this prefix (2 row tiles per K/V tile, a
    # 4 MB K/V, work far below the suffix's) gets a quarter of the SMs next to
    # a dynamic decode, or the SMs a static plan leaves free
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if n > 0:
        want_p = n
    else:
        want_p = sms - (3 * sms) // 4 if schedule == "dynamic" else sms - ctas
    want_d = min(ctas, sms - want_p) if schedule == "dynamic" else ctas
    assert pkc.last_launch_blocks() == (want_p, want_d)


def test_automatic_split_same_bits_timed_untimed_and_graph(gqa):
    p, d, (ref_o, ref_lse) = gqa
    buf = pkc.plan(p["cache_seqlens"], PLAN_CTAS)
    ws = workspace_for(pkc, p, num_ctas=PLAN_CTAS)
    pkc.plan_upload(buf, ws)
    o = torch.empty_like(d["q"])
    lse = torch.empty(p["q"].shape[:2], dtype=torch.float32, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:  # torch creates the CUDA event on its first record
        e.record()
    pkc.set_stage_events(ev)
    _cascade(p, d, buf, ws, o, lse)
    torch.cuda.synchronize()
    timed = (o.clone(), lse.clone())
    assert all(ev[i].elapsed_time(ev[i + 1]) > 0 for i in range(3))
    o.zero_()
    _cascade(p, d, buf, ws, o, lse)  # the decode next to the prefix (launch chain)
    torch.cuda.synchronize()
    assert torch.equal(o, timed[0]) and torch.equal(lse, timed[1])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            _cascade(p, d, buf, ws, o, lse)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, timed[0]) and torch.equal(lse, timed[1])
    assert pkc.device_status(ws) == pkc.PKC_OK
    compare(o, lse, ref_o, ref_lse)


@pytest.mark.parametrize("n", [3, 40])
def test_multilevel_with_capped_prefix_blocks(prefix_ctas, n):
    # a 700-token prompt for all 24 requests, 300 and 170 tokens for two
    # halves; G = 8 (16/2 heads), so the top group has 2 row tiles per head
    lens = [5, 0, 17, 300, 1, 64, 33, 129, 2, 16, 90, 7, 450, 3, 61, 16, 0, 222, 9, 31, 128, 77, 1, 500]
    p = workloads.make_problem(batch=len(lens), hq=16, hkv=2, d=128, dtype="bf16",
                               prefix_lens=[700, 300, 170], prefix_groups=[1, 1, 1],
                               suffix=("list", lens), page_size=16, seed=92, poison=True)
    ranges = [(0, 24), (0, 12), (12, 24)]
    prefix_ctas(n)
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], 9)
    ws = workspace_for(pkc, p, num_ctas=9)
    pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode_multilevel(
        d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], ranges, d["k_cache"],
        d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    a = oracle_args(p)
    a.pop("prefix_req_indptr")
    ref_o, ref_lse = oracle.attention_rows(p["q"], prefix_req_ranges=ranges, **a)
    compare(o, lse, ref_o, ref_lse)


@pytest.mark.parametrize("n", [0, 7])
def test_paged_prefix_with_split_blocks(prefix_ctas, n):
    # prefixes kept in the page pool (NaN past their ends): a 700-token prompt
    # for 40 requests x 4 heads (2 row tiles per KV head), then 150 tokens for
    # the first half; a dynamic decode over 148 plan CTAs
    lens = [int(x) for x in (np.random.default_rng(93).integers(0, 1500, size=40))]
    p = workloads.make_problem(batch=40, hq=32, hkv=8, d=128, dtype="bf16",
                               prefix_lens=[700, 150], prefix_groups=[1, 1],
                               suffix=("list", lens), page_size=16, seed=93, poison=True)
    kc, vc, pages, page_indptr = workloads.pool_prefixes(p, 93)
    ranges = [(0, 40), (0, 20)]
    prefix_ctas(n)
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], PLAN_CTAS)
    ws = workspace_for(pkc, p, num_ctas=PLAN_CTAS)
    pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode_paged_prefix(
        d["q"], dev(pages), page_indptr, p["prefix_kv_indptr"], ranges, dev(kc), dev(vc),
        d["block_table"], d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    if n > 0:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        assert pkc.last_launch_blocks() == (n, min(PLAN_CTAS, sms - n))
    a = oracle_args(p)
    a.pop("prefix_req_indptr")
    ref_o, ref_lse = oracle.attention_rows(p["q"], prefix_req_ranges=ranges, **a)
    compare(o, lse, ref_o, ref_lse)
