"""The two schedules of a planned decode on the GPU: blocks running their
CTA's list of the plan (static) and blocks taking the plan's chunks from a
shared longest-first queue (dynamic).  Every chunk is computed the same way
wherever it runs, so the two must agree bit for bit, and both with the
oracle; the queue's counters must come back to zero after every launch."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


@pytest.fixture
def schedule():
    def force(which):
        pkc.set_decode_schedule(which)
    yield force
    pkc.set_decode_schedule("dynamic")
    pkc.set_decode_kernel("auto")


def _status_block(ws):
    return ws[:256].view(torch.int32).cpu().numpy()


CASES = [
    # (hq, hkv, dtype, kv dtype, page_size, lengths, CTAs)
    (32, 8, "bf16", None, 16, [3, 250, 16, 0, 1000, 7, 2400, 64, 31], 7),      # G 4, tensor cores
    (32, 32, "f16", None, 16, [1, 15, 16, 17, 100, 0, 513, 260], 6),           # G 1, 4 head groups
    (16, 2, "bf16", None, 8, [6, 7, 8, 49, 50, 333, 1200], 5),                 # G 8, 2 heads per block
    (32, 8, "f16", "e4m3", 16, [40, 900, 16, 3, 0, 777], 4),                   # fp8 cache
]


@pytest.mark.parametrize("which", ["auto", "simt"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_static_and_dynamic_agree_bit_for_bit(schedule, which, case):
    hq, hkv, dtype, kvd, ps, lens, C = CASES[case]
    if kvd and which == "simt":
        pytest.skip("an fp8 cache always takes the tensor-core kernel")
    pkc.set_decode_kernel(which)
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype, kv_dtype=kvd,
                               k_scale=0.5 if kvd else 1.0, v_scale=1.25 if kvd else 1.0,
                               prefix_lens=[], prefix_groups=[], suffix=("list", lens),
                               page_size=ps, seed=70 + case, poison=True)
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], C)
    ws = workspace_for(pkc, p, num_ctas=C, prefix_splits=0)
    pkc.plan_upload(buf, ws)

    def run():
        if kvd:
            o, lse = pkc.paged_decode_state_fp8(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                                d["cache_seqlens"], p["sm_scale"], ws,
                                                k_scale=p["k_scale"], v_scale=p["v_scale"], plan_buf=buf)
        else:
            o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                            d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
        torch.cuda.synchronize()
        return o.clone(), lse.clone()

    schedule("static")
    o_s, lse_s = run()
    assert pkc.device_status(ws) == pkc.PKC_OK
    schedule("dynamic")
    outs = [run() for _ in range(3)]  # the queue is reset between launches
    assert pkc.device_status(ws) == pkc.PKC_OK
    assert not _status_block(ws)[16:18].any()
    for o, lse in outs:
        assert torch.equal(o, o_s) and torch.equal(lse, lse_s)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o_s, lse_s, ref_o, ref_lse)


def test_dynamic_cascade_gqa_workload_rows():
    """The cascade at the GQA workload shape with the default (dynamic)
    decode against the static one: the same bits.  The prefix's SM share
    depends on the schedule, so it is pinned to every SM here."""
    w = dict(workloads.WORKLOADS["gqa_cascade_lb"])
    p = workloads.make_problem(**dict(w, batch=64, prefix_lens=[8192], prefix_groups=[64]))
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], 148)
    ws = workspace_for(pkc, p, num_ctas=148)
    pkc.plan_upload(buf, ws)
    res = {}
    pkc.set_prefix_ctas(torch.cuda.get_device_properties(0).multi_processor_count)
    try:
        for which in ("static", "dynamic"):
            pkc.set_decode_schedule(which)
            o, lse = pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                        p["prefix_req_indptr"], d["k_cache"], d["v_cache"],
                                        d["block_table"], d["cache_seqlens"], p["sm_scale"], ws,
                                        plan_buf=buf)
            torch.cuda.synchronize()
            assert pkc.device_status(ws) == pkc.PKC_OK
            res[which] = (o.clone(), lse.clone())
    finally:
        pkc.set_decode_schedule("dynamic")
        pkc.set_prefix_ctas(0)
    assert torch.equal(res["static"][0], res["dynamic"][0])
    assert torch.equal(res["static"][1], res["dynamic"][1])
    assert not _status_block(ws)[16:18].any()


def test_cascade_side_stream_and_timed_sequential_run_agree():
    """The cascade forks its prefix stage onto a side stream next to the
    decode; a call with stage events runs the stages in order on one stream.
    Both give the same bits, also replayed from a CUDA graph."""
    w = dict(workloads.WORKLOADS["gqa_cascade_lb"])
    p = workloads.make_problem(**dict(w, batch=32, prefix_lens=[2048], prefix_groups=[32]))
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], 40)
    ws = workspace_for(pkc, p, num_ctas=40)
    pkc.plan_upload(buf, ws)
    o = torch.empty_like(d["q"])
    lse = torch.empty(p["q"].shape[:2], dtype=torch.float32, device="cuda")

    def run():
        pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                           p["prefix_req_indptr"], d["k_cache"], d["v_cache"], d["block_table"],
                           d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf, o=o, lse=lse)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:  # torch creates the CUDA event on its first record
        e.record()
    pkc.set_stage_events(ev)
    run()
    torch.cuda.synchronize()
    seq = (o.clone(), lse.clone())
    assert all(ev[i].elapsed_time(ev[i + 1]) > 0 for i in range(3))
    o.zero_()
    run()  # forked
    torch.cuda.synchronize()
    assert torch.equal(o, seq[0]) and torch.equal(lse, seq[1])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run()
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, seq[0]) and torch.equal(lse, seq[1])
    assert pkc.device_status(ws) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


def test_binding_refuses_mismatched_cache_dtype_and_shapes():
    """A 1-byte e4m3 cache handed to the 16-bit decode would be read as twice
    its size: the binding refuses it, and mismatched shapes, in Python."""
    q = torch.zeros(2, 8, 128, dtype=torch.float16, device="cuda")
    kc8 = torch.zeros(4, 16, 2, 128, dtype=torch.uint8, device="cuda")
    kc = torch.zeros(4, 16, 2, 128, dtype=torch.float16, device="cuda")
    bt = torch.zeros(2, 4, dtype=torch.int32, device="cuda")
    sl = torch.zeros(2, dtype=torch.int32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(TypeError):
        pkc.paged_decode_state(q, kc8, kc8, bt, sl, 0.1, ws)
    with pytest.raises(TypeError):
        pkc.paged_decode_state_fp8(q, kc, kc, bt, sl, 0.1, ws)
    with pytest.raises(ValueError):
        pkc.paged_decode_state(q, kc, kc[:2], bt, sl, 0.1, ws)
    with pytest.raises(ValueError):
        pkc.paged_decode_state(q, kc, kc, bt[:1], sl, 0.1, ws)
    with pytest.raises(TypeError):
        pkc.paged_decode_state(q, kc, kc, bt.long(), sl, 0.1, ws)
