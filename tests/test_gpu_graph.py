"""cascade_decode captured once in a CUDA graph and replayed every step.

The plan runs on the host each generation step and is copied into the
workspace outside the graph; the captured call reads every per-step quantity
(chunk lists, partial slots, lengths) from device memory (FlashInfer MLSys'25
notes, A3: plan per step on the CPU, not captured; run captured, fixed grid,
fixed workspace pointers).  Three steps with different suffix lengths replay
the same graph and must each match the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, oracle_args, to_device

pytestmark = pytest.mark.gpu


def test_captured_cascade_replays_with_new_lengths_each_step():
    B, Hq, Hkv, C, ps = 12, 32, 8, 19, 16
    max_len = 3000
    base = workloads.make_problem(batch=B, hq=Hq, hkv=Hkv, d=128, dtype="bf16",
                                  prefix_lens=[500, 700], prefix_groups=[5, 7],
                                  suffix=("const", max_len), page_size=ps, seed=71)
    d = to_device(base)
    ws = torch.empty(pkc.workspace_size(B, Hq, C, 64), dtype=torch.uint8, device="cuda")
    pkc.workspace_init(ws)
    plan_buf = pkc.plan(base["cache_seqlens"], C)
    pkc.plan_upload(plan_buf, ws)
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    def run():
        pkc.cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], base["prefix_kv_indptr"],
                           base["prefix_req_indptr"], d["k_cache"], d["v_cache"],
                           d["block_table"], d["cache_seqlens"], base["sm_scale"], ws,
                           plan_buf=plan_buf, o=o, lse=lse, stream=stream)

    with torch.cuda.stream(stream):
        run()  # warm-up outside capture (tensor-map encoding, kernel attributes)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
    rng = np.random.default_rng(5)
    for step in range(3):
        lens = rng.integers(0, max_len + 1, size=B).astype(np.int32)
        lens[step] = 0
        p = dict(base)
        p["cache_seqlens"] = lens
        # the host plans the new lengths and uploads them outside the graph
        new_plan = pkc.plan(lens, C)
        with torch.cuda.stream(stream):
            d["cache_seqlens"].copy_(torch.from_numpy(lens), non_blocking=False)
            pkc.plan_upload(new_plan, ws, stream=stream)
            g.replay()
        stream.synchronize()
        assert pkc.device_status(ws) == pkc.PKC_OK
        ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
        compare(o, lse, ref_o, ref_lse)
