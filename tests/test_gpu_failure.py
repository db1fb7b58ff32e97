"""Failure detection on the GPU without a fault: a bounded wait that runs
out records PKC_ERR_TIMEOUT and returns, and the context stays usable."""
import time

import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    ws = torch.empty(pkc.workspace_size(1, 1, 0, 0), dtype=torch.uint8, device="cuda")
    pkc.workspace_init(ws)
    t0 = time.time()
    assert pkc.selftest_wait_timeout(ws)  # the wait gave up instead of hanging
    elapsed = time.time() - t0
    assert 1.5 < elapsed < 60, elapsed   # the 2 s limit, not an early exit
    assert pkc.device_status(ws) == 6    # PKC_ERR_TIMEOUT, read (and cleared) on the host
    assert pkc.device_status(ws) == pkc.PKC_OK
    # the same context still runs a planned decode correctly
    p = workloads.make_problem(batch=5, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [3, 300, 17, 0, 64]),
                               page_size=16, seed=90, poison=True)
    d = to_device(p)
    buf = pkc.plan(p["cache_seqlens"], 6)
    ws2 = workspace_for(pkc, p, num_ctas=6, prefix_splits=0)
    pkc.plan_upload(buf, ws2)
    o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["cache_seqlens"], p["sm_scale"], ws2, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws2) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)
