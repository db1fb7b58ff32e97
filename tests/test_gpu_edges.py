"""Degenerate sizes through the public calls on the GPU: no requests, no
tokens, no rows.  Each call returns cleanly with empty (or identity)
results and a clean status word."""
import numpy as np
import pytest
import torch

import paged_kv_cascade_gb300 as pkc

pytestmark = pytest.mark.gpu


def _empty_decode_inputs(hq=32, hkv=8, dtype=torch.bfloat16):
    q = torch.empty(0, hq, 128, dtype=dtype, device="cuda")
    kc = torch.zeros(4, 16, hkv, 128, dtype=dtype, device="cuda")
    bt = torch.empty(0, 1, dtype=torch.int32, device="cuda")
    sl = torch.empty(0, dtype=torch.int32, device="cuda")
    return q, kc, bt, sl


def test_no_requests_decode_and_cascade():
    q, kc, bt, sl = _empty_decode_inputs()
    ws = torch.empty(pkc.workspace_size(0, 32, 4, 4), dtype=torch.uint8, device="cuda")
    pkc.workspace_init(ws)
    o, lse = pkc.paged_decode_state(q, kc, kc, bt, sl, 0.1, ws)
    assert o.shape == (0, 32, 128) and lse.shape == (0, 32)
    buf = pkc.plan(np.zeros(0, np.int32), 4)
    pkc.plan_upload(buf, ws)
    pkc.paged_decode_state(q, kc, kc, bt, sl, 0.1, ws, plan_buf=buf)
    kp = torch.zeros(10, 8, 128, dtype=torch.bfloat16, device="cuda")
    o, lse = pkc.cascade_decode(q, kp, kp, [0, 10], [0, 0], kc, kc, bt, sl, 0.1, ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert o.shape == (0, 32, 128)
    assert pkc.device_status(ws) == pkc.PKC_OK


def test_requests_without_tokens_give_the_empty_state():
    # three requests with no cached tokens and no prefix: O = 0, LSE = -inf
    q = torch.randn(3, 32, 128, dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros(4, 16, 8, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.full((3, 2), -1, dtype=torch.int32, device="cuda")
    sl = torch.zeros(3, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkc.workspace_size(3, 32, 5, 4), dtype=torch.uint8, device="cuda")
    pkc.workspace_init(ws)
    for buf in (None, pkc.plan(np.zeros(3, np.int32), 5)):
        if buf is not None:
            pkc.plan_upload(buf, ws)
        o, lse = pkc.paged_decode_state(q, kc, kc, bt, sl, 0.1, ws, plan_buf=buf)
        torch.cuda.synchronize()
        assert pkc.device_status(ws) == pkc.PKC_OK
        assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_merge_of_no_rows():
    v = torch.empty(0, 32, 128, dtype=torch.float32, device="cuda")
    s = torch.empty(0, 32, dtype=torch.float32, device="cuda")
    vo, so = pkc.merge_state(v, s, v, s)
    vn, sn = pkc.merge_states(torch.empty(0, 16, 32, 128, device="cuda"), torch.empty(0, 16, 32, device="cuda"))
    torch.cuda.synchronize()
    assert vo.shape == (0, 32, 128) and vn.shape == (0, 32, 128)
