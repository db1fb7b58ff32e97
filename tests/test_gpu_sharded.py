"""KV-sequence sharding on one GPU: the ranks' parts of the keys computed one
after another on the same device with the library's calls, their float32
states stacked as an all-gather would deliver them, and merged by the
library's n-ary merge into q's dtype.  The result must be the oracle's
attention over the whole key set ("Attention States and Recursive
Attention", Applications)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from paged_kv_cascade_gb300.sharded import kv_shard_range, kv_sharded_cascade_decode, merge_gathered
from pkc_testing import compare, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


def _part_state(part, o_out, lse_out, num_ctas):
    d = to_device(part)
    k_pre = d["k_prefix"] if d["k_prefix"] is not None else torch.empty((0, part["num_kv_heads"], 128),
                                                                        dtype=d["q"].dtype, device="cuda")
    ws = workspace_for(pkc, part, num_ctas=num_ctas or 0)
    buf = None
    if num_ctas:
        buf = pkc.plan(part["cache_seqlens"], num_ctas)
        pkc.plan_upload(buf, ws)
    pkc.cascade_decode_state(d["q"], k_pre, d["v_prefix"] if d["v_prefix"] is not None else k_pre,
                             part["prefix_kv_indptr"], part["prefix_req_indptr"], d["k_cache"], d["v_cache"],
                             d["block_table"], d["cache_seqlens"], part["sm_scale"], ws, plan_buf=buf,
                             o=o_out, lse=lse_out)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK


@pytest.mark.parametrize("world,num_ctas", [(2, None), (3, 17), (5, 148)])
def test_sharded_cascade_on_one_device_matches_the_oracle(world, num_ctas):
    p = workloads.make_problem(batch=9, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[700, 130],
                               prefix_groups=[5, 3], suffix=("list", [0, 5, 900, 17, 16, 2, 3000, 1, 64]),
                               page_size=16, seed=81, poison=True, extra_pages=3)
    B, Hq, D = p["q"].shape
    o_all = torch.empty((world, B, Hq, D), dtype=torch.float32, device="cuda")
    l_all = torch.empty((world, B, Hq), dtype=torch.float32, device="cuda")
    for r in range(world):
        _part_state(workloads.shard_problem(p, r, world, kv_shard_range), o_all[r], l_all[r], num_ctas)
    o, lse = merge_gathered(o_all, l_all, torch.bfloat16)
    torch.cuda.synchronize()
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


def test_sharded_call_without_a_process_group_is_the_whole_cascade():
    p = workloads.make_problem(batch=5, hq=16, hkv=4, d=128, dtype="f16", prefix_lens=[257],
                               prefix_groups=[5], suffix=("list", [31, 0, 400, 16, 77]),
                               page_size=16, seed=82, poison=True)
    d = to_device(p)
    ws = workspace_for(pkc, p, num_ctas=7)
    buf = pkc.plan(p["cache_seqlens"], 7)
    pkc.plan_upload(buf, ws)
    o, lse = kv_sharded_cascade_decode(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                       p["prefix_req_indptr"], d["k_cache"], d["v_cache"],
                                       d["block_table"], d["cache_seqlens"], p["sm_scale"], ws,
                                       plan_buf=buf)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16 and pkc.device_status(ws) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)


def test_merge_states_to_rounds_once_from_float32():
    rng = np.random.default_rng(3)
    T, n, H, D = 7, 5, 6, 128
    v = torch.from_numpy(rng.standard_normal((T, n, H, D)).astype(np.float32)).cuda()
    s = torch.from_numpy(rng.uniform(-10, 10, (T, n, H)).astype(np.float32)).cuda()
    s[0, :, 0] = -float("inf")  # an all-empty row
    ref_v, ref_s = oracle.merge_n(np.moveaxis(v.cpu().numpy().astype(np.float64), 1, 0),
                                  np.moveaxis(s.cpu().numpy(), 1, 0))
    for dt, mant in ((torch.bfloat16, 7), (torch.float16, 10)):
        vo, so = pkc.merge_states_to(v, s, dt)
        v32, s32 = pkc.merge_states(v, s)
        torch.cuda.synchronize()
        # one rounding of the fp32 result, and the same LSE
        assert torch.equal(vo, v32.to(dt))
        assert torch.equal(so, s32)
        got = vo.float().cpu().numpy()
        e = np.floor(np.log2(np.maximum(np.abs(ref_v), 2.0 ** -14)))
        assert np.all(np.abs(got - ref_v) <= 1e-5 + 0.5 * 2.0 ** (e - mant))
