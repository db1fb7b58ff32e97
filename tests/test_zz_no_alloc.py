"""The decode entry point that allocates nothing, against the workspace one.

pkc_paged_decode_state_noalloc serves callers that cannot call cudaMalloc
(code inside another framework's pre-reserved memory pool, or on a fixed
memory budget): its split-KV scratch is a fixed array inside the library.
Two calls in a row, on different problems and plans, must each match
pkc_paged_decode_state on the same inputs -- the second call must not be
affected by what the first left in the shared array.  The test goes
through the C ABI directly.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import O_TOL, LSE_TOL, half_ulp, to_device, workspace_for

pytestmark = pytest.mark.gpu


def _problem(seed, lens, hq, hkv, dtype):
    return workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype,
                                  prefix_lens=[], prefix_groups=[], suffix=("list", lens),
                                  page_size=16, seed=seed, poison=True, extra_pages=2)


def _with_workspace(p, d, plan_buf, num_ctas):
    ws = workspace_for(pkc, p, num_ctas=num_ctas, prefix_splits=0)
    pkc.plan_upload(plan_buf, ws)
    o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["cache_seqlens"], p["sm_scale"], ws, plan_buf=plan_buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    return o, lse


def _no_alloc_via_c_abi(p, d, plan_buf):
    L = pkc.lib()
    B, Hq, D = d["q"].shape
    P, ps, Hkv, _ = d["k_cache"].shape
    o = torch.empty_like(d["q"])
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dtype = pkc.BF16 if d["q"].dtype == torch.bfloat16 else pkc.F16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.pkc_paged_decode_state_noalloc(
        d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
        d["block_table"].data_ptr(), d["block_table"].shape[1], d["cache_seqlens"].data_ptr(),
        B, Hq, Hkv, D, ps, P, float(p["sm_scale"]), ctypes.c_void_p(plan_buf.ctypes.data),
        o.data_ptr(), lse.data_ptr(), status.data_ptr(), dtype, stream)
    assert rc == pkc.PKC_OK, L.pkc_last_error()
    torch.cuda.synchronize()
    assert int(status.item()) == pkc.PKC_OK
    return o, lse


def _close(a_o, a_lse, b_o, b_lse):
    ref = b_o.float().cpu().numpy().astype(np.float64)
    got = a_o.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= O_TOL + half_ulp(ref, a_o.dtype))
    la, lb = a_lse.cpu().numpy(), b_lse.cpu().numpy()
    assert np.array_equal(np.isneginf(la), np.isneginf(lb))
    fin = ~np.isneginf(lb)
    assert np.all(np.abs(la[fin] - lb[fin]) <= LSE_TOL)


def _set_up_call():
    """A batch-0 call: reads no tensor and only places the scratch array on
    the current device (done once, before the memory checks below)."""
    L = pkc.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.pkc_paged_decode_state_noalloc(None, None, None, None, 1, None, 0, 8, 8, 128, 16, 0,
                                          1.0, None, None, None, None, pkc.F16, stream)
    assert rc == pkc.PKC_OK, L.pkc_last_error()
    torch.cuda.synchronize()


def test_no_alloc_matches_workspace_entry_point_two_calls_in_a_row():
    _set_up_call()
    first = _problem(41, [900, 0, 33, 4000, 17, 250], 32, 8, "bf16")
    second = _problem(42, [5, 1200, 64, 2], 16, 16, "f16")
    for p, num_ctas in ((first, 148), (second, 37)):
        d = to_device(p)
        plan_buf = pkc.plan(p["cache_seqlens"], num_ctas)
        want_o, want_lse = _with_workspace(p, d, plan_buf, num_ctas)
        got_o, got_lse = _no_alloc_via_c_abi(p, d, plan_buf)
        _close(got_o, got_lse, want_o, want_lse)


def test_no_alloc_calls_take_no_device_memory():
    """After the set-up call and one call of each kernel kind (which loads
    the kernels' code), further calls leave the device's free memory and
    torch's allocator exactly where they were."""
    _set_up_call()
    probs = [(_problem(44, [700, 3, 2100, 64], 32, 8, "bf16"), 148),
             (_problem(45, [17, 900, 0], 16, 16, "f16"), 29)]
    prepared = []
    for p, num_ctas in probs:
        d = to_device(p)
        plan_buf = pkc.plan(p["cache_seqlens"], num_ctas)
        B, Hq, _ = d["q"].shape
        outs = (torch.empty_like(d["q"]), torch.empty((B, Hq), dtype=torch.float32, device="cuda"),
                torch.zeros((1,), dtype=torch.int32, device="cuda"))
        prepared.append((p, d, plan_buf, outs))

    def call(p, d, plan_buf, outs):
        L = pkc.lib()
        B, Hq, D = d["q"].shape
        P, ps, Hkv, _ = d["k_cache"].shape
        dtype = pkc.BF16 if d["q"].dtype == torch.bfloat16 else pkc.F16
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = L.pkc_paged_decode_state_noalloc(
            d["q"].data_ptr(), d["k_cache"].data_ptr(), d["v_cache"].data_ptr(),
            d["block_table"].data_ptr(), d["block_table"].shape[1], d["cache_seqlens"].data_ptr(),
            B, Hq, Hkv, D, ps, P, float(p["sm_scale"]), ctypes.c_void_p(plan_buf.ctypes.data),
            outs[0].data_ptr(), outs[1].data_ptr(), outs[2].data_ptr(), dtype, stream)
        assert rc == pkc.PKC_OK, L.pkc_last_error()

    for args in prepared:  # warm-up: kernel code of both kinds loaded
        call(*args)
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    alloc_before = torch.cuda.memory_allocated()
    for _ in range(2):
        for args in prepared:
            call(*args)
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc_before
    assert free_after == free_before
    for args in prepared:
        assert int(args[3][2].item()) == pkc.PKC_OK


def test_no_alloc_rejects_a_plan_beyond_its_scratch():
    p = _problem(43, [10, 20], 64, 64, "f16")
    d = to_device(p)
    plan_buf = pkc.plan(p["cache_seqlens"], 600)  # 2*600*64 rows of partials > 8 MiB
    with pytest.raises(pkc.PkcError) as e:
        pkc.paged_decode_state_noalloc(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                       d["cache_seqlens"], p["sm_scale"], plan_buf=plan_buf)
    assert e.value.code == 3 and "8388608" in str(e.value)


def test_no_alloc_full_size_plan_matches_the_oracle():
    """The GQA suffix shape at full size (batch 256, 32/8 heads, lognormal
    lengths up to 16384 tokens, plan over 148 CTAs: long requests split over
    many chunks, so the partial states fill much of the scratch array), every
    row against the oracle."""
    import oracle
    from pkc_testing import compare, oracle_args
    _set_up_call()
    p = workloads.workload("gqa_cascade_lb", prefix_lens=[], prefix_groups=[])
    d = to_device(p)
    plan_buf = pkc.plan(p["cache_seqlens"], 148)
    got_o, got_lse = _no_alloc_via_c_abi(p, d, plan_buf)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(got_o, got_lse, ref_o, ref_lse)
