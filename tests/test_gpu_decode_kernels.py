"""Both paged-decode kernels (CUDA cores and tensor cores) against the oracle,
and the FP8 KV cache path (e4m3 codes, fp16 q and O), on the GPU."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


@pytest.fixture
def kernel():
    """Force one decode kernel for the test, then restore the automatic choice."""
    def force(which):
        pkc.set_decode_kernel(which)
    yield force
    pkc.set_decode_kernel("auto")


def _decode(p, num_ctas, fp8=False):
    d = to_device(p)
    plan_buf = pkc.plan(p["cache_seqlens"], num_ctas) if num_ctas else None
    ws = workspace_for(pkc, p, num_ctas=num_ctas or 0, prefix_splits=0)
    if plan_buf is not None:
        pkc.plan_upload(plan_buf, ws)
    if fp8:
        o, lse = pkc.paged_decode_state_fp8(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                            d["cache_seqlens"], p["sm_scale"], ws,
                                            k_scale=p["k_scale"], v_scale=p["v_scale"],
                                            plan_buf=plan_buf)
    else:
        o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                        d["cache_seqlens"], p["sm_scale"], ws, plan_buf=plan_buf)
    torch.cuda.synchronize()
    return o, lse, pkc.device_status(ws)


CASES = [
    # (hq, hkv, dtype, page_size, lengths); ragged tails, empty rows, one token
    (32, 8, "bf16", 16, [3, 250, 16, 0, 1000, 7]),     # G 4, 8 heads per block
    (32, 32, "f16", 16, [1, 15, 16, 17, 100, 0, 513]),  # G 1
    (8, 4, "f16", 32, [30, 32, 70, 64]),               # G 2, 4 heads per block
    (16, 2, "bf16", 8, [6, 7, 8, 49, 50, 333]),        # G 8, 2 heads per block
    (8, 1, "f16", 16, [5, 16, 31, 200]),               # G 8, 1 head per block
    (64, 8, "bf16", 4, [1, 4, 5, 77]),                 # 4-slot pages, 2 slices per warp
]


@pytest.mark.parametrize("which", ["simt", "mma"])
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("num_ctas", [None, 5, 40])
def test_both_kernels_small(kernel, which, case, num_ctas):
    hq, hkv, dtype, ps, lens = CASES[case]
    kernel(which)
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype,
                               prefix_lens=[], prefix_groups=[], suffix=("list", lens),
                               page_size=ps, seed=30 + case, extra_pages=3, poison=True)
    o, lse, status = _decode(p, num_ctas)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


@pytest.mark.parametrize("which", ["simt", "mma"])
def test_both_kernels_peaky_softmax(kernel, which):
    # q x 8: sharp softmax, the lazy reference maximum moves often
    kernel(which)
    p = workloads.make_problem(batch=6, hq=32, hkv=8, d=128, dtype="bf16", prefix_lens=[],
                               prefix_groups=[], suffix=("list", [300, 1, 64, 65, 900, 17]),
                               page_size=16, seed=78, q_scale=8.0, poison=True)
    o, lse, status = _decode(p, 7)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_kernels_agree_on_the_gqa_suffix_shape(kernel):
    # the cascade workload's suffix (batch 256, 32/8 heads, 148 CTAs), no prefix
    # every row of both kernels against the oracle
    p = workloads.workload("gqa_cascade_lb", prefix_lens=[], prefix_groups=[])
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    kernel("mma")
    o, lse, st = _decode(p, 148)
    assert st == pkc.PKC_OK
    compare(o, lse, ref_o, ref_lse)
    kernel("simt")
    o2, lse2, st2 = _decode(p, 148)
    assert st2 == pkc.PKC_OK
    compare(o2, lse2, ref_o, ref_lse)


FP8_CASES = [
    (32, 8, 16, [3, 250, 16, 0, 1000, 7]),
    (32, 32, 16, [1, 15, 16, 17, 100, 0, 513]),
    (8, 4, 32, [30, 32, 70, 64]),
    (16, 2, 8, [6, 7, 8, 49, 50, 333]),
    (64, 8, 4, [1, 4, 5, 77]),
]


@pytest.mark.parametrize("case", range(len(FP8_CASES)))
@pytest.mark.parametrize("num_ctas", [None, 5, 40])
def test_fp8_cache_small(case, num_ctas):
    hq, hkv, ps, lens = FP8_CASES[case]
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype="f16",
                               kv_dtype="e4m3", k_scale=0.5, v_scale=1.25, prefix_lens=[],
                               prefix_groups=[], suffix=("list", lens), page_size=ps,
                               seed=50 + case, extra_pages=3, poison=True)
    o, lse, status = _decode(p, num_ctas, fp8=True)
    assert status == pkc.PKC_OK
    assert o.dtype == torch.float16
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_fp8_cache_peaky_and_scaled():
    # a large k_scale sharpens the softmax; v_scale must reach the output
    p = workloads.make_problem(batch=5, hq=32, hkv=8, d=128, dtype="f16", kv_dtype="e4m3",
                               k_scale=3.0, v_scale=0.0625, prefix_lens=[], prefix_groups=[],
                               suffix=("list", [500, 2, 129, 48, 1100]), page_size=16, seed=61,
                               poison=True)
    o, lse, status = _decode(p, 9, fp8=True)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_fp8_workload_every_row():
    """e4m3 cache, batch 256, 32/8 heads, lognormal lengths, 148 CTAs: every
    row against the oracle's decoding of the same codes."""
    p = workloads.workload("paged_decode_fp8")
    o, lse, status = _decode(p, 148, fp8=True)
    assert status == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, prefix=False))
    compare(o, lse, ref_o, ref_lse)


def test_fp8_all_empty_and_bad_page():
    p = workloads.make_problem(batch=3, hq=8, hkv=8, d=128, dtype="f16", kv_dtype="e4m3",
                               prefix_lens=[], prefix_groups=[], suffix=("list", [0, 0, 0]),
                               page_size=16, seed=1, extra_pages=1)
    o, lse, status = _decode(p, None, fp8=True)
    assert status == pkc.PKC_OK
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    p = workloads.make_problem(batch=2, hq=8, hkv=8, d=128, dtype="f16", kv_dtype="e4m3",
                               prefix_lens=[], prefix_groups=[], suffix=("list", [40, 20]),
                               page_size=16, seed=2)
    p["block_table"] = p["block_table"].copy()
    p["block_table"][1, 0] = 10 ** 6
    _, _, status = _decode(p, None, fp8=True)
    assert status == 4  # PKC_ERR_BLOCK_TABLE, reported, no fault
