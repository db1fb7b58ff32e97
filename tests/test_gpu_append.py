"""In-place KV append on the GPU: bytes against the oracle's next-slot rule,
then a decode over the grown cache against the oracle's attention."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, dev, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


def _problem(lens, hkv=4, dtype="bf16", kv_dtype=None, ps=16, seed=3):
    """A cache whose tables already hold the page of each request's next token."""
    p = workloads.make_problem(batch=len(lens), hq=4 * hkv, hkv=hkv, d=128, dtype=dtype,
                               kv_dtype=kv_dtype, prefix_lens=[], prefix_groups=[],
                               suffix=("list", [n + 1 for n in lens]), page_size=ps, seed=seed,
                               extra_pages=2)
    p["cache_seqlens"] = np.asarray(lens, np.int32)
    return p


def _new_kv(p, seed):
    B = len(p["cache_seqlens"])
    hkv = p["num_kv_heads"]
    kvd = p["kv_dtype"]
    k = workloads.normal((B, hkv, 128), seed, 7, kvd)
    v = workloads.normal((B, hkv, 128), seed, 8, kvd)
    return k, v


def _expected(p, k_new, v_new, mask=None):
    """Host copy of the caches with each appending request's token written at
    the oracle's next slot."""
    kc, vc = p["k_cache"].copy(), p["v_cache"].copy()
    lens = p["cache_seqlens"].copy()
    for b, (page, slot) in enumerate(oracle.next_slot(p["block_table"], lens, p["page_size"])):
        if mask is not None and not mask[b]:
            continue
        kc[page, slot] = k_new[b]
        vc[page, slot] = v_new[b]
        lens[b] += 1
    return kc, vc, lens


def _host(t, like):
    a = t.cpu()
    if a.dtype == torch.bfloat16:
        a = a.view(torch.int16)
    return a.numpy().view(like.dtype)


@pytest.mark.parametrize("kv_dtype", [None, "e4m3"])
def test_append_writes_next_slot_and_grows_lengths(kv_dtype):
    dtype = "f16" if kv_dtype else "bf16"
    p = _problem([15, 16, 0, 31, 5, 47], dtype=dtype, kv_dtype=kv_dtype)  # page-boundary cases
    k_new, v_new = _new_kv(p, 11)
    d = to_device(p)
    ws = workspace_for(pkc, p, prefix_splits=0)
    pkc.append_kv(dev(k_new), dev(v_new), d["k_cache"], d["v_cache"], d["block_table"],
                  d["cache_seqlens"], ws)
    assert pkc.device_status(ws) == pkc.PKC_OK
    kc, vc, lens = _expected(p, k_new, v_new)
    np.testing.assert_array_equal(_host(d["k_cache"], kc).view(np.uint8), kc.view(np.uint8))
    np.testing.assert_array_equal(_host(d["v_cache"], vc).view(np.uint8), vc.view(np.uint8))
    np.testing.assert_array_equal(d["cache_seqlens"].cpu().numpy(), lens)


def test_append_mask_and_missing_page():
    p = _problem([3, 16, 9, 32])
    p["block_table"] = p["block_table"].copy()
    p["block_table"][1, 1] = -1  # request 1's next token starts a page that is not there
    k_new, v_new = _new_kv(p, 12)
    mask = np.array([1, 1, 0, 1], np.uint8)
    d = to_device(p)
    ws = workspace_for(pkc, p, prefix_splits=0)
    pkc.append_kv(dev(k_new), dev(v_new), d["k_cache"], d["v_cache"], d["block_table"],
                  d["cache_seqlens"], ws, append_mask=dev(mask))
    assert pkc.device_status(ws) == 4  # PKC_ERR_BLOCK_TABLE, reported, no fault
    mask_eff = mask.copy()
    mask_eff[1] = 0  # skipped: nothing written, length unchanged
    kc, vc, lens = _expected(p, k_new, v_new, mask_eff)
    np.testing.assert_array_equal(_host(d["k_cache"], kc).view(np.uint8), kc.view(np.uint8))
    np.testing.assert_array_equal(_host(d["v_cache"], vc).view(np.uint8), vc.view(np.uint8))
    np.testing.assert_array_equal(d["cache_seqlens"].cpu().numpy(), lens)


def test_decode_after_append_sees_the_new_token():
    p = _problem([40, 16, 1, 200], hkv=8, seed=5)
    k_new, v_new = _new_kv(p, 13)
    d = to_device(p)
    ws = workspace_for(pkc, p, num_ctas=6, prefix_splits=0)
    pkc.append_kv(dev(k_new), dev(v_new), d["k_cache"], d["v_cache"], d["block_table"],
                  d["cache_seqlens"], ws)
    kc, vc, lens = _expected(p, k_new, v_new)
    grown = dict(p, k_cache=kc, v_cache=vc, cache_seqlens=lens)
    buf = pkc.plan(lens, 6)
    pkc.plan_upload(buf, ws)
    o, lse = pkc.paged_decode_state(d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                    d["cache_seqlens"], p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(grown, prefix=False))
    compare(o, lse, ref_o, ref_lse)
