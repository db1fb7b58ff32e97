"""More shared-prefix cases on the GPU against the oracle: groups of 256
and more query rows per KV head (several row tiles, ragged last tiles),
g = 8, an empty prefix, a peaky softmax that exercises the lazy rescale,
and three levels with the prefixes both contiguous and in the page pool."""
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, dev, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


CASES = [
    # (hq, hkv, dtype, prefix_lens, groups, batch, q_scale)
    (32, 32, "f16", [256], [4], 4, 1.0),                # 4 rows per KV head
    (32, 8, "bf16", [300, 77], [40, 30], 70, 1.0),      # 160 / 120 rows: one partial pair each
    (32, 8, "bf16", [1000, 129], [70, 64], 134, 1.0),   # 280 rows (a pair and a ragged one), 256 rows
    (8, 1, "bf16", [1000], [40], 45, 1.0),              # g = 8: 320 rows, requests outside the group
    (16, 8, "f16", [129, 0, 512], [5, 2, 9], 16, 1.0),  # an empty prefix
    # peaky softmax (q x 8: lazy rescales), 320 rows; fp16, whose P keeps 11
    # bits (with bf16 P this case reaches 3.2e-3, beyond the 2e-3 tolerance)
    (32, 8, "f16", [700], [80], 80, 8.0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_prefix_cases_match_oracle(case):
    hq, hkv, dtype, pl, groups, batch, qs = CASES[case]
    p = workloads.make_problem(batch=batch, hq=hq, hkv=hkv, d=128, dtype=dtype, prefix_lens=pl,
                               prefix_groups=groups, suffix=("const", 0), page_size=16,
                               seed=60 + case, q_scale=qs)
    d = to_device(p)
    ws = workspace_for(pkc, p)
    o, lse = pkc.prefix_attention_state(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"],
                                        p["prefix_req_indptr"], p["sm_scale"], ws)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p, suffix=False))
    compare(o, lse, ref_o, ref_lse)


def test_cascade_levels_contiguous_and_paged_prefix():
    # three levels: 300 tokens for all 64 requests (256 rows per KV head),
    # then 200 / 130 tokens for halves of them; ragged caches
    lens = [5, 0, 17, 300, 1, 64, 33, 129] * 8
    p = workloads.make_problem(batch=len(lens), hq=32, hkv=8, d=128, dtype="bf16",
                               prefix_lens=[300, 200, 130], prefix_groups=[1, 1, 1],
                               suffix=("list", lens), page_size=16, seed=77, poison=True)
    ranges = [(0, 64), (0, 32), (32, 64)]
    d = to_device(p)
    ws = workspace_for(pkc, p, num_ctas=11)
    buf = pkc.plan(p["cache_seqlens"], 11)
    pkc.plan_upload(buf, ws)
    o, lse = pkc.cascade_decode_multilevel(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], ranges,
                                           d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"],
                                           p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    a = oracle_args(p)
    a.pop("prefix_req_indptr")
    ref_o, ref_lse = oracle.attention_rows(p["q"], prefix_req_ranges=ranges, **a)
    compare(o, lse, ref_o, ref_lse)
    # the same prefixes read in place from the page pool
    kc, vc, pages, page_indptr = workloads.pool_prefixes(p, 77)
    o2, lse2 = pkc.cascade_decode_paged_prefix(d["q"], dev(pages), page_indptr, p["prefix_kv_indptr"], ranges,
                                               dev(kc), dev(vc), d["block_table"], d["cache_seqlens"],
                                               p["sm_scale"], ws, plan_buf=buf)
    torch.cuda.synchronize()
    assert pkc.device_status(ws) == pkc.PKC_OK
    compare(o2, lse2, ref_o, ref_lse)
