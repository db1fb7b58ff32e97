"""The small-batch cascade: an unplanned cascade whose prefix groups hold few
query rows per KV head runs as one decode launch that reads each request's
prefix as the first pages of its keys (pkc_set_cascade_small).  It must give
the oracle's attention over prefix u suffix, like the regular cascade."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cascade_gb300 as pkc
import workloads
from pkc_testing import compare, oracle_args, to_device, workspace_for

pytestmark = pytest.mark.gpu


@pytest.fixture
def small_path():
    yield pkc.set_cascade_small
    pkc.set_cascade_small(16)


def _cascade(p, state=False):
    d = to_device(p)
    ws = workspace_for(pkc, p)
    call = pkc.cascade_decode_state if state else pkc.cascade_decode
    o, lse = call(d["q"], d["k_prefix"], d["v_prefix"], p["prefix_kv_indptr"], p["prefix_req_indptr"],
                  d["k_cache"], d["v_cache"], d["block_table"], d["cache_seqlens"], p["sm_scale"], ws)
    torch.cuda.synchronize()
    return o, lse, pkc.device_status(ws)


SMALL = [
    # (hq, hkv, dtype, prefix_lens, groups, suffix lens, page_size)
    (32, 32, "f16", [256], [4], [32, 32, 32, 32], 16),          # the tiny workload's shape
    (32, 32, "f16", [256], [4], [32, 0, 1, 33], 16),
    (32, 8, "bf16", [160, 0, 48], [2, 1, 3], [5, 0, 300, 16, 17, 2, 9], 16),  # G = 4, an empty prefix, one request outside
    (16, 2, "f16", [64, 96], [1, 2], [100, 7, 64], 32),             # G = 8, page size 32
    (8, 4, "bf16", [16], [5], [1, 15, 16, 31, 0], 16),              # G = 2
    # stages wholly inside a prefix (one box per tensor) next to stages that
    # mix prefix and suffix pages:
    (16, 8, "f16", [320], [4], [10, 40, 0, 3], 32),                 # page size 32: two slices per page
    (32, 32, "bf16", [208, 96], [12, 12],                           # 24 requests: 4 KV heads per block
     [3, 50, 0, 17, 1, 64, 9, 33, 2, 80, 5, 16, 7, 0, 41, 12, 1, 30, 6, 72, 15, 8, 3, 20], 16),
    (32, 32, "f16", [304, 64, 160], [16, 16, 16],                   # 48 requests: 8 KV heads per block
     [int(x) for x in np.random.default_rng(7).integers(0, 90, 48)], 16),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_small_batch_cascade_matches_oracle_and_regular_path(small_path, case):
    hq, hkv, dtype, pl, groups, lens, ps = SMALL[case]
    p = workloads.make_problem(batch=len(lens), hq=hq, hkv=hkv, d=128, dtype=dtype, prefix_lens=pl,
                               prefix_groups=groups, suffix=("list", lens), page_size=ps,
                               seed=130 + case, poison=True, extra_pages=2)
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    small_path(16)
    o, lse, st = _cascade(p)
    assert st == pkc.PKC_OK
    assert pkc.last_launch_blocks()[0] == 0  # no prefix kernel
    compare(o, lse, ref_o, ref_lse)
    small_path(0)  # the regular cascade on the same problem
    o2, lse2, st2 = _cascade(p)
    assert st2 == pkc.PKC_OK
    assert pkc.last_launch_blocks()[0] > 0 or int(np.sum(pl)) == 0
    compare(o2, lse2, ref_o, ref_lse)


def test_small_batch_state_is_float32(small_path):
    p = workloads.make_problem(batch=3, hq=16, hkv=4, d=128, dtype="bf16", prefix_lens=[128],
                               prefix_groups=[3], suffix=("list", [40, 1, 0]), page_size=16, seed=140,
                               poison=True)
    small_path(16)
    o, lse, st = _cascade(p, state=True)
    assert st == pkc.PKC_OK and o.dtype == torch.float32
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse, o_tol=1e-5)


def test_small_batch_bad_page_id_is_reported(small_path):
    p = workloads.make_problem(batch=2, hq=8, hkv=8, d=128, dtype="f16", prefix_lens=[32], prefix_groups=[2],
                               suffix=("list", [40, 20]), page_size=16, seed=141)
    p["block_table"] = p["block_table"].copy()
    p["block_table"][1, 0] = 10 ** 6
    small_path(16)
    _, _, st = _cascade(p)
    assert st == 4  # PKC_ERR_BLOCK_TABLE, reported, no fault


def test_prefix_not_in_whole_pages_takes_the_regular_path(small_path):
    p = workloads.make_problem(batch=3, hq=8, hkv=8, d=128, dtype="f16", prefix_lens=[100], prefix_groups=[3],
                               suffix=("list", [10, 20, 0]), page_size=16, seed=142, poison=True)
    small_path(16)
    o, lse, st = _cascade(p)
    assert st == pkc.PKC_OK and pkc.last_launch_blocks()[0] > 0
    ref_o, ref_lse = oracle.attention_rows(p["q"], **oracle_args(p))
    compare(o, lse, ref_o, ref_lse)
