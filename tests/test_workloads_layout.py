"""Input layout helpers (no GPU): the non-cascade form of a cascade problem.

Laying each shared prefix into pages of the cache pool and listing those
pages ahead of every request's own pages in its block table must describe
exactly the same key set, in the same order, as the cascade problem."""
import numpy as np
import pytest

import oracle
import workloads
from pkc_testing import oracle_args


def test_noncascade_layout_is_the_same_attention_problem():
    p = workloads.make_problem(batch=7, hq=8, hkv=2, d=128, dtype="bf16", prefix_lens=[32, 64],
                               prefix_groups=[2, 3], suffix=("list", [5, 0, 17, 33, 1, 9, 16]),
                               page_size=16, seed=3, poison=True, extra_pages=2)
    n = workloads.noncascade_problem(p, 9)
    assert n["k_prefix"] is None
    # requests 0-1 hold prefix 0 (2 pages), 2-4 prefix 1 (4 pages), 5-6 none
    assert list(n["cache_seqlens"]) == [37, 32, 81, 97, 65, 9, 16]
    o1, l1 = oracle.attention_rows(p["q"], **oracle_args(p))
    o2, l2 = oracle.attention_rows(n["q"], **oracle_args(n, prefix=False))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_noncascade_layout_needs_whole_prefix_pages():
    p = workloads.make_problem(batch=2, hq=4, hkv=4, d=128, dtype="f16", prefix_lens=[20],
                               prefix_groups=[2], suffix=("list", [3, 4]), page_size=16, seed=1)
    with pytest.raises(ValueError):
        workloads.noncascade_problem(p, 1)
