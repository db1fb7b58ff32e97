"""Pins of the oracle's multi-level cascade (CPU only).

A request may belong to several prefix groups (levels: e.g. a system prompt
shared by every request, then a per-group prompt).  Its key set is all those
prefixes, then its own cached tokens.  Attention over a set does not depend
on how the set is split ([T] "Attention States and Recursive Attention":
the state of a union is the merge of the parts' states), so the multi-level
result must equal a single-level problem whose one prefix is the
concatenation, and brute-force softmax attention over the explicit keys.
"""
import math

import numpy as np
import torch

import oracle
import workloads


def _levels_problem():
    # 6 requests, 4/2 heads; level 0: one 40-token prompt for all; level 1:
    # 17 tokens for requests 0-2, 0 tokens for 3, 9 tokens for requests 3-5
    p = workloads.make_problem(batch=6, hq=4, hkv=2, d=128, dtype="f16",
                               prefix_lens=[40, 17, 9], prefix_groups=[6, 3, 3],
                               suffix=("list", [5, 0, 19, 3, 1, 33]), page_size=8, seed=21)
    ranges = [(0, 6), (0, 3), (3, 6)]
    return p, ranges


def _args(p, **over):
    a = dict(sm_scale=p["sm_scale"], num_kv_heads=p["num_kv_heads"], k_prefix=p["k_prefix"],
             v_prefix=p["v_prefix"], prefix_kv_indptr=p["prefix_kv_indptr"],
             k_cache=p["k_cache"], v_cache=p["v_cache"], block_table=p["block_table"],
             cache_seqlens=p["cache_seqlens"], page_size=p["page_size"])
    a.update(over)
    return a


def _concatenated(p, ranges, b):
    """One request's prefix keys: every group holding it, in group order."""
    ind = p["prefix_kv_indptr"]
    parts = [np.arange(ind[j], ind[j + 1]) for j, (lo, hi) in enumerate(ranges) if lo <= b < hi]
    return np.concatenate(parts) if parts else np.zeros(0, np.int64)


def test_levels_equal_one_concatenated_prefix_per_request():
    p, ranges = _levels_problem()
    o, lse = oracle.attention_rows(p["q"], **_args(p, prefix_req_ranges=ranges))
    Hq = p["q"].shape[1]
    for b in range(6):
        idx = _concatenated(p, ranges, b)
        kp, vp = p["k_prefix"][idx], p["v_prefix"][idx]
        one = oracle.attention_rows(p["q"][b:b + 1], **_args(
            p, k_prefix=kp, v_prefix=vp, prefix_kv_indptr=[0, len(idx)], prefix_req_indptr=[0, 1],
            block_table=p["block_table"][b:b + 1], cache_seqlens=p["cache_seqlens"][b:b + 1]))
        np.testing.assert_allclose(o[b * Hq:(b + 1) * Hq], one[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b * Hq:(b + 1) * Hq], one[1], rtol=0, atol=1e-12)


def test_levels_match_brute_force_softmax():
    p, ranges = _levels_problem()
    o, lse = oracle.attention_rows(p["q"], **_args(p, prefix_req_ranges=ranges))
    Hq, hkv = p["q"].shape[1], p["num_kv_heads"]
    g = Hq // hkv
    kc = torch.from_numpy(p["k_cache"].astype(np.float64))
    vc = torch.from_numpy(p["v_cache"].astype(np.float64))
    for b in range(6):
        idx = _concatenated(p, ranges, b)
        n = int(p["cache_seqlens"][b])
        pages = [p["block_table"][b, t // p["page_size"]] for t in range(n)]
        slots = [t % p["page_size"] for t in range(n)]
        for h in range(Hq):
            kv = h // g
            keys = [torch.from_numpy(p["k_prefix"][idx, kv].astype(np.float64))]
            vals = [torch.from_numpy(p["v_prefix"][idx, kv].astype(np.float64))]
            if n:
                keys.append(kc[pages, slots, kv])
                vals.append(vc[pages, slots, kv])
            K, V = torch.cat(keys), torch.cat(vals)
            q = torch.from_numpy(p["q"][b, h].astype(np.float64))
            s = (K @ q) * p["sm_scale"]
            ref_lse = torch.logsumexp(s, 0).item()
            ref_o = (torch.softmax(s, 0) @ V).numpy()
            r = b * Hq + h
            assert abs(lse[r] - ref_lse) < 1e-10
            np.testing.assert_allclose(o[r], ref_o, rtol=0, atol=1e-12)


def test_a_request_in_no_group_and_the_old_single_group_rule_differ():
    p, ranges = _levels_problem()
    multi = oracle.attention_rows(p["q"], **_args(p, prefix_req_ranges=ranges))
    # keeping only the last group that holds a request (a two-level reading)
    # must give a different answer: the pins above can see that mistake
    last_only = [(0, 0), (0, 3), (3, 6)]
    single = oracle.attention_rows(p["q"], **_args(p, prefix_req_ranges=last_only))
    assert np.abs(multi[0] - single[0]).max() > 1e-3
    # a request outside every group attends to its cache only
    none = oracle.attention_rows(p["q"], **_args(p, prefix_req_ranges=[(0, 0)] * 3))
    cache_only = oracle.attention_rows(p["q"], **_args(p, k_prefix=None, v_prefix=None))
    np.testing.assert_allclose(none[0], cache_only[0], rtol=0, atol=0)
    assert math.isinf(cache_only[1][4 * 1]) and cache_only[1][4 * 1] < 0  # request 1: no tokens at all
