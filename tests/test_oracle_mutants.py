"""Planted mistakes in copies of the oracle must fail the pins (CPU only).

Each mutant is a plausible slip (a dropped term, a wrong sign, an off-by-one
index, a flipped tie-break).  The checks below are the same facts the pins
use; a mutant that passed them would mean the pins could not see that
mistake.
"""
import heapq
import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _partition_ok(merge2, state):
    rng = np.random.default_rng(3)
    sc = rng.normal(size=40) * 3
    vals = rng.normal(size=(40, 8))
    fv, fs = oracle.state(sc, vals)  # the full state, pinned against SDPA
    a, b = state(sc[:13], vals[:13]), state(sc[13:], vals[13:])
    ok = True
    for x, y in ((a, b), (b, a)):  # both merge orders, as the pin does
        mv, ms = merge2(x[0], x[1], y[0], y[1])
        ok &= bool(np.allclose(mv, fv, atol=1e-10) and abs(float(ms) - fs) < 1e-10)
    return ok


def _commutes(merge2):
    rng = np.random.default_rng(4)
    va, vb = rng.normal(size=(2, 3, 8))
    sa, sb = rng.uniform(-5, 5, size=(2, 3))
    x = merge2(va, sa, vb, sb)
    y = merge2(vb, sb, va, sa)
    return np.allclose(x[0], y[0]) and np.allclose(x[1], y[1])


def _singleton_ok(state):
    v = np.arange(4.0)
    out_v, out_s = state([2.5], v[None])
    return out_s == 2.5 and np.array_equal(out_v, v)


def test_real_oracle_passes_the_checks():
    assert _partition_ok(oracle.merge2, oracle.state)
    assert _commutes(oracle.merge2)
    assert _singleton_ok(oracle.state)


def test_merge_with_dropped_term_is_caught():
    def bad(v_a, s_a, v_b, s_b):
        m = np.maximum(s_a, s_b)
        w_a, w_b = np.exp(s_a - m), np.exp(s_b - m)
        return v_a * (w_a / (w_a + w_b))[..., None], m + np.log(w_a + w_b)
    assert not _partition_ok(bad, oracle.state)


def test_merge_with_wrong_weight_sign_is_caught():
    def bad(v_a, s_a, v_b, s_b):
        m = np.maximum(s_a, s_b)
        w_a, w_b = np.exp(-(s_a - m)), np.exp(s_b - m)
        v = (v_a * w_a[..., None] + v_b * w_b[..., None]) / (w_a + w_b)[..., None]
        return v, m + np.log(w_a + w_b)
    assert not _partition_ok(bad, oracle.state)
    assert not _commutes(bad)


def test_state_without_max_restored_is_caught():
    def bad(scores, values):
        s = np.asarray(scores, float)
        m = s.max()
        e = np.exp(s - m)
        return (e[:, None] * values).sum(0) / e.sum(), math.log(e.sum())
    assert not _singleton_ok(bad)


def test_resolve_off_by_one_slot_is_caught():
    gold = json.load(open(os.path.join(GOLDEN, "hf_paged_attention_decode_block_table.json")))

    def bad_next_slot(bt, lens, ps):
        return [(int(bt[b][(n - 1) // ps]), int((n - 1) % ps) + 1) for b, n in enumerate(lens)]
    got = bad_next_slot(gold["block_table"], gold["cache_seqlens"], gold["page_size"])
    assert [list(x) for x in got] != gold["expected_next_token_slot"]


def test_plan_with_flipped_tie_break_is_caught():
    # Same greedy rule but ties go to the higher CTA index: the hand table
    # (kv [10, 3, 5] over 2 CTAs) must then differ.
    work = [(0, 0, 9), (0, 9, 10), (1, 0, 3), (2, 0, 5)]
    order = sorted(range(4), key=lambda w: -(work[w][2] - work[w][1]))
    heap = [(0.0, -c) for c in range(2)]
    heapq.heapify(heap)
    lists = [[], []]
    for w in order:
        cost, nc = heapq.heappop(heap)
        lists[-nc].append(w)
        heapq.heappush(heap, (cost + 1 + work[w][2] - work[w][1], nc))
    assert lists != oracle.plan_ref([1, 1, 1], [10, 3, 5], 1, 2)["cta_work"]
