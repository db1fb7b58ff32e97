"""Pins of the oracle's load-balanced schedule (CPU only).

The pages give the scheduling rule (FlashInfer MLSys'25 notes, A3,
load-balanced scheduling, steps 1-7; appendix D) but no worked plan, so the
exact values are pinned by small tables computed by hand here and by
invariants that must hold for any input.
"""
import math

import numpy as np
import pytest

import oracle
import workloads


def test_hand_table_split_and_tie_break():
    # kv [10, 3, 5], 2 CTAs: total 18 -> L_kv 9.  Chunks: w0=[0,9) w1=[9,10)
    # (request 0), w2=[0,3), w3=[0,5).  Longest first: w0 w3 w2 w1.
    # CTA0 <- w0 (cost 10); CTA1 <- w3 (6); CTA1 <- w2 (10); tie 10/10 goes
    # to the lower index: CTA0 <- w1 (12).
    p = oracle.plan_ref([1, 1, 1], [10, 3, 5], 1, 2)
    assert p["kv_chunk"] == 9
    assert p["work"] == [(0, 0, 9), (0, 9, 10), (1, 0, 3), (2, 0, 5)]
    assert p["cta_work"] == [[0, 1], [3, 2]]
    assert p["cta_cost"] == [12.0, 10.0]
    assert p["partial"] == [0, 1, -1, -1]
    assert p["split_units"] == [0] and p["empty_units"] == []
    assert p["order"] == [0, 3, 2, 1]


def test_hand_table_empty_request_and_idle_cta():
    # kv [0, 4], 3 CTAs: L_kv = ceil(4/3) = 2; request 0 has no chunk.
    p = oracle.plan_ref([1, 1], [0, 4], 1, 3)
    assert p["kv_chunk"] == 2
    assert p["work"] == [(1, 0, 2), (1, 2, 4)]
    assert p["cta_work"] == [[0], [1], []]
    assert p["cta_cost"] == [3.0, 3.0, 0.0]
    assert p["partial"] == [0, 1]
    assert p["empty_units"] == [0] and p["split_units"] == [1]


def test_hand_table_query_tiles_and_alpha():
    # T_q 2, qo [3, 1], kv [4, 2], alpha 2: units (0,0,l_q=2) (0,1,1) (1,0,1);
    # total 2*4 + 1*2 = 10 -> L_kv 5, no split.  CTA0 <- w0 cost 2*2+4 = 8;
    # CTA1 <- w1 cost 2+4 = 6; CTA1 <- w2 cost 6 + 2 + 2 = 10.
    p = oracle.plan_ref([3, 1], [4, 2], 2, 2, alpha=2.0, beta=1.0)
    assert p["units"] == [(0, 0, 2), (0, 1, 1), (1, 0, 1)]
    assert p["kv_chunk"] == 5
    assert p["cta_work"] == [[0], [1, 2]]
    assert p["cta_cost"] == [8.0, 10.0]
    assert p["partial"] == [-1, -1, -1] and p["split_units"] == []


def _check_invariants(qo, kv, T, C, alpha, beta):
    p = oracle.plan_ref(qo, kv, T, C, alpha, beta)
    L = p["kv_chunk"]
    total = sum(-(-q // T) * k for q, k in zip(qo, kv))
    assert L == max(1, -(-total // C))
    # every token of every unit covered exactly once, in order, chunks <= L
    for u, (i, _, _) in enumerate(p["units"]):
        ws = p["unit_chunks"][u]
        spans = [p["work"][w][1:] for w in ws]
        pos = 0
        for b, e in spans:
            assert b == pos and 0 < e - b <= L
            pos = e
        assert pos == kv[i]
    assigned = sorted(w for lst in p["cta_work"] for w in lst)
    assert assigned == list(range(len(p["work"])))
    n_units = len(p["units"])
    assert len(p["work"]) <= C + n_units
    # partial outputs fit 2 * #CTA * T_q rows (appendix D bound)
    assert p["n_partials"] <= 2 * C
    # brute-force replay of the greedy rule with a linear scan
    order = sorted(range(len(p["work"])),
                   key=lambda w: (-(p["work"][w][2] - p["work"][w][1]), w))
    cost = [0.0] * C
    lists = [[] for _ in range(C)]
    for w in order:
        c = min(range(C), key=lambda c: (cost[c], c))
        lists[c].append(w)
        u, b, e = p["work"][w]
        cost[c] = cost[c] + (alpha * p["units"][u][2] + beta * (e - b))
    assert lists == p["cta_work"]
    assert cost == p["cta_cost"]
    return p


@pytest.mark.parametrize("seed", range(30))
def test_invariants_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 40))
    T = int(rng.choice([1, 1, 2, 16, 128]))
    qo = [int(x) for x in rng.integers(1, 300 if T > 1 else 2, size=n)]
    kv = [int(x) for x in rng.integers(0, 5000, size=n)]
    C = int(rng.integers(1, 200))
    _check_invariants(qo, kv, T, C, float(rng.choice([1.0, 0.5, 2.0])),
                      float(rng.choice([1.0, 1.5])))


def test_invariants_at_gqa_workload():
    # the workload's lengths over 148 CTAs (pinned values) and over the
    # workload's own plan CTA count
    w = workloads.WORKLOADS["gqa_cascade_lb"]
    lens = workloads.suffix_lengths(w["suffix"], w["batch"],
                                    np.random.default_rng(w["seed"]))
    p = _check_invariants([1] * w["batch"], lens.tolist(), 1, 148,
                          w["alpha"], w["beta"])
    assert p["kv_chunk"] == 2974
    assert len(p["split_units"]) == 37
    assert max(len(p["unit_chunks"][u]) for u in range(w["batch"])) == 6
    _check_invariants([1] * w["batch"], lens.tolist(), 1, w["num_ctas"], w["alpha"], w["beta"])


def test_all_zero_lengths():
    p = oracle.plan_ref([1, 1, 1], [0, 0, 0], 1, 4)
    assert p["kv_chunk"] == 1 and p["work"] == []
    assert p["empty_units"] == [0, 1, 2]
    assert p["cta_work"] == [[], [], [], []]
