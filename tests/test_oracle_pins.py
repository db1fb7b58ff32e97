"""Pins of the oracle to facts fixed outside it (CPU only).

Each check compares the oracle with something it does not compute itself:
values printed on the pages (tests/golden), closed forms, algebraic
identities of the merge operator, and library routines (numpy's float16,
torch's bfloat16 conversion, torch float64 SDPA and logsumexp).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# Element decoding: the oracle's own fp16 / bf16 decoders
# ---------------------------------------------------------------------------

def test_f16_decoder_matches_numpy_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode_scalar(int(b), oracle.F16) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoder_matches_torch_all_patterns():
    bits = torch.arange(1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode_scalar(int(b) & 0xFFFF, oracle.BF16)
                    for b in range(1 << 16)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_encoding_round_trips_through_torch():
    x = np.random.default_rng(0).standard_normal(4096).astype(np.float32) * 100
    ours = workloads.f32_to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)


# ---------------------------------------------------------------------------
# The attention state of one index set
# ---------------------------------------------------------------------------

def test_singleton_state_is_the_element():
    # Blog "Cascade Inference", Recursive Attention: for I = {i},
    # s(I) = s_i and v(I) = v_i.
    rng = np.random.default_rng(1)
    for _ in range(20):
        s = float(rng.normal() * 5)
        v = rng.normal(size=7)
        out_v, out_s = oracle.state([s], v[None])
        assert out_s == s
        assert np.array_equal(out_v, v)


def test_empty_state_is_identity():
    v, s = oracle.state(np.zeros(0), np.zeros((0, 4)))
    assert s == -math.inf and np.array_equal(v, np.zeros(4))


def _dense_problem(rng, n, d, dtype="f16", q_zero=False, equal_k=False,
                   const_v=None):
    """One request, one head, no paging: k, v [n, 1, d] as a prefix."""
    q = workloads.normal((1, 1, d), int(rng.integers(1 << 30)), 1, dtype)
    k = workloads.normal((n, 1, d), int(rng.integers(1 << 30)), 2, dtype)
    v = workloads.normal((n, 1, d), int(rng.integers(1 << 30)), 3, dtype)
    if q_zero:
        q[...] = 0
    if equal_k:
        k[...] = k[:1]
    if const_v is not None:
        v[...] = const_v
    return q, k, v


def _run_dense(q, k, v, scale):
    return oracle.attention_rows(
        q, sm_scale=scale, num_kv_heads=1, k_prefix=k, v_prefix=v,
        prefix_kv_indptr=np.array([0, k.shape[0]], np.int32),
        prefix_req_indptr=np.array([0, 1], np.int32))


def _f64(x):
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


@pytest.mark.parametrize("n", [1, 5, 300])
def test_closed_form_zero_query(n):
    # q = 0: every score is 0, so s(I) = log n and v(I) = mean of v.
    rng = np.random.default_rng(n)
    q, k, v = _dense_problem(rng, n, 32, q_zero=True)
    o, lse = _run_dense(q, k, v, 0.3)
    assert abs(lse[0] - math.log(n)) < 1e-12
    np.testing.assert_allclose(o[0], _f64(v)[:, 0].mean(axis=0), rtol=0, atol=1e-12)


def test_closed_form_constant_values():
    # All v_i = c: any convex combination is c.
    rng = np.random.default_rng(2)
    q, k, v = _dense_problem(rng, 64, 16, const_v=np.float16(1.5))
    o, _ = _run_dense(q, k, v, 0.25)
    np.testing.assert_allclose(o[0], np.full(16, 1.5), rtol=0, atol=1e-12)


def test_closed_form_equal_keys():
    # All k_i equal: uniform weights; s(I) = s + log n.
    rng = np.random.default_rng(3)
    n, d, scale = 50, 32, 1 / math.sqrt(32)
    q, k, v = _dense_problem(rng, n, d, equal_k=True)
    o, lse = _run_dense(q, k, v, scale)
    s = scale * float(_f64(q)[0, 0] @ _f64(k)[0, 0])
    assert abs(lse[0] - (s + math.log(n))) < 1e-10
    np.testing.assert_allclose(o[0], _f64(v)[:, 0].mean(axis=0), rtol=0, atol=1e-12)


def _paged_from_dense(rng, dense_k, dense_v, lens, page_size, extra_pages=3):
    """Scatter per-request contiguous KV into randomly permuted pages."""
    hkv, d = dense_k[0].shape[1:]
    need = [(n + page_size - 1) // page_size for n in lens]
    P = sum(need) + extra_pages
    perm = rng.permutation(P)
    kc = np.full((P, page_size, hkv, d), np.nan, np.float16)
    vc = np.full((P, page_size, hkv, d), np.nan, np.float16)
    bt = np.full((len(lens), max(need) + 2), -1, np.int32)
    off = 0
    for b, n in enumerate(lens):
        for j in range(need[b]):
            p = perm[off + j]
            bt[b, j] = p
            m = min(page_size, n - j * page_size)
            kc[p, :m] = dense_k[b][j * page_size:j * page_size + m]
            vc[p, :m] = dense_v[b][j * page_size:j * page_size + m]
        off += need[b]
    return kc, vc, bt


def test_full_attention_matches_torch_sdpa_and_logsumexp():
    # v({1..n}) is ordinary attention output (tutorial, after the v(I)
    # definition): compare with torch float64 SDPA; s(I) with logsumexp.
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D, ps = 3, 4, 2, 32, 4
    g = Hq // Hkv
    prefix_len = [9, 5]
    groups = [2, 1]
    lens = [0, 7, 13]
    scale = 1 / math.sqrt(D)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16)
    kp = rng.standard_normal((sum(prefix_len), Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((sum(prefix_len), Hkv, D)).astype(np.float16)
    dk = [rng.standard_normal((n, Hkv, D)).astype(np.float16) for n in lens]
    dv = [rng.standard_normal((n, Hkv, D)).astype(np.float16) for n in lens]
    kc, vc, bt = _paged_from_dense(rng, dk, dv, lens, ps)
    kv_ptr = np.array([0, 9, 14], np.int32)
    req_ptr = np.array([0, 2, 3], np.int32)
    o, lse = oracle.attention_rows(
        q, sm_scale=scale, num_kv_heads=Hkv, k_prefix=kp, v_prefix=vp,
        prefix_kv_indptr=kv_ptr, prefix_req_indptr=req_ptr, k_cache=kc,
        v_cache=vc, block_table=bt, cache_seqlens=np.array(lens, np.int32),
        page_size=ps)
    r = 0
    for b in range(B):
        j = 0 if b < 2 else 1
        for h in range(Hq):
            kvh = h // g
            K = np.concatenate([kp[kv_ptr[j]:kv_ptr[j + 1], kvh], dk[b][:, kvh]])
            V = np.concatenate([vp[kv_ptr[j]:kv_ptr[j + 1], kvh], dv[b][:, kvh]])
            tq = torch.from_numpy(q[b, h].astype(np.float64))[None, None, None]
            tk = torch.from_numpy(K.astype(np.float64))[None, None]
            tv = torch.from_numpy(V.astype(np.float64))[None, None]
            ref_o = torch.nn.functional.scaled_dot_product_attention(
                tq, tk, tv, scale=scale)[0, 0, 0].numpy()
            ref_lse = torch.logsumexp(scale * (tk[0, 0] @ tq[0, 0, 0]), 0).item()
            np.testing.assert_allclose(o[r], ref_o, rtol=0, atol=1e-12)
            assert abs(lse[r] - ref_lse) < 1e-12
            r += 1


def test_row_subset_equals_full_rows():
    p = workloads.workload("tiny_cascade", suffix=("const", 20), poison=True)
    args = dict(sm_scale=p["sm_scale"], num_kv_heads=p["num_kv_heads"],
                k_prefix=p["k_prefix"], v_prefix=p["v_prefix"],
                prefix_kv_indptr=p["prefix_kv_indptr"],
                prefix_req_indptr=p["prefix_req_indptr"], k_cache=p["k_cache"],
                v_cache=p["v_cache"], block_table=p["block_table"],
                cache_seqlens=p["cache_seqlens"], page_size=p["page_size"])
    o, lse = oracle.attention_rows(p["q"], **args)
    rows = np.array([[3, 31], [0, 0], [2, 17]], np.int32)
    o2, lse2 = oracle.attention_rows(p["q"], rows=rows, **args)
    for i, (b, h) in enumerate(rows):
        assert np.array_equal(o2[i], o[b * 32 + h]) and lse2[i] == lse[b * 32 + h]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_zero_length_request_gives_identity():
    p = workloads.make_problem(batch=2, hq=2, hkv=1, d=16, dtype="bf16",
                               prefix_lens=[], prefix_groups=[],
                               suffix=("list", [0, 5]), page_size=4, seed=9,
                               poison=True)
    o, lse = oracle.attention_rows(
        p["q"], sm_scale=0.25, num_kv_heads=1, k_cache=p["k_cache"],
        v_cache=p["v_cache"], block_table=p["block_table"],
        cache_seqlens=p["cache_seqlens"], page_size=4)
    assert np.all(lse[:2] == -np.inf) and np.all(o[:2] == 0)
    assert np.all(np.isfinite(lse[2:]))


def test_bad_block_table_entry_inside_used_range_is_rejected():
    p = workloads.make_problem(batch=2, hq=1, hkv=1, d=8, dtype="f16",
                               prefix_lens=[], prefix_groups=[],
                               suffix=("list", [5, 9]), page_size=4, seed=1)
    bt = p["block_table"].copy()
    bt[1, 2] = -1  # third page of request 1 is needed (tokens 8..8)
    with pytest.raises(ValueError):
        oracle.attention_rows(p["q"], sm_scale=1.0, num_kv_heads=1,
                              k_cache=p["k_cache"], v_cache=p["v_cache"],
                              block_table=bt, cache_seqlens=p["cache_seqlens"],
                              page_size=4)


# ---------------------------------------------------------------------------
# The merge operator
# ---------------------------------------------------------------------------

def _rand_states(rng, n, shape=(5, 3), d=8):
    v = rng.normal(size=(n,) + shape + (d,))
    s = rng.uniform(-10, 10, size=(n,) + shape)
    return v, s


def test_merge_commutative_and_associative():
    rng = np.random.default_rng(11)
    v, s = _rand_states(rng, 3)
    ab = oracle.merge2(v[0], s[0], v[1], s[1])
    ba = oracle.merge2(v[1], s[1], v[0], s[0])
    np.testing.assert_allclose(ab[0], ba[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ab[1], ba[1], rtol=0, atol=1e-13)
    left = oracle.merge2(*ab, v[2], s[2])
    bc = oracle.merge2(v[1], s[1], v[2], s[2])
    right = oracle.merge2(v[0], s[0], *bc)
    np.testing.assert_allclose(left[0], right[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(left[1], right[1], rtol=0, atol=1e-12)


def test_merge_n_equals_fold_of_merge2():
    rng = np.random.default_rng(12)
    v, s = _rand_states(rng, 16)
    nv, ns = oracle.merge_n(v, s)
    fv, fs = v[0], s[0]
    for i in range(1, 16):
        fv, fs = oracle.merge2(fv, fs, v[i], s[i])
    np.testing.assert_allclose(nv, fv, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ns, fs, rtol=0, atol=1e-12)


def test_merge_empty_is_identity_and_two_empties_stay_empty():
    rng = np.random.default_rng(13)
    v, s = _rand_states(rng, 1)
    ev, es = np.zeros_like(v[0]), np.full_like(s[0], -np.inf)
    out = oracle.merge2(v[0], s[0], ev, es)
    assert np.array_equal(out[0], v[0]) and np.array_equal(out[1], s[0])
    out = oracle.merge2(ev, es, ev, es)
    assert np.all(out[0] == 0) and np.all(out[1] == -np.inf)
    assert not np.any(np.isnan(out[0]))
    nv, ns = oracle.merge_n(np.stack([ev, ev, ev]), np.stack([es, es, es]))
    assert np.all(nv == 0) and np.all(ns == -np.inf)


@pytest.mark.parametrize("seed", range(5))
def test_random_partition_merged_in_random_order_equals_full_state(seed):
    # Any partition of the KV, merged in any order, gives the state of the
    # whole set (tutorial: "the final result is mathematically equivalent";
    # blog Fig. 2).  The full state is checked against SDPA above.
    rng = np.random.default_rng(100 + seed)
    n, d = int(rng.integers(2, 200)), 16
    sc = rng.normal(size=n) * 3
    vals = rng.normal(size=(n, d))
    full_v, full_s = oracle.state(sc, vals)
    idx = rng.permutation(n)
    cuts = np.sort(rng.choice(np.arange(1, n), size=min(n - 1, int(rng.integers(1, 8))), replace=False))
    parts = np.split(idx, cuts)
    states = [oracle.state(sc[p], vals[p]) for p in parts]
    while len(states) > 1:  # random merge tree
        i, j = sorted(rng.choice(len(states), 2, replace=False))
        merged = oracle.merge2(states[i][0], states[i][1], states[j][0], states[j][1])
        states = [st for k, st in enumerate(states) if k not in (i, j)] + [merged]
    np.testing.assert_allclose(states[0][0], full_v, rtol=0, atol=1e-12)
    assert abs(float(states[0][1]) - full_s) < 1e-12
    nv, ns = oracle.merge_n(np.stack([oracle.state(sc[p], vals[p])[0] for p in parts]),
                            np.array([oracle.state(sc[p], vals[p])[1] for p in parts]))
    np.testing.assert_allclose(nv, full_v, rtol=0, atol=1e-12)
    assert abs(float(ns) - full_s) < 1e-12


def test_cascade_split_of_the_c_oracle_rows():
    # Prefix-only state (+) suffix-only state = state over prefix u suffix,
    # all three from the C oracle.
    p = workloads.workload("tiny_cascade", suffix=("list", [0, 3, 17, 32]),
                           poison=True)
    common = dict(sm_scale=p["sm_scale"], num_kv_heads=p["num_kv_heads"])
    pref = dict(k_prefix=p["k_prefix"], v_prefix=p["v_prefix"],
                prefix_kv_indptr=p["prefix_kv_indptr"],
                prefix_req_indptr=p["prefix_req_indptr"])
    suf = dict(k_cache=p["k_cache"], v_cache=p["v_cache"],
               block_table=p["block_table"], cache_seqlens=p["cache_seqlens"],
               page_size=p["page_size"])
    o_full, l_full = oracle.attention_rows(p["q"], **common, **pref, **suf)
    o_p, l_p = oracle.attention_rows(p["q"], **common, **pref)
    o_s, l_s = oracle.attention_rows(p["q"], **common, **suf)
    o_m, l_m = oracle.merge2(o_p, l_p, o_s, l_s)
    np.testing.assert_allclose(o_m, o_full, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l_m, l_full, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Paged-cache indexing: the worked examples printed on the pages
# ---------------------------------------------------------------------------

def test_block_table_worked_example():
    gold = _golden("hf_paged_attention_decode_block_table.json")
    ps = gold["page_size"]
    res = oracle.resolve(gold["block_table"], gold["cache_seqlens"], ps, 7)
    for b, toks in enumerate(res):
        pages = []
        counts = []
        for page, slot in toks:
            if not pages or pages[-1] != page:
                pages.append(page)
                counts.append(0)
            counts[-1] += 1
        assert pages == gold["expected_pages_read"][b]
        assert counts == gold["expected_tokens_per_page"][b]
        assert [slot for _, slot in toks] == [t % ps for t in range(len(toks))]
    nxt = oracle.next_slot(np.array(gold["block_table"]), gold["cache_seqlens"], ps)
    assert [list(x) for x in nxt] == gold["expected_next_token_slot"]


def test_cu_seq_lens_worked_example():
    gold = _golden("hf_paged_attention_varlen_cu_seq_lens.json")
    cq, mq = oracle.cu_seq_lens(gold["q_lens"])
    ck, mk = oracle.cu_seq_lens(gold["k_lens"])
    assert cq == gold["cu_seq_lens_q"] and ck == gold["cu_seq_lens_k"]
    assert mq == gold["max_length_q"] and mk == gold["max_length_k"]
    qi = [r for r in range(3) for _ in range(cq[r], cq[r + 1])]
    ki = [r for r in range(3) for _ in range(ck[r], ck[r + 1])]
    assert qi == gold["q_request_index"] and ki == gold["k_request_index"]


def test_resolve_round_trips_a_random_permutation():
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 40, size=6)]
    ps = 8
    need = [(n + ps - 1) // ps for n in lens]
    perm = rng.permutation(sum(need) + 4)
    bt = np.full((6, max(need) + 1), -1, np.int32)
    truth = []
    off = 0
    for b, n in enumerate(lens):
        bt[b, :need[b]] = perm[off:off + need[b]]
        truth.append([(int(perm[off + t // ps]), t % ps) for t in range(n)])
        off += need[b]
    assert oracle.resolve(bt, lens, ps, len(perm)) == truth


def test_resolve_rejects_unallocated_page_in_use():
    with pytest.raises(ValueError):
        oracle.resolve([[2, -1]], [40], 32, 7)
    with pytest.raises(ValueError):
        oracle.resolve([[9]], [3], 32, 7)  # page id >= num_pages
    # entries past the used range are never read, whatever they hold
    assert len(oracle.resolve([[2, 99999]], [32], 32, 7)[0]) == 32
