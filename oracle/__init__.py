"""Oracle for the paged-KV cascade decode library -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library
(``paged_kv_cascade_gb300``) and never imports it; the only code both sides
use is the seeded input generator module ``workloads``, which holds none of
the method's arithmetic.

Everything here is the plain statement of what the pages define, in float64
(or exact integers), with each function citing the passage it follows:

* ``state``                 -- s(I), v(I) of an index set (attention state)
* ``merge2`` / ``merge_n``  -- the binary and n-ary merge operator
* ``attention_rows``        -- full attention state of (request, head) rows over
                               shared prefix + paged suffix (C, float64)
* ``resolve`` / ``next_slot`` -- block-table resolution of cached tokens
* ``cu_seq_lens``           -- cumulative sequence lengths of a ragged batch
* ``plan_ref``              -- the load-balanced CTA schedule

Pins: every function above is checked in ``tests/test_oracle_*.py`` against
worked examples printed on the pages (``tests/golden``), closed forms,
invariants, and library routines (torch float64 SDPA / logsumexp).  The
plan has no worked example on the pages; its exact values are pinned only by
hand-computed tiny tables and invariants (see ``plan_ref``).
"""
from __future__ import annotations

import ctypes
import heapq
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkc_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpkc_oracle.so")
_lib = None
_lock = threading.Lock()

F32, F16, BF16, E4M3 = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile the C part of the oracle with gcc (plain -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.pkc_oracle_f16_to_f64.restype = ctypes.c_double
            lib.pkc_oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.pkc_oracle_bf16_to_f64.restype = ctypes.c_double
            lib.pkc_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.pkc_oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.pkc_oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.pkc_oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a):
    if a is None:
        return None
    return ctypes.c_void_p(a.ctypes.data)


def _dtype_code(a) -> int:
    """Element type of a host array: float32, float16, bf16 bits (uint16),
    or e4m3 codes (uint8)."""
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float16:
        return F16
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8:
        return E4M3
    raise TypeError(f"unsupported element type {a.dtype}")


def max_threads() -> int:
    return int(_load().pkc_oracle_max_threads())


def decode_scalar(bits: int, dtype: int) -> float:
    """float64 value of one fp16 / bf16 / e4m3 bit pattern (oracle's own
    decoder)."""
    lib = _load()
    if dtype == F16:
        return lib.pkc_oracle_f16_to_f64(bits)
    if dtype == E4M3:
        return lib.pkc_oracle_e4m3_to_f64(bits)
    return lib.pkc_oracle_bf16_to_f64(bits)


# ---------------------------------------------------------------------------
# Attention state and the merge operator
# ---------------------------------------------------------------------------

def state(scores, values):
    """Attention state (v(I), s(I)) of one index set.

    "Attention States and Recursive Attention" (FlashInfer tutorial), the
    definitions s(I) = log sum_{i in I} exp(s_i) and
    v(I) = sum_{i in I} exp(s_i) v_i / exp(s(I)); the same pair is (O(T),
    LSE(T)) in the MLSys'25 notes, A2 "Attention Composition".  The maximum
    is subtracted before exp ("in practice ... for numerical stability");
    it cancels exactly.  An empty set gives the identity (0, -inf).

    scores: [n] float64, values: [n, D] -> (v [D], s scalar)
    """
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    if s.shape[0] == 0:
        return np.zeros(v.shape[1:], np.float64), -math.inf
    m = s.max()
    e = np.exp(s - m)
    total = e.sum()
    return (e[:, None] * v).sum(axis=0) / total, m + math.log(total)


def merge2(v_a, s_a, v_b, s_b):
    """Binary merge operator: (v(I), s(I)) (+) (v(J), s(J)) = state of I u J.

    "Attention States and Recursive Attention", binary merge equation;
    "Cascade Inference" blog, section "Recursive Attention", same equation:
      v = (v_I e^{s_I} + v_J e^{s_J}) / (e^{s_I} + e^{s_J})
      s = log(e^{s_I} + e^{s_J})
    evaluated with the larger s subtracted first.  Works elementwise over
    leading (token, head) axes: v [..., D], s [...].  A side with s = -inf is
    the empty set and contributes nothing; two empty sides give (0, -inf).
    """
    v_a = np.asarray(v_a, np.float64)
    v_b = np.asarray(v_b, np.float64)
    s_a = np.asarray(s_a, np.float64)
    s_b = np.asarray(s_b, np.float64)
    m = np.maximum(s_a, s_b)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w_a = np.where(np.isneginf(s_a), 0.0, np.exp(s_a - m_safe))
    w_b = np.where(np.isneginf(s_b), 0.0, np.exp(s_b - m_safe))
    den = w_a + w_b
    den_safe = np.where(empty, 1.0, den)
    v = (v_a * w_a[..., None] + v_b * w_b[..., None]) / den_safe[..., None]
    s = np.where(empty, -np.inf, m_safe + np.log(den_safe))
    return v, s


def merge_n(v, s):
    """n-ary merge operator over axis 0 of v [n, ..., D], s [n, ...].

    "Attention States and Recursive Attention", n-ary merge equation:
      v = sum_i softmax(s(I_i)) v(I_i),   s = log sum_i exp(s(I_i)),
    with the softmax taken over the n states and the maximum subtracted
    first.  Empty states (s = -inf) get weight 0; all-empty gives (0, -inf).
    """
    v = np.asarray(v, np.float64)
    s = np.asarray(s, np.float64)
    m = s.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.where(np.isneginf(s), 0.0, np.exp(s - m_safe[None]))
    den = w.sum(axis=0)
    den_safe = np.where(empty, 1.0, den)
    out_v = (w[..., None] * v).sum(axis=0) / den_safe[..., None]
    out_s = np.where(empty, -np.inf, m_safe + np.log(den_safe))
    return out_v, out_s


# ---------------------------------------------------------------------------
# Full attention of (request, head) rows: the C oracle
# ---------------------------------------------------------------------------

def attention_rows(q, *, rows=None, sm_scale, num_kv_heads,
                   k_prefix=None, v_prefix=None, prefix_kv_indptr=None,
                   prefix_req_indptr=None, prefix_req_ranges=None, k_cache=None, v_cache=None,
                   block_table=None, cache_seqlens=None, page_size=None,
                   k_scale=1.0, v_scale=1.0, n_threads=0):
    """Attention state of each (request, query head) row over its full key set.

    The key set of request b is the shared prefix of b's group (requests
    prefix_req_indptr[j] <= b < prefix_req_indptr[j+1] share prefix j, tokens
    prefix_kv_indptr[j]..prefix_kv_indptr[j+1]-1 of k/v_prefix [L, Hkv, D])
    followed by its cache_seqlens[b] cached tokens, read through block_table
    from k/v_cache [P, page_size, Hkv, D].  A multi-level cascade gives
    prefix_req_ranges = [(begin_j, end_j)] instead: the ranges may overlap and
    a request attends to the prefixes of every group that holds it, in group
    order, then to its cache
    from k/v_cache [P, page_size, Hkv, D].  Computed in float64 from the
    definition (see pkc_oracle.c).

    q: [B, Hq, D] float16 / bf16-bits uint16 / float32 host array.  The
    prefixes have q's element type; the paged cache has it too, or holds
    e4m3 codes (uint8), the cached key and value then being k_scale and
    v_scale times the decoded codes (an fp8 cache with per-tensor scales).
    rows: int array [n, 2] of (request, head); default all B*Hq rows.
    Returns (o [n, D] float64, lse [n] float64).
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    B, Hq, D = q.shape
    dt = _dtype_code(q)
    if rows is None:
        bb, hh = np.meshgrid(np.arange(B), np.arange(Hq), indexing="ij")
        rows = np.stack([bb.ravel(), hh.ravel()], axis=1)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    n = rows.shape[0]
    o = np.empty((n, D), np.float64)
    lse = np.empty((n,), np.float64)
    n_prefix = 0
    req_begin = req_end = None
    if k_prefix is not None:
        k_prefix = np.ascontiguousarray(k_prefix)
        v_prefix = np.ascontiguousarray(v_prefix)
        prefix_kv_indptr = np.ascontiguousarray(prefix_kv_indptr, np.int32)
        n_prefix = len(prefix_kv_indptr) - 1
        if prefix_req_ranges is not None:
            rr = np.asarray(prefix_req_ranges, np.int32).reshape(-1, 2)
        else:
            ind = np.asarray(prefix_req_indptr, np.int32)
            rr = np.stack([ind[:-1], ind[1:]], axis=1)
        assert rr.shape[0] == n_prefix
        req_begin = np.ascontiguousarray(rr[:, 0])
        req_end = np.ascontiguousarray(rr[:, 1])
        assert _dtype_code(k_prefix) == dt and _dtype_code(v_prefix) == dt
    num_pages = 0
    bt_stride = 0
    kv_dt = dt
    if k_cache is not None:
        k_cache = np.ascontiguousarray(k_cache)
        v_cache = np.ascontiguousarray(v_cache)
        block_table = np.ascontiguousarray(block_table, np.int32)
        cache_seqlens = np.ascontiguousarray(cache_seqlens, np.int32)
        num_pages = k_cache.shape[0]
        bt_stride = block_table.shape[1]
        assert k_cache.shape[1] == page_size
        kv_dt = _dtype_code(k_cache)
        assert _dtype_code(v_cache) == kv_dt and kv_dt in (dt, E4M3)
        if kv_dt != E4M3:
            assert k_scale == 1.0 and v_scale == 1.0, "scales apply to an e4m3 cache only"
    rc = lib.pkc_oracle_attention_rows(
        _ptr(q), ctypes.c_int(B), ctypes.c_int(Hq), ctypes.c_int(num_kv_heads),
        ctypes.c_int(D), ctypes.c_int(dt), ctypes.c_double(sm_scale),
        _ptr(k_prefix), _ptr(v_prefix), _ptr(prefix_kv_indptr),
        _ptr(req_begin), _ptr(req_end), ctypes.c_int(n_prefix),
        _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
        ctypes.c_int64(bt_stride), _ptr(cache_seqlens),
        ctypes.c_int(page_size or 0), ctypes.c_int64(num_pages),
        ctypes.c_int(kv_dt), ctypes.c_double(k_scale), ctypes.c_double(v_scale),
        _ptr(rows), ctypes.c_int64(n), ctypes.c_int(n_threads),
        _ptr(o), _ptr(lse))
    if rc == 1:
        raise ValueError("block table entry out of range inside a used page")
    if rc != 0:
        raise RuntimeError(f"oracle attention_rows failed with code {rc}")
    return o, lse


# ---------------------------------------------------------------------------
# Paged-cache indexing
# ---------------------------------------------------------------------------

def resolve(block_table, cache_seqlens, page_size, num_pages):
    """(page, slot) of every cached token, request after request.

    Hugging Face "Paged attention", decoding path, indexing mechanism: row b
    of block_table lists the physical pages of request b, cache_seqlens[b]
    its number of cached tokens, -1 an unallocated entry.  Token t lives in
    page block_table[b][t // page_size] at slot t % page_size; entries past
    the last used page are never read.  Returns a list (per request) of
    lists of (page, slot); raises ValueError on an invalid page that must be
    read.
    """
    lib = _load()
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(cache_seqlens, np.int32)
    total = int(sl.sum())
    pages = np.empty(max(total, 1), np.int32)
    slots = np.empty(max(total, 1), np.int32)
    rc = lib.pkc_oracle_resolve(_ptr(bt), ctypes.c_int64(bt.shape[1]),
                                _ptr(sl), ctypes.c_int(bt.shape[0]),
                                ctypes.c_int(page_size),
                                ctypes.c_int64(num_pages), _ptr(pages),
                                _ptr(slots))
    if rc != 0:
        raise ValueError(f"block table cannot be resolved (code {rc})")
    out, k = [], 0
    for n in sl.tolist():
        out.append([(int(pages[k + i]), int(slots[k + i])) for i in range(n)])
        k += n
    return out


def next_slot(block_table, cache_seqlens, page_size):
    """(page, slot) where each request's next token would be written.

    Same passage as ``resolve``: the next token of a request with len cached
    tokens goes to entry len // page_size of its block-table row, slot
    len % page_size (a new page when the last one is full).
    """
    bt = np.asarray(block_table)
    return [(int(bt[b, n // page_size]), int(n % page_size))
            for b, n in enumerate(np.asarray(cache_seqlens).tolist())]


def cu_seq_lens(lengths):
    """Cumulative lengths [0, l0, l0+l1, ...] and the maximum length.

    Hugging Face "Paged attention", varlen path, indexing mechanism
    (cu_seq_lens_q/k, max_length_q/k).
    """
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out, (max(int(n) for n in lengths) if len(lengths) else 0)


# ---------------------------------------------------------------------------
# Load-balanced schedule
# ---------------------------------------------------------------------------

def plan_ref(qo_len, kv_len, tile_q, num_ctas, alpha=1.0, beta=1.0):
    """The load-balanced schedule of work chunks onto CTAs.

    FlashInfer MLSys'25 notes, A3 "Dynamic-aware runtime", load-balanced
    scheduling, steps 1-7, and appendix D (split-K direct write).  Readings
    where the pages leave a step open (listed in the design notes):

    * L_kv = ceil(sum_i ceil(l_qo(i)/T_q) * l_kv(i) / #CTA), at least 1,
      exact integers.
    * Work units are (request, query tile) in request-major order; each is
      cut into consecutive KV chunks [0, L_kv), [L_kv, 2 L_kv), ... with the
      remainder last.  A unit with l_kv = 0 has no chunk.  The work index w
      numbers chunks unit by unit, chunk by chunk.
    * W is sorted by chunk length, longest first; equal lengths keep
      ascending w.
    * The priority queue pops the least (cost, CTA index); the popped CTA
      gets the chunk and its cost grows by cost(l_q, l_kv) = alpha*l_q +
      beta*l_kv, l_q the tile's query rows.
    * A unit with one chunk writes its output directly; chunks of units
      with two or more chunks get partial slots numbered in w order.

    Returns a dict of plain Python ints / lists.
    """
    n = len(qo_len)
    assert len(kv_len) == n and tile_q >= 1 and num_ctas >= 1
    units = []  # (request, q tile, rows l_q)
    for i in range(n):
        n_tiles = -(-int(qo_len[i]) // tile_q)
        for j in range(n_tiles):
            units.append((i, j, min(tile_q, int(qo_len[i]) - j * tile_q)))
    total = sum(-(-int(qo_len[i]) // tile_q) * int(kv_len[i]) for i in range(n))
    L = max(1, -(-total // num_ctas))
    work = []  # (unit, kv_begin, kv_end)
    unit_chunks = []
    for u, (i, _, _) in enumerate(units):
        first = len(work)
        for b in range(0, int(kv_len[i]), L):
            work.append((u, b, min(b + L, int(kv_len[i]))))
        unit_chunks.append(list(range(first, len(work))))
    order = sorted(range(len(work)), key=lambda w: -(work[w][2] - work[w][1]))
    heap = [(0.0, c) for c in range(num_ctas)]
    heapq.heapify(heap)
    cta_work = [[] for _ in range(num_ctas)]
    for w in order:
        cost, c = heapq.heappop(heap)
        u, b, e = work[w]
        cta_work[c].append(w)
        heapq.heappush(heap, (cost + (alpha * units[u][2] + beta * (e - b)), c))
    cta_cost = [0.0] * num_ctas
    for cost, c in heap:
        cta_cost[c] = cost
    partial = [-1] * len(work)
    slot = 0
    for u in range(len(units)):
        if len(unit_chunks[u]) >= 2:
            for w in unit_chunks[u]:
                partial[w] = slot
                slot += 1
    return {
        "kv_chunk": L,
        "units": units,
        "work": work,
        "cta_work": cta_work,
        "cta_cost": cta_cost,
        "partial": partial,
        "unit_chunks": unit_chunks,
        "split_units": [u for u in range(len(units)) if len(unit_chunks[u]) >= 2],
        "empty_units": [u for u in range(len(units)) if len(unit_chunks[u]) == 0],
        "n_partials": slot,
        "order": order,
    }
