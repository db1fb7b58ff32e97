"""Seeded synthetic inputs for the paged-KV cascade decode workloads.

This module is the only code shared by the CUDA library's tests/bench and
the oracle.  It holds no arithmetic of the method: it draws lengths, page
permutations and N(0,1) / uniform tensors, encodes them as fp16 / bf16 bytes,
and lays them out.  Both sides read the same bytes.

Element encodings on the host:
  fp16 -> numpy float16;  bf16 -> numpy uint16 holding the bf16 bit pattern
  (float32 rounded to nearest-even, the same rounding torch uses);  fp32 ->
  numpy float32;  e4m3 -> numpy uint8 codes, float32 rounded by torch's own
  cast to float8_e4m3fn (used for fp8 KV caches only).

Workload shapes follow the pages' evaluation setup (LLaMA2-7B-like 32 heads
x 128 dims, page size 16, shared prompts up to 32768 tokens, batches up to
256; blog "Cascade Inference", section "Evaluation"), with the five named
workloads below.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 22  # elements per independently seeded generator block

WORKLOADS = {
    # batch 4, 32/32 heads, d 128, fp16; shared prefix 256, suffix 32 each.
    # No plan: one decode block per (request, KV-head group) reads its whole
    # suffix and writes the state directly (a plan over 148 CTAs would cut
    # every 32-token suffix into 1-token chunks: 34 against 16 us per step).
    "tiny_cascade": dict(batch=4, hq=32, hkv=32, d=128, dtype="f16",
                         prefix_lens=[256], prefix_groups=[4],
                         suffix=("const", 32), page_size=16, seed=1, plan=False),
    # merge_state: 4096 tokens x 32 heads x 128, fp32 v ~ N(0,1),
    # s ~ U[-10, 10]; binary and 16-ary
    "merge": dict(tokens=4096, heads=32, d=128, n_states=16, seed=2),
    # non-cascade paged decode: batch 64, kv len ~ U{512..4096}
    "paged_decode": dict(batch=64, hq=32, hkv=32, d=128, dtype="f16",
                         prefix_lens=[], prefix_groups=[],
                         suffix=("uniform", 512, 4096), page_size=16, seed=3),
    # cascade at the long-prompt shape: prefix 32768, suffix 256, batch 128
    "cascade_long_prompt": dict(batch=128, hq=32, hkv=32, d=128, dtype="f16",
                                prefix_lens=[32768], prefix_groups=[128],
                                suffix=("const", 256), page_size=16, seed=4),
    # FP8 KV paged decode at the GQA suffix shape: 32/8 heads, fp16 q and O,
    # e4m3 cache with per-tensor scales, batch 256, lognormal lengths
    "paged_decode_fp8": dict(batch=256, hq=32, hkv=8, d=128, dtype="f16",
                             kv_dtype="e4m3", k_scale=0.5, v_scale=1.25,
                             prefix_lens=[], prefix_groups=[],
                             suffix=("lognormal", 7.0, 1.0, 16, 16384),
                             page_size=16, seed=6, num_ctas=148),
    # the same shape with an fp16 cache (the 16-bit counterpart)
    "paged_decode_gqa": dict(batch=256, hq=32, hkv=8, d=128, dtype="f16",
                             prefix_lens=[], prefix_groups=[],
                             suffix=("lognormal", 7.0, 1.0, 16, 16384),
                             page_size=16, seed=6, num_ctas=148),
    # three-level cascade at the GQA shape: a 2048-token prompt for all 256
    # requests (level 0), then 4 prompts x 8192 tokens for 64 requests each
    # (level 1, request ranges in "prefix_ranges"), then the paged suffixes
    "gqa_cascade_3level": dict(batch=256, hq=32, hkv=8, d=128, dtype="bf16",
                               prefix_lens=[2048] + [8192] * 4, prefix_groups=[1] * 5,
                               prefix_ranges=[(0, 256), (0, 64), (64, 128), (128, 192), (192, 256)],
                               suffix=("lognormal", 7.0, 1.0, 16, 16384),
                               page_size=16, seed=7, num_ctas=148, alpha=1.0, beta=1.0),
    # GQA 32/8, bf16, batch 256; 4 prefixes x 8192 tokens, 64 requests each;
    # suffix ~ lognormal(7, 1) clipped to [16, 16384]; plan over 148 CTAs
    "gqa_cascade_lb": dict(batch=256, hq=32, hkv=8, d=128, dtype="bf16",
                           prefix_lens=[8192] * 4, prefix_groups=[64] * 4,
                           suffix=("lognormal", 7.0, 1.0, 16, 16384),
                           page_size=16, seed=5, num_ctas=148, alpha=1.0,
                           beta=1.0),
}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest-even); NaN stays a quiet NaN."""
    x = np.ascontiguousarray(x, np.float32)
    u = x.view(np.uint32)
    lsb = (u >> 16) & 1
    out = ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def f32_to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Round float32 to e4m3 codes with the library cast (torch)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _encode(x32: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return x32.astype(np.float16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x32)
    if dtype == "f32":
        return x32.astype(np.float32)
    if dtype == "e4m3":
        return f32_to_e4m3_codes(x32)
    raise ValueError(dtype)


_NP_DTYPE = {"f16": np.float16, "bf16": np.uint16, "f32": np.float32, "e4m3": np.uint8}


def _nan_value(dtype: str):
    return {"f16": np.float16(np.nan), "bf16": np.uint16(0x7FC0),
            "f32": np.float32(np.nan), "e4m3": np.uint8(0x7F)}[dtype]


def normal(shape, seed: int, tag: int, dtype: str, scale: float = 1.0,
           threads: int = 8) -> np.ndarray:
    """N(0, scale^2) tensor of `shape`, encoded as `dtype`.

    Generated in fixed blocks of 2^22 elements, block j from its own PCG64
    stream seeded by (seed, tag, j), so the values do not depend on the
    number of threads used to draw them.
    """
    n = int(np.prod(shape))
    np_dtype = _NP_DTYPE[dtype]
    out = np.empty(n, np_dtype)

    def fill(j):
        lo = j * _CHUNK
        hi = min(n, lo + _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, j])))
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[lo:hi] = _encode(x, dtype)

    blocks = (n + _CHUNK - 1) // _CHUNK
    if blocks <= 1 or threads <= 1:
        for j in range(blocks):
            fill(j)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(blocks)))
    return out.reshape(shape)


def suffix_lengths(spec, batch: int, rng: np.random.Generator) -> np.ndarray:
    """Per-request cached (suffix) lengths, drawn first from the workload rng."""
    kind = spec[0]
    if kind == "const":
        return np.full(batch, int(spec[1]), np.int32)
    if kind == "uniform":  # inclusive integer range
        return rng.integers(spec[1], spec[2], size=batch, endpoint=True).astype(np.int32)
    if kind == "lognormal":  # clip(rint(lognormal(mu, sigma)), lo, hi)
        x = rng.lognormal(spec[1], spec[2], size=batch)
        return np.clip(np.rint(x), spec[3], spec[4]).astype(np.int32)
    if kind == "list":
        return np.asarray(spec[1], np.int32)
    raise ValueError(kind)


def make_problem(*, batch, hq, hkv, d, dtype, prefix_lens, prefix_groups,
                 suffix, page_size, seed, max_blocks=None, extra_pages=0,
                 poison=False, q_scale=1.0, threads=8, kv_dtype=None, k_scale=1.0,
                 v_scale=1.0, **_ignored):
    """A full decode problem: queries, shared prefixes and a paged cache.

    Layouts: q [B, Hq, D]; k/v_prefix [sum(prefix_lens), Hkv, D] with
    prefix_kv_indptr / prefix_req_indptr (requests of group j are
    prefix_req_indptr[j] .. prefix_req_indptr[j+1]-1, contiguous);
    k/v_cache [P, page_size, Hkv, D]; block_table int32 [B, max_blocks],
    -1 where unallocated; cache_seqlens int32 [B].

    Pages: request b gets ceil(len_b / page_size) pages, taken in request
    order from a seeded permutation of the P pages (P = the pages needed
    plus `extra_pages` never referenced).  With `poison`, every cache slot
    no request may read (tails of last pages, unreferenced pages) is NaN.

    kv_dtype (default: dtype) is the paged cache's encoding; "e4m3" stores
    N(0,1) draws as e4m3 codes, and the problem then carries per-tensor
    k_scale / v_scale (the cached key is k_scale times the decoded code).
    The prefixes always have q's dtype.
    """
    kv_dtype = kv_dtype or dtype
    if kv_dtype != dtype and (kv_dtype != "e4m3" or dtype != "f16"):
        raise ValueError("an e4m3 cache goes with fp16 queries")
    if kv_dtype != "e4m3" and (k_scale != 1.0 or v_scale != 1.0):
        raise ValueError("k_scale / v_scale apply to an e4m3 cache only")
    rng = np.random.default_rng(seed)
    lens = suffix_lengths(suffix, batch, rng)
    n_pages_req = (lens + page_size - 1) // page_size
    need = int(n_pages_req.sum())
    num_pages = need + int(extra_pages)
    perm = rng.permutation(num_pages).astype(np.int32)
    if max_blocks is None:
        max_blocks = max(1, int(n_pages_req.max()) if batch else 1)
    bt = np.full((batch, max_blocks), -1, np.int32)
    off = 0
    for b in range(batch):
        k = int(n_pages_req[b])
        bt[b, :k] = perm[off:off + k]
        off += k
    q = normal((batch, hq, d), seed, 1, dtype, q_scale, threads)
    Lp = int(sum(prefix_lens))
    if Lp > 0:
        k_prefix = normal((Lp, hkv, d), seed, 2, dtype, 1.0, threads)
        v_prefix = normal((Lp, hkv, d), seed, 3, dtype, 1.0, threads)
    else:
        k_prefix = v_prefix = None
    k_cache = normal((num_pages, page_size, hkv, d), seed, 4, kv_dtype, 1.0, threads)
    v_cache = normal((num_pages, page_size, hkv, d), seed, 5, kv_dtype, 1.0, threads)
    if poison:
        used = np.zeros((num_pages, page_size), bool)
        for b in range(batch):
            n = int(lens[b])
            for j in range(int(n_pages_req[b])):
                used[bt[b, j], :min(page_size, n - j * page_size)] = True
        nanv = _nan_value(kv_dtype)
        k_cache[~used] = nanv
        v_cache[~used] = nanv
    kv_indptr = np.zeros(len(prefix_lens) + 1, np.int32)
    kv_indptr[1:] = np.cumsum(prefix_lens)
    req_indptr = np.zeros(len(prefix_groups) + 1, np.int32)
    req_indptr[1:] = np.cumsum(prefix_groups)
    return dict(q=q, k_prefix=k_prefix, v_prefix=v_prefix,
                prefix_kv_indptr=kv_indptr, prefix_req_indptr=req_indptr,
                k_cache=k_cache, v_cache=v_cache, block_table=bt,
                cache_seqlens=lens, page_size=page_size, num_kv_heads=hkv,
                sm_scale=1.0 / math.sqrt(d), dtype=dtype, kv_dtype=kv_dtype,
                k_scale=float(k_scale), v_scale=float(v_scale))


def pool_prefixes(p, seed, poison=True):
    """Lay a problem's shared prefixes into pages of its cache pool.

    The suffix pages stay first; the prefix pages are appended in a seeded
    order (group after group, page after page); with `poison` every slot past
    a prefix's end in its last page is NaN.  Returns (k_pool, v_pool,
    prefix_pages int32, prefix_page_indptr int32)."""
    ps = p["page_size"]
    ind = p["prefix_kv_indptr"]
    lens = np.diff(ind).astype(np.int64)
    n_pg = [(int(L) + ps - 1) // ps for L in lens]
    P0 = p["k_cache"].shape[0]
    total = sum(n_pg)
    order = np.random.default_rng(seed).permutation(total).astype(np.int32) + P0
    shape = (total,) + p["k_cache"].shape[1:]
    kc = np.concatenate([p["k_cache"], np.zeros(shape, p["k_cache"].dtype)])
    vc = np.concatenate([p["v_cache"], np.zeros(shape, p["v_cache"].dtype)])
    nanv = _nan_value(p["kv_dtype"]) if poison else 0
    pages, off = [], 0
    for j, L in enumerate(lens):
        lo = int(ind[j])
        for i in range(n_pg[j]):
            page = int(order[off + i])
            n = min(ps, int(L) - i * ps)
            kc[page] = nanv
            vc[page] = nanv
            kc[page, :n] = p["k_prefix"][lo + i * ps:lo + i * ps + n]
            vc[page, :n] = p["v_prefix"][lo + i * ps:lo + i * ps + n]
            pages.append(page)
        off += n_pg[j]
    page_indptr = np.concatenate([[0], np.cumsum(n_pg)]).astype(np.int32)
    return kc, vc, np.asarray(pages, np.int32), page_indptr


def noncascade_problem(p, seed, poison=False):
    """The same attention problem with no shared-prefix stage: each prefix is
    laid into pages of the cache pool (``pool_prefixes``; the pages are shared,
    not copied per request) and every request's block table lists its group's
    prefix pages, then its own suffix pages; its cached length becomes prefix
    + suffix.  Every prefix must fill whole pages (a page cannot end a prefix
    part-way and then continue with the suffix).  Returns a problem dict
    without prefixes."""
    ps = p["page_size"]
    ind = p["prefix_kv_indptr"]
    req = p["prefix_req_indptr"]
    lens_p = np.diff(ind).astype(np.int64)
    if np.any(lens_p % ps):
        raise ValueError("every prefix must be a whole number of pages")
    kc, vc, pages, page_indptr = pool_prefixes(p, seed, poison=poison)
    B = p["q"].shape[0]
    bt_s = p["block_table"]
    n_suffix_pages = (p["cache_seqlens"].astype(np.int64) + ps - 1) // ps
    pre_of = np.full(B, -1, np.int64)
    for j in range(len(lens_p)):
        pre_of[int(req[j]):int(req[j + 1])] = j
    n_pre = np.array([(page_indptr[j + 1] - page_indptr[j]) if j >= 0 else 0 for j in pre_of], np.int64)
    width = max(1, int((n_pre + n_suffix_pages).max()) if B else 1)
    bt = np.full((B, width), -1, np.int32)
    lens = np.array(p["cache_seqlens"], np.int32)
    for b in range(B):
        j = int(pre_of[b])
        k = 0
        if j >= 0:
            k = int(n_pre[b])
            bt[b, :k] = pages[page_indptr[j]:page_indptr[j + 1]]
            lens[b] += int(lens_p[j])
        m = int(n_suffix_pages[b])
        bt[b, k:k + m] = bt_s[b, :m]
    out = dict(p)
    out.update(k_prefix=None, v_prefix=None, prefix_kv_indptr=np.zeros(1, np.int32),
               prefix_req_indptr=np.zeros(1, np.int32), k_cache=kc, v_cache=vc,
               block_table=bt, cache_seqlens=lens)
    return out


def shard_problem(p, rank, world, shard_range):
    """Rank `rank`'s part of a problem's keys when they are sharded over
    `world` devices: for each prefix group the token slice
    shard_range(L_j, rank, world, 1) of its prefix, and for each request the
    page-aligned slice shard_range(len_b, rank, world, page_size) of its
    cached suffix (its block table row cut to those pages; the page pool is
    kept whole).  The requests, queries and prefix grouping are unchanged.
    Returns a problem dict of the same form."""
    ps = p["page_size"]
    ind = p["prefix_kv_indptr"]
    parts, new_ind = [], [0]
    for j in range(len(ind) - 1):
        lo, hi = shard_range(int(ind[j + 1] - ind[j]), rank, world, 1)
        if p["k_prefix"] is not None and hi > lo:
            parts.append((int(ind[j]) + lo, int(ind[j]) + hi))
        new_ind.append(new_ind[-1] + (hi - lo))
    kp = vp = None
    if p["k_prefix"] is not None:
        shape = (new_ind[-1],) + p["k_prefix"].shape[1:]
        kp = np.concatenate([p["k_prefix"][a:b] for a, b in parts]) if parts else np.zeros(shape, p["k_prefix"].dtype)
        vp = np.concatenate([p["v_prefix"][a:b] for a, b in parts]) if parts else np.zeros(shape, p["v_prefix"].dtype)
    lens = p["cache_seqlens"]
    B = len(lens)
    rows, new_lens = [], np.zeros(B, np.int32)
    for b in range(B):
        lo, hi = shard_range(int(lens[b]), rank, world, ps)
        rows.append(p["block_table"][b, lo // ps:(hi + ps - 1) // ps])
        new_lens[b] = hi - lo
    width = max(1, max((len(r) for r in rows), default=1))
    bt = np.full((B, width), -1, np.int32)
    for b, r in enumerate(rows):
        bt[b, :len(r)] = r
    out = dict(p)
    out.update(k_prefix=kp, v_prefix=vp, prefix_kv_indptr=np.asarray(new_ind, np.int32),
               block_table=bt, cache_seqlens=new_lens)
    return out


def make_merge(*, tokens, heads, d, n_states, seed, v_dtype="f32", threads=8,
               **_ignored):
    """merge_state inputs: two states per (token, head), plus n stacked.

    v ~ N(0,1) [T, H, D]; s ~ U[-10, 10] [T, H] (float32).  The n-ary inputs
    are v [T, n, H, D], s [T, n, H].
    """
    rng = np.random.default_rng(seed)
    s_a = rng.uniform(-10, 10, size=(tokens, heads)).astype(np.float32)
    s_b = rng.uniform(-10, 10, size=(tokens, heads)).astype(np.float32)
    s_n = rng.uniform(-10, 10, size=(tokens, n_states, heads)).astype(np.float32)
    v_a = normal((tokens, heads, d), seed, 11, v_dtype, 1.0, threads)
    v_b = normal((tokens, heads, d), seed, 12, v_dtype, 1.0, threads)
    v_n = normal((tokens, n_states, heads, d), seed, 13, v_dtype, 1.0, threads)
    return dict(v_a=v_a, s_a=s_a, v_b=v_b, s_b=s_b, v_n=v_n, s_n=s_n)


def workload(name: str, **overrides):
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    if name == "merge":
        return make_merge(**cfg)
    return make_problem(**cfg)


def effective_bytes(problem) -> int:
    """Algorithmic bytes of one cascade decode step: every valid KV token
    once (a shared prefix once), plus q, the final O and the fp32 LSE."""
    q = problem["q"]
    B, Hq, D = q.shape
    Hkv = problem["num_kv_heads"]
    esz = q.dtype.itemsize
    kv_esz = problem["k_cache"].dtype.itemsize
    lp = int(problem["prefix_kv_indptr"][-1])
    s = int(problem["cache_seqlens"].sum())
    kv = lp * 2 * Hkv * D * esz + s * 2 * Hkv * D * kv_esz
    return kv + 2 * B * Hq * D * esz + B * Hq * 4
