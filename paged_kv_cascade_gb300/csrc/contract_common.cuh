// The contraction of attention states into a request's final O and LSE, and
// its fused form.
//
// Every (request, query head) row of the output is the (+) of its sources
// ("Attention States and Recursive Attention", n-ary merge): the pieces of
// every shared prefix the request attends to (prefix stage), then its
// suffix state -- one direct state or the partial states of its KV chunks,
// in ascending KV order (MLSys'25 notes, A3: the final output is the
// contraction of the partial outputs).  contract_row() is that merge for
// one row, by one warp; the standalone contraction kernel runs it over all
// rows after the stages.
//
// Fused (MLSys'25 notes, A3: attention and contraction in one persistent
// kernel): the kernels that write the sources count them instead.  After a
// warp has written a source of (request, KV head) it adds one to that
// pair's arrival counter; the warp that brings the counter to the number
// of sources the pair has merges the pair's G rows itself, so no kernel
// ever waits for another and no contraction launch follows.  Writers make
// their stores visible (__threadfence) before the count; the merging warp
// fences again after it and reads the sources past L1 (ld.global.cg).
#pragma once
#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {

__device__ __forceinline__ float ld_cg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ float4 ld_cg4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

// Pieces of group j's (row tile, KV head) pair that hold row (req, h), and
// their first partial slot.  The pair covering flat KV tiles [a, a + kvt)
// was computed by prefix blocks block_of(a) .. block_of(a + kvt - 1), piece
// i in slot slot_base[j] + i.
template <class CP>
__device__ __forceinline__ int group_pieces(const CP& p, int j, int req, int h, int& base) {
  base = 0;
  const int kvt = (p.prefix_kv_indptr[j + 1] - p.prefix_kv_indptr[j] + 127) / 128;
  if (kvt <= 0 || p.prefix_tiles <= 0) return 0;
  const int rr = (req - p.prefix_req_begin[j]) * p.g + h % p.g;  // row within the group's rows
  const int pair = (rr / 128) * p.hkv + h / p.g;
  // block_of(x) = ((x + 1) C - 1) / T, in 32 bits (the host keeps T C < 2^31)
  const int a = p.prefix_kvt_indptr[j] + pair * kvt;
  const int T = (int)p.prefix_tiles, C = p.prefix_blocks;
  base = p.prefix_slot_base[j];
  return ((a + kvt) * C - 1) / T - ((a + 1) * C - 1) / T + 1;
}

template <class CP>
__device__ __forceinline__ bool in_group(const CP& p, int j, int req) {
  return p.prefix_req_begin[j] <= req && req < p.prefix_req_end[j];
}

// One warp: (+) over every source of row (req, h), lane i owning dims
// 4i .. 4i+3, written as the final O row (out_dtype) and LSE.  `unit` is the
// request's unit of the plan (the request itself for decode plans).
template <class CP>
__device__ __forceinline__ void contract_row(const CP& p, int req, int unit, int h, int lane) {
  constexpr int D = PKC_HEAD_DIM;
  const int32_t* pl = p.plan;
  // Running state of the merge: maximum m, denominator den, unnormalised
  // acc.  Sources go in batches of 4 whose loads are all in flight
  // together; the running state is rescaled between batches.  (Batches of 4
  // keep the standalone kernel at 56 registers, 4 blocks per SM: more rows
  // in flight than batches of 8 at 3 blocks per SM.)
  constexpr int kB = 4;
  float m = neg_inf(), den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t row_off = (int64_t)req * p.hq + h;
  // Sources: the prefix pieces of every group holding the request (one
  // group in a two-level cascade, several in a multi-level one), then the
  // suffix.  One pass per group; the last pass also takes the suffix, so a
  // two-level row is a single pass.
  auto next_group = [&](int j) {  // first group after j holding the request, or -1
    if (!p.prefix_o) return -1;
    for (++j; j < p.n_prefix; ++j)
      if (in_group(p, j, req)) return j;
    return -1;
  };
  auto prefix_lse = [&](int slot) { return p.prefix_lse + (int64_t)slot * p.prefix_stride_lse + row_off; };
  auto prefix_o = [&](int slot) { return p.prefix_o + (int64_t)slot * p.prefix_stride_o + row_off * D; };
  // The first group's first batch of prefix pieces depends on no plan word:
  // its loads go out before the plan's words are read, so both arrive in
  // one memory round trip.
  int j = next_group(-1), base = 0;
  int n_pref = j >= 0 ? group_pieces(p, j, req, h, base) : 0;
  float ls[kB];
  float4 xs[kB];
#pragma unroll
  for (int k = 0; k < kB; ++k) {
    const bool in = k < n_pref;
    ls[k] = in ? ld_cg(prefix_lse(base + k)) : neg_inf();
    xs[k] = in ? ld_cg4(prefix_o(base + k) + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  int suf_kind = 0, suf_begin = 0, suf_n = 0;  // 1: direct state, 2: partial slots
  if (pl) {
    const int nch = pl[p.off_unit_n_chunks + unit];  // both loads in flight together
    const int pbeg = pl[p.off_unit_partial_begin + unit];
    if (nch >= 2) { suf_kind = 2; suf_begin = pbeg; suf_n = nch; }
    else if (nch == 1 && p.suffix_o) { suf_kind = 1; suf_n = 1; }
  } else if (p.suffix_o) {
    suf_kind = 1; suf_n = 1;
  }
  bool preloaded = true;  // ls / xs hold the first batch's prefix pieces
  for (;;) {
    const int jn = j >= 0 ? next_group(j) : -1;
    const int n_suf = jn < 0 ? suf_n : 0;  // the last pass takes the suffix
    const int n_src = n_pref + n_suf;
    auto src_lse = [&](int i) -> const float* {
      if (i < n_pref) return prefix_lse(base + i);
      if (suf_kind == 1) return p.suffix_lse + row_off;
      return p.part_lse + (int64_t)(suf_begin + i - n_pref) * p.hq + h;
    };
    auto src_o = [&](int i) -> const float* {
      if (i < n_pref) return prefix_o(base + i);
      if (suf_kind == 1) return p.suffix_o + row_off * D;
      return p.part_o + ((int64_t)(suf_begin + i - n_pref) * p.hq + h) * D;
    };
    for (int i0 = 0; i0 < n_src; i0 += kB) {
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        if (preloaded && k < n_pref) continue;  // loaded before the plan's words
        const bool in = i0 + k < n_src;
        ls[k] = in ? ld_cg(src_lse(i0 + k)) : neg_inf();
        xs[k] = in ? ld_cg4(src_o(i0 + k) + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      preloaded = false;
      float mb = m;
#pragma unroll
      for (int k = 0; k < kB; ++k) mb = fmaxf(mb, ls[k]);
      if (mb == neg_inf()) continue;
      const float c = ex2((m - mb) * kLog2e);  // 0 when m is -inf
      den *= c;
      acc.x *= c; acc.y *= c; acc.z *= c; acc.w *= c;
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        const float w = ex2((ls[k] - mb) * kLog2e);  // 0 for empty states
        den += w;
        acc.x = fmaf(w, xs[k].x, acc.x); acc.y = fmaf(w, xs[k].y, acc.y);
        acc.z = fmaf(w, xs[k].z, acc.z); acc.w = fmaf(w, xs[k].w, acc.w);
      }
      m = mb;
    }
    preloaded = false;
    if (jn < 0) break;
    j = jn;
    n_pref = group_pieces(p, j, req, h, base);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
  const int64_t row = (int64_t)req * p.hq + h;
  if (p.out_dtype == PKC_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.o) + row * D + lane * 4) = acc;
  } else if (p.out_dtype == PKC_F16) {
    uint2 u = make_uint2(Elem<__half>::from_f2(acc.x, acc.y), Elem<__half>::from_f2(acc.z, acc.w));
    *reinterpret_cast<uint2*>(static_cast<__half*>(p.o) + row * D + lane * 4) = u;
  } else {
    uint2 u = make_uint2(Elem<__nv_bfloat16>::from_f2(acc.x, acc.y), Elem<__nv_bfloat16>::from_f2(acc.z, acc.w));
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + row * D + lane * 4) = u;
  }
  if (lane == 0) p.lse[row] = den > 0.f ? m + lg2(den) * kLn2 : neg_inf();
}

// Sources of the pair (req, kvh) that the fused kernels count: the prefix
// pieces of every group holding the request, plus the suffix states the
// decode writes for it (its chunks when split; one direct state in a
// cascade, whose suffix states are merged with the prefix; none for an
// empty request or, outside a cascade, an unsplit one, which the decode
// writes as its final output at once).
__device__ __forceinline__ int fuse_expected(const FuseParams& f, int req, int kvh) {
  int n = 0;
  if (f.plan) {
    const int nch = f.plan[f.off_unit_n_chunks + req];
    n = nch >= 2 ? nch : (nch == 1 && f.suffix_o ? 1 : 0);
  } else if (f.suffix_o) {
    n = 1;
  }
  if (f.prefix_o) {
    for (int j = 0; j < f.n_prefix; ++j) {
      if (!in_group(f, j, req)) continue;
      int base;
      n += group_pieces(f, j, req, kvh * f.g, base);
    }
  }
  return n;
}

// One source of (req, kvh) written by this thread (and the threads it has
// synchronised with): count it.  True for the thread whose count was the
// pair's last; that thread's view then includes every source.
__device__ __forceinline__ bool fuse_count(const FuseParams& f, int req, int kvh) {
  const int expected = fuse_expected(f, req, kvh);
  __threadfence();  // the sources written so far are visible before the count
  const int before = atomicAdd(f.arrive + (int64_t)req * f.hkv + kvh, 1);
  return before == expected - 1;
}

// (+) of the G rows of (req, kvh) into the final output, by one warp.
__device__ __forceinline__ void fuse_merge(const FuseParams& f, int req, int kvh, int lane) {
  for (int hd = 0; hd < f.g; ++hd) contract_row(f, req, req, kvh * f.g + hd, lane);
}

// Warp-collective, after the warp has written its source of (req, kvh): the
// count, and the merge if this was the pair's last source.  Not inlined:
// it runs once per work item, and inlined into the decode loops its
// registers would be added to theirs (which then spill).
static __device__ __noinline__ void fuse_arrive(const FuseParams& f, int req, int kvh, int lane) {
  __syncwarp();
  int last = 0;
  if (lane == 0) last = fuse_count(f, req, kvh) ? 1 : 0;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __threadfence();  // every lane reads the other writers' sources after the count
  fuse_merge(f, req, kvh, lane);
}

// Rows with no source at all (an empty request outside every prefix group)
// get the empty state (0, -inf); warp `w` of `n_w` takes every n_w-th
// request.
static __device__ __noinline__ void fuse_write_empty(const FuseParams& f, int w, int n_w, int lane) {
  constexpr int D = PKC_HEAD_DIM;
  for (int req = w; req < f.batch; req += n_w) {
    for (int kvh = 0; kvh < f.hkv; ++kvh) {
      if (fuse_expected(f, req, kvh) != 0) continue;
      // A planned decode writes an unsplit request itself: only empty ones here.
      if (f.plan && f.plan[f.off_unit_n_chunks + req] != 0) continue;
      if (!f.plan && !f.suffix_o) continue;  // not a planned call: nothing to cover
      for (int hd = 0; hd < f.g; ++hd) {
        const int64_t row = (int64_t)req * f.hq + kvh * f.g + hd;
        if (f.out_dtype == PKC_F32)
          *reinterpret_cast<float4*>(static_cast<float*>(f.o) + row * D + lane * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
        else
          *reinterpret_cast<uint2*>(static_cast<uint16_t*>(f.o) + row * D + lane * 4) = make_uint2(0u, 0u);
        if (lane == 0) f.lse[row] = neg_inf();
      }
    }
  }
}

}  // namespace pkc
