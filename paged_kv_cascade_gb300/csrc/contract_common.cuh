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
// kernel): the kernels that write the sources count them instead (in the
// kernels' fused instantiations, whose other code is unchanged).  After a
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

// One warp: (+) over every source of rows (req, h0 + r), r < nr <= R, lane i
// owning dims 4i .. 4i+3 of each, written as the final O rows (out_dtype)
// and LSEs.  The rows are query heads of one KV head, so they share one row
// tile of every prefix group and the same sources; they are merged in
// lockstep so that all their loads are in flight together, each row with
// exactly the arithmetic it would get alone.  `unit` is the request's unit
// of the plan (the request itself for decode plans).
// kWaitGrid: the standalone kernel, launched as a programmatic dependent of
// the suffix decode, loads what the decode does not write (the prefix
// pieces, written by a grid it fully depends on, and the plan) first and
// waits for the decode's grid (griddepcontrol.wait) only before its suffix
// loads.
template <int R, class CP, bool kWaitGrid = false>
__device__ __forceinline__ void contract_rows(const CP& p, int req, int unit, int h0, int nr, int lane) {
  constexpr int D = PKC_HEAD_DIM;
  const int32_t* pl = p.plan;
  // Running state of each row's merge: maximum m, denominator den,
  // unnormalised acc.  Sources go in batches whose loads are all in flight
  // together; the running state is rescaled between batches, so the
  // batch size is part of the result's rounding.  It follows the call's G
  // (2 sources per batch when G >= 2, where the standalone kernel takes two
  // rows per warp, else 4), never the rows per warp: every kernel that
  // merges a call's rows then gets the same bits.  kB sizes the arrays; a
  // slot past kb holds the empty state (-inf, 0), which adds exact zeros.
  // (Small batches keep the standalone kernel at few registers and many
  // rows in flight per SM: faster than batches of 8.)
  constexpr int kB = R >= 2 ? 2 : 4;
  const int kb = p.g >= 2 ? 2 : kB;
  float m[R], den[R];
  float4 acc[R];
  int64_t row_off[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    m[r] = neg_inf();
    den[r] = 0.f;
    acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    row_off[r] = (int64_t)req * p.hq + h0 + (r < nr ? r : 0);
  }
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
  // The first group's first batch of prefix pieces depends on no plan word:
  // its loads go out before the plan's words are read, so both arrive in
  // one memory round trip.
  int j = next_group(-1), base = 0;
  int n_pref = j >= 0 ? group_pieces(p, j, req, h0, base) : 0;
  // Launched next to a prefix stage that may still run (a cascade's
  // contraction whose decode followed the prefix as its programmatic
  // dependent), the prefix pieces are ready only once the wait returns.
  bool waited = false;
  if constexpr (kWaitGrid) {
    if (p.prefix_after_wait) {
      grid_wait_prerequisites();
      waited = true;
    }
  }
  float ls[R][kB];
  float4 xs[R][kB];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int k = 0; k < kB; ++k) {
      const bool in = r < nr && k < kb && k < n_pref;
      const int64_t slot = base + k;
      ls[r][k] = in ? ld_cg(p.prefix_lse + slot * p.prefix_stride_lse + row_off[r]) : neg_inf();
      xs[r][k] = in ? ld_cg4(p.prefix_o + slot * p.prefix_stride_o + row_off[r] * D + lane * 4)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
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
  if constexpr (kWaitGrid) {
    if (!waited) grid_wait_prerequisites();
  }
  bool preloaded = true;  // ls / xs hold the first batch's prefix pieces
  for (;;) {
    const int jn = j >= 0 ? next_group(j) : -1;
    const int n_suf = jn < 0 ? suf_n : 0;  // the last pass takes the suffix
    const int n_src = n_pref + n_suf;
    // Source i of row r: its LSE and its O row.
    auto src_lse = [&](int i, int r) -> const float* {
      if (i < n_pref) return p.prefix_lse + (int64_t)(base + i) * p.prefix_stride_lse + row_off[r];
      if (suf_kind == 1) return p.suffix_lse + row_off[r];
      return p.part_lse + (int64_t)(suf_begin + i - n_pref) * p.hq + (row_off[r] - (int64_t)req * p.hq);
    };
    auto src_o = [&](int i, int r) -> const float* {
      if (i < n_pref) return p.prefix_o + (int64_t)(base + i) * p.prefix_stride_o + row_off[r] * D;
      if (suf_kind == 1) return p.suffix_o + row_off[r] * D;
      return p.part_o + ((int64_t)(suf_begin + i - n_pref) * p.hq + (row_off[r] - (int64_t)req * p.hq)) * D;
    };
    for (int i0 = 0; i0 < n_src; i0 += kb) {
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int k = 0; k < kB; ++k) {
          if (preloaded && k < kb && k < n_pref) continue;  // loaded before the plan's words
          const bool in = r < nr && k < kb && i0 + k < n_src;
          ls[r][k] = in ? ld_cg(src_lse(i0 + k, r)) : neg_inf();
          xs[r][k] = in ? ld_cg4(src_o(i0 + k, r) + lane * 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      preloaded = false;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float mb = m[r];
#pragma unroll
        for (int k = 0; k < kB; ++k) mb = fmaxf(mb, ls[r][k]);
        if (mb == neg_inf()) continue;
        // Explicitly rounded operations: the compiler may not contract them
        // differently in different callers, so every caller gets the same bits.
        const float c = ex2(__fmul_rn(m[r] - mb, kLog2e));  // 0 when m is -inf
        den[r] = __fmul_rn(den[r], c);
        acc[r].x = __fmul_rn(acc[r].x, c); acc[r].y = __fmul_rn(acc[r].y, c);
        acc[r].z = __fmul_rn(acc[r].z, c); acc[r].w = __fmul_rn(acc[r].w, c);
#pragma unroll
        for (int k = 0; k < kB; ++k) {
          const float w = ex2(__fmul_rn(ls[r][k] - mb, kLog2e));  // 0 for empty states
          den[r] = __fadd_rn(den[r], w);
          acc[r].x = __fmaf_rn(w, xs[r][k].x, acc[r].x); acc[r].y = __fmaf_rn(w, xs[r][k].y, acc[r].y);
          acc[r].z = __fmaf_rn(w, xs[r][k].z, acc[r].z); acc[r].w = __fmaf_rn(w, xs[r][k].w, acc[r].w);
        }
        m[r] = mb;
      }
    }
    preloaded = false;
    if (jn < 0) break;
    j = jn;
    n_pref = group_pieces(p, j, req, h0, base);
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    if (r >= nr) continue;
    const float inv = den[r] > 0.f ? __frcp_rn(den[r]) : 0.f;
    float4 a = acc[r];
    a.x = __fmul_rn(a.x, inv); a.y = __fmul_rn(a.y, inv); a.z = __fmul_rn(a.z, inv); a.w = __fmul_rn(a.w, inv);
    const int64_t row = row_off[r];
    if (p.out_dtype == PKC_F32) {
      *reinterpret_cast<float4*>(static_cast<float*>(p.o) + row * D + lane * 4) = a;
    } else if (p.out_dtype == PKC_F16) {
      uint2 u = make_uint2(Elem<__half>::from_f2(a.x, a.y), Elem<__half>::from_f2(a.z, a.w));
      *reinterpret_cast<uint2*>(static_cast<__half*>(p.o) + row * D + lane * 4) = u;
    } else {
      uint2 u = make_uint2(Elem<__nv_bfloat16>::from_f2(a.x, a.y), Elem<__nv_bfloat16>::from_f2(a.z, a.w));
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + row * D + lane * 4) = u;
    }
    if (lane == 0) p.lse[row] = den[r] > 0.f ? __fmaf_rn(lg2(den[r]), kLn2, m[r]) : neg_inf();
  }
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

__device__ __forceinline__ int ld_acquire(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One source of (req, kvh) has been written by this thread and the threads
// it has synchronised with: is it the pair's last?  If every other source
// is already counted, it is, and nothing is added (no other writer is
// left); otherwise it is counted, and the count tells.  Either way exactly
// one writer of the pair gets true, and its view then includes every
// source.
__device__ __forceinline__ bool fuse_last(const FuseParams& f, int req, int kvh) {
  const int expected = fuse_expected(f, req, kvh);
  int32_t* ctr = f.arrive + (int64_t)req * f.hkv + kvh;
  if (ld_acquire(ctr) == expected - 1) return true;
  __threadfence();  // the sources written so far are visible before the count
  const bool last = atomicAdd(ctr, 1) == expected - 1;
  if (last) __threadfence();
  return last;
}

// Warp-collective, after the warp has written its source of (req, kvh) (a
// chunk's partial state or a cascade's suffix state): if it was the pair's
// last source, merge the pair's G query-head rows, R at a time in lockstep.
// f is the block's shared-memory copy of the call's FuseParams.  Inlined
// into the fused instantiations of the decode kernels only.
template <int G>
__device__ __forceinline__ void fuse_arrive(const FuseParams* f, int req, int kvh, int lane) {
  __syncwarp();
  int last = 0;
  if (lane == 0) last = fuse_last(*f, req, kvh) ? 1 : 0;
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  __syncwarp();  // lane 0's acquire orders the other lanes' loads too
  constexpr int R = G < 2 ? G : 2;
#pragma unroll 1
  for (int hd = 0; hd < G; hd += R) contract_rows<R>(*f, req, req, kvh * G + hd, R, lane);
}

// Prefix kernel, warp-collective: the warp has written one piece's state of
// the pairs (r0 + i, kvh), i < n (lanes i < n count one pair each); merge
// the pairs whose last source this was, one row at a time.
__device__ __forceinline__ void fuse_arrive_prefix(const FuseParams* f, int r0, int n, int kvh, int lane) {
  __syncwarp();
  const bool last = lane < n && fuse_last(*f, r0 + lane, kvh);
  unsigned lm = __ballot_sync(0xffffffffu, last);
  if (!lm) return;
  __syncwarp();
  const int g = f->g;
  while (lm) {
    const int i = __ffs(lm) - 1;
    lm &= lm - 1;
#pragma unroll 1
    for (int hd = 0; hd < g; ++hd) contract_rows<1>(*f, r0 + i, r0 + i, kvh * g + hd, 1, lane);
  }
}

// Rows with no source at all get the empty state (0, -inf): the plan's
// empty units (requests with no cached token) outside every prefix group;
// without a plan every request has a suffix state.  Warp `w` of `n_w`
// takes every n_w-th empty unit.
__device__ __forceinline__ void fuse_write_empty(const FuseParams* fp, int w, int n_w, int lane) {
  constexpr int D = PKC_HEAD_DIM;
  const FuseParams& f = *fp;
  if (!f.plan) return;
  const int n_split = f.plan[PKC_PLAN_N_SPLIT], n_empty = f.plan[PKC_PLAN_N_EMPTY];
  for (int i = w; i < n_empty; i += n_w) {
    const int unit = f.plan[f.off_unit_list + n_split + i];
    const int req = f.plan[f.off_unit_req + unit];
    for (int kvh = 0; kvh < f.hkv; ++kvh) {
      if (fuse_expected(f, req, kvh) != 0) continue;  // a prefix covers it
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

// Copy of the call's FuseParams into shared memory (the fused helpers read
// it there), by the threads of the block; a __syncthreads() must follow.
__device__ __forceinline__ void fuse_params_to_smem(const FuseParams& f, FuseParams* dst) {
  const int* src = reinterpret_cast<const int*>(&f);
  int* d = reinterpret_cast<int*>(dst);
  for (int i = threadIdx.x; i < (int)(sizeof(FuseParams) / 4); i += blockDim.x) d[i] = src[i];
}

}  // namespace pkc
