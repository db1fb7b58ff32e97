// Multi-query prefix state on the 5th-generation tensor cores.
//
// Blog "Cascade Inference", algorithm step 1 and section "Multi-query vs
// single-query kernels": every request in a group shares the same prefix
// KV, so one thread block loads each KV tile into shared memory once and
// computes all the group's queries against it on the tensor cores.  The
// query rows of a tile are (request, query head) pairs of one KV head, GQA
// heads fused with the request dimension (MLSys'25 notes, appendix A), 128
// rows per tile.
//
// Work split: the KV tiles of all (row tile, KV head) pairs are laid end to
// end and cut evenly over one block per SM (see prefix_block_begin).  A
// block walks its range piece by piece; a piece is the part of one pair
// inside the range and yields a partial state in the pair's partial slot,
// merged by the contraction kernel with (+) (MLSys'25 notes, A3: the final
// output is the contraction of the partial outputs).
//
// Per 128-token KV tile j (FlashAttention-style online softmax, blog
// section "Recursive Attention"):
//   S_j = Q K_j^T              tcgen05.mma, M=N=128, K=128, fp32 in TMEM
//   P_j = exp2(S_j*c - m_ref)  softmax warps: TMEM -> registers -> smem (16b)
//   O  += P_j V_j              tcgen05.mma, P K-major, V MN-major, O in TMEM
// m_ref is a per-row reference maximum.  It changes only when a tile's row
// maximum exceeds it by more than 2^8 (P stays <= 256); then the row's O
// columns are rescaled in TMEM before the next P.V.  With a stable maximum
// nothing touches O until the end of the piece.
// Roles: warp 0 issues TMA loads of each piece's Q tile and of K into a
// 2-slot ring, warp 10 of V into a 2-slot ring, warp 1 allocates TMEM and
// issues MMAs, warps 2..9 own 16 query rows each.  A K slot frees as soon as
// QK has read it, so the K loads run ahead of the softmax; P has two buffers
// of its own (by tile parity), so the softmax of tile j never waits for the
// P.V of tile j - 1.  They read S with the 16x256b TMEM shape, four threads per row and
// two rows per thread, so row maxima and sums are two shuffles and no
// softmax warp waits for another; P goes back to shared memory with
// stmatrix.  The exponent argument S c - m and the row sums use packed
// two-wide fp32 FMAs.  TMEM: S double buffer (2 x 128 columns) + O
// double buffer (2 x 128): a piece's O is read out while the next piece
// accumulates into the other.  All waits are bounded (2 s) and set
// PKC_ERR_TIMEOUT when they run out.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "contract_common.cuh"
#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

constexpr int kRows = 128;       // query rows per tile (MMA M)
constexpr int kKvTile = 128;     // tokens per KV tile (MMA N of S, K of PV)
constexpr int kStagesK = 2;      // K ring: a slot frees once QK has read it
constexpr int kStagesV = 2;      // V ring: a slot frees once P.V has read it
constexpr int kSubTile = 16384;  // 128 rows x 128 bytes (64 elements)
constexpr int kQBytes = 2 * kSubTile;
constexpr int kTileBytes = 2 * kSubTile;  // one K or V tile (two 64-dim halves)
constexpr int kThreads = 352;  // K/Q TMA warp, MMA warp, 8 softmax warps, V TMA warp
constexpr int kVWarp = 10;
constexpr uint32_t kTmemCols = 512;

struct __align__(8) Barriers {
  uint64_t q_full, q_empty;  // a piece's Q tile landed / no longer read
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t p_free[2];        // P buffer b has been read by its last P.V
  uint64_t s_full[2], s_free[2], p_full[2], o_full;
  uint64_t o_done;           // a piece's O is final
  uint64_t o_free[2];        // O buffer b has been read out
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// A piece of a block's range: KV tiles of one (row tile, KV head) pair.
struct Piece {
  int grp, mt, kvh, slot;  // prefix group, row tile within it, KV head, partial slot
  int kv_lo, kv_hi;        // its prefix tokens
  int n;                   // its KV tiles
  int next;                // the flat tile after it
};

// The piece that starts at flat tile x of a block whose range ends at s1.
__device__ __forceinline__ Piece piece_at(const PrefixParams& p, int x, int s1) {
  int j = 0;
  while (j + 1 < p.n_prefix && p.kvt_indptr[j + 1] <= x) ++j;
  const int kvt = (p.kv_indptr[j + 1] - p.kv_indptr[j] + kKvTile - 1) / kKvTile;
  const int off = x - p.kvt_indptr[j];
  const int q = off / kvt, kt0 = off % kvt;
  const int pair0 = p.kvt_indptr[j] + q * kvt;
  const int end = min(s1, pair0 + kvt);
  Piece g;
  g.grp = j;
  g.mt = q / p.hkv;
  g.kvh = q % p.hkv;
  g.slot = p.slot_base[j] + (int)blockIdx.x - prefix_block_of(pair0, p.total_tiles, p.n_blocks);
  g.n = end - x;
  g.kv_lo = p.kv_indptr[j] + kt0 * kKvTile;
  g.kv_hi = min(p.kv_indptr[j + 1], g.kv_lo + g.n * kKvTile);
  g.next = end;
  return g;
}

// Q, P, the K ring, the V ring and the barriers (256 B).  The base must be
// 1024-byte aligned for the 128B-swizzled TMA tiles; with no static shared
// memory it is, and the kernel checks it.
constexpr int kPOffset = kQBytes;                  // two P buffers, by tile parity
constexpr int kKOffset = kPOffset + 2 * kTileBytes;
constexpr int kVOffset = kKOffset + kStagesK * kTileBytes;
constexpr int kBarOffset = kVOffset + kStagesV * kTileBytes;
constexpr int kFuseOffset = kBarOffset + 256;  // the block's copy of the fused contraction's parameters
constexpr int kSmemBytes = kFuseOffset + (int)((sizeof(FuseParams) + 15) & ~size_t(15));
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

template <typename T, bool kFuse>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_state_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ PrefixParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023) != 0) {  // uniform: no thread has started yet
    if (threadIdx.x == 0) report(p.status, PKC_ERR_UNSUPPORTED);
    return;
  }
  // A decode launched after this grid as its programmatic dependent may start
  // now, next to it (it reads nothing this grid writes, and waits for this
  // grid before it exits).
  grid_launch_dependents();
  if (kFuse && p.fuse.plan && !device_plan_ok(p.fuse.plan, p.fuse.plan_words, p.fuse.batch)) {
    if (threadIdx.x == 0) report(p.status, PKC_ERR_PLAN);  // the fused merges would follow its offsets
    return;
  }
  const uint32_t s_q = smem_u32(smem);
  const uint32_t s_p = s_q + kPOffset, s_k0 = s_q + kKOffset, s_v0 = s_q + kVOffset;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kBarOffset);
  FuseParams* fuse = reinterpret_cast<FuseParams*>(smem + kFuseOffset);
  if constexpr (kFuse) fuse_params_to_smem(p.fuse, fuse);
  static_assert(sizeof(Barriers) <= 256, "barrier block");
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.g;
  // This block's flat KV tiles [s0, s1); every role walks the same pieces.
  // (T fits in 32 bits: the host checks it.)
  const int s0 = (int)prefix_block_begin((int)blockIdx.x, p.total_tiles, p.n_blocks);
  const int s1 = (int)prefix_block_begin((int)blockIdx.x + 1, p.total_tiles, p.n_blocks);

  auto bar = [&](uint64_t& b) { return smem_u32(&b); };
  if (threadIdx.x == 0) {
    mbar_init(bar(bars->q_full), 1);
    mbar_init(bar(bars->q_empty), 1);
    for (int s = 0; s < kStagesK; ++s) {
      mbar_init(bar(bars->k_full[s]), 1);
      mbar_init(bar(bars->k_empty[s]), 1);
    }
    for (int s = 0; s < kStagesV; ++s) {
      mbar_init(bar(bars->v_full[s]), 1);
      mbar_init(bar(bars->v_empty[s]), 1);
    }
    mbar_init(bar(bars->p_free[0]), 1);
    mbar_init(bar(bars->p_free[1]), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(bars->s_full[b]), 1);
      mbar_init(bar(bars->s_free[b]), 256);
      mbar_init(bar(bars->p_full[b]), 256);
    }
    mbar_init(bar(bars->o_full), 1);
    mbar_init(bar(bars->o_done), 1);
    mbar_init(bar(bars->o_free[0]), 256);
    mbar_init(bar(bars->o_free[1]), 256);
    mbar_init(bar(bars->drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0 || warp == kVWarp) {
    // ---------------- TMA producers ----------------
    // Warp 0 loads each piece's Q tile and the K tiles into the K ring; warp
    // 10 loads the V tiles into the V ring.  A K slot frees as soon as QK has
    // read it and a V slot once P.V has, so the loads of later tiles never
    // wait for this tile's softmax.  The whole warp runs the loop; lane 0
    // waits on the barriers and the warp learns the result.  A contiguous
    // tile is two boxes from lane 0; a paged tile is two boxes per page,
    // issued by the lanes in parallel.
    const bool is_v = warp == kVWarp;
    const int n_st = is_v ? kStagesV : kStagesK;
    const uint32_t ring0 = is_v ? s_v0 : s_k0;
    uint64_t* full = is_v ? bars->v_full : bars->k_full;
    uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
    const void* tmap = is_v ? (const void*)&tm_v : (const void*)&tm_k;
    const uint64_t pol = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    int g = 0, q_issued = 0;  // tiles and Q tiles issued
    bool ok = true;
    auto wait0 = [&](uint64_t& b, uint32_t parity) -> bool {
      bool got = true;
      if (lane == 0) got = mbar_wait(bar(b), parity, abort, p.status);
      return __shfl_sync(0xffffffffu, got, 0);
    };
    for (int x = s0; ok && x < s1;) {
      const Piece pc = piece_at(p, x, s1);
      x = pc.next;
      auto load_tile = [&](int u) -> bool {
        const int s = g % n_st;
        if (!wait0(empty[s], ((g / n_st) & 1) ^ 1)) return false;
        const uint32_t st = ring0 + s * kTileBytes;
        const uint32_t fb = bar(full[s]);
        const int t0 = pc.kv_lo + u * kKvTile;
        if (lane == 0) mbar_arrive_expect_tx(fb, kTileBytes);
        __syncwarp();
        if (!p.prefix_pages) {
          if (lane == 0) {
            tma_load_3d(st, tmap, fb, 0, pc.kvh, t0, pol);
            tma_load_3d(st + kSubTile, tmap, fb, 64, pc.kvh, t0, pol);
          }
        } else {
          // Box c: page c / 2 of the tile, dims 0-63 or 64-127 by c % 2,
          // {64 dims, 1 head, page_size slots}.  Pages past the group's list
          // load from page num_pages, outside the pool: zero fill.
          const int ps = p.page_size;
          const int rel = t0 - p.kv_indptr[pc.grp];  // token offset within the group
          const int pg0 = p.page_indptr[pc.grp], n_pg = p.page_indptr[pc.grp + 1] - pg0;
          for (int c = lane; c < 2 * (kKvTile / ps); c += 32) {
            const int r = (c >> 1) * ps, half = c & 1;
            const int pi = (rel + r) / ps;
            int32_t page = pi < n_pg ? p.prefix_pages[pg0 + pi] : (int32_t)p.num_pages;
            if (pi < n_pg && (page < 0 || page >= p.num_pages)) {
              report(p.status, PKC_ERR_BLOCK_TABLE);
              page = (int32_t)p.num_pages;  // read as zeros
            }
            tma_load_4d(st + half * kSubTile + (uint32_t)r * 128, tmap, fb, half * 64, pc.kvh, 0, page, pol);
          }
        }
        ++g;
        return true;
      };
      if (is_v) {
        for (int u = 0; ok && u < pc.n; ++u) ok = load_tile(u);
        continue;
      }
      // After the first piece, the K ring fills with this piece's tiles while
      // the previous piece's products still read the Q buffer.
      const int pre = q_issued > 0 ? min(pc.n, n_st) : 0;
      for (int u = 0; ok && u < pre; ++u) ok = load_tile(u);
      if (!ok) break;
      if (q_issued > 0 && !wait0(bars->q_empty, (q_issued - 1) & 1)) break;
      const int b0 = p.req_begin[pc.grp] + pc.mt * (kRows / G);
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(bars->q_full), kQBytes);
        tma_load_3d(s_q, &tm_q, bar(bars->q_full), 0, pc.kvh * G, b0, pol_q);
        tma_load_3d(s_q + kSubTile, &tm_q, bar(bars->q_full), 64, pc.kvh * G, b0, pol_q);
      }
      ++q_issued;
      for (int u = pre; ok && u < pc.n; ++u) ok = load_tile(u);
    }
    if (*abort && lane == 0) {
      // Let the copies already issued land before the block exits.
      volatile int no_abort = 0;
      if (q_issued > 0) mbar_wait(bar(bars->q_full), (q_issued - 1) & 1, &no_abort, p.status);
      for (int jt = g > n_st ? g - n_st : 0; jt < g; ++jt)
        mbar_wait(bar(full[jt % n_st]), (jt / n_st) & 1, &no_abort, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value ? 1 : 0;
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, kBf16, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, 128, kBf16, 0, 1);
      bool ok = true;
      int g = 0, k = 0;  // first KV tile of the piece, piece index
      for (int x = s0; ok && x < s1; ++k) {
        const Piece pc = piece_at(p, x, s1);
        x = pc.next;
        ok = mbar_wait(bar(bars->q_full), k & 1, abort, p.status);
        if (!ok) break;
        tc_fence_after();
        for (int u = 0; ok && u <= pc.n; ++u) {
          if (u < pc.n) {
            const int j = g + u, s = j % kStagesK, b = j & 1;
            ok = mbar_wait(bar(bars->k_full[s]), (j / kStagesK) & 1, abort, p.status) &&
                 mbar_wait(bar(bars->s_free[b]), ((j >> 1) & 1) ^ 1, abort, p.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kb = s_k0 + s * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * kSubTile + (kk & 3) * 32;
              tc_mma_f16(tmem + b * 128, smem_desc_sw128(s_q + off, 16, 1024),
                         smem_desc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0);
            }
            tc_commit(bar(bars->s_full[b]));
            tc_commit(bar(bars->k_empty[s]));                  // K_j read: its slot may refill
            if (u == pc.n - 1) tc_commit(bar(bars->q_empty));  // the piece's last read of Q
          }
          if (u >= 1) {
            const int jp = g + u - 1, sv = jp % kStagesV, bp = jp & 1;
            ok = mbar_wait(bar(bars->p_full[bp]), (jp >> 1) & 1, abort, p.status) &&
                 mbar_wait(bar(bars->v_full[sv]), (jp / kStagesV) & 1, abort, p.status);
            // The first P.V of a piece overwrites O: the previous piece's O
            // must have been read out.
            // (O is double-buffered: piece k uses buffer k & 1, last read
            // out by the epilogue of piece k - 2.)
            if (ok && u == 1 && k > 1) ok = mbar_wait(bar(bars->o_free[k & 1]), ((k >> 1) - 1) & 1, abort, p.status);
            if (!ok) break;
            tc_fence_after();
            const uint32_t pb = s_p + bp * kTileBytes;
            const uint32_t vb = s_v0 + sv * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {  // O accumulates over the piece's tiles
              const uint32_t a_off = (kk >> 2) * kSubTile + (kk & 3) * 32;
              tc_mma_f16(tmem + 256 + (k & 1) * 128, smem_desc_sw128(pb + a_off, 16, 1024),
                         smem_desc_sw128(vb + kk * 2048, kSubTile, 1024), idesc_pv, (u > 1 || kk > 0) ? 1u : 0u);
            }
            tc_commit(bar(bars->o_full));
            tc_commit(bar(bars->v_empty[sv]));
            tc_commit(bar(bars->p_free[bp]));
          }
        }
        if (!ok) break;
        tc_commit(bar(bars->o_done));
        g += pc.n;
      }
      // Drain: every MMA issued above completes before TMEM is released.
      tc_commit(bar(bars->drain));
      volatile int no_abort = 0;
      mbar_wait(bar(bars->drain), 0, &no_abort, p.status);
    }
  } else {
    // ------- softmax: 16 rows per warp, four threads per row -------
    // The 16x256b TMEM shape gives each thread two rows (the warp's rows l
    // and l + 8) and 32 columns of each (pairs 8j + 2c, +1 with c = lane % 4),
    // so a row's maximum and sum take two shuffles among its four threads and
    // no softmax warp ever waits for another.
    const int quad = warp & 3;                // TMEM lane quadrant
    const int hq16 = (warp - 2) >> 2;         // which 16 lanes of the quadrant
    const int rbase = quad * 32 + hq16 * 16;  // the warp's first row
    const int g4 = lane >> 2, c4 = lane & 3;
    const uint32_t lane_base = tmem + ((uint32_t)rbase << 16);
    constexpr float kRescaleLog2 = 8.f;  // move m_ref only when the max grows by > 2^8
    const uint64_t c2 = pk2(p.scale_log2, p.scale_log2), one2 = pk2(1.f, 1.f);
    bool ok = true;
    int g = 0, k = 0;  // first KV tile of the piece, piece index
    for (int x = s0; ok && x < s1; ++k) {
      const int x_piece = x;
      int n_kv, kv_lo, kv_hi;
      {
        const Piece pc = piece_at(p, x, s1);
        x = pc.next;
        n_kv = pc.n;
        kv_lo = pc.kv_lo;
        kv_hi = pc.kv_hi;
      }
      float mt_ref = neg_inf(), mb_ref = neg_inf();  // rows l (top) and l + 8 (bottom)
      uint64_t lt2 = 0ull, lb2 = 0ull;                 // packed row sums
      const uint32_t o_base = lane_base + 256 + (k & 1) * 128;  // this piece's O buffer
      for (int u = 0; u < n_kv; ++u) {
        const int j = g + u, b = j & 1;
        const bool got = ok && mbar_wait(bar(bars->s_full[b]), (j >> 1) & 1, abort, p.status);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        const int vrow = min(kKvTile, kv_hi - (kv_lo + u * kKvTile));  // valid columns
        uint32_t sr[2][32];  // [64-column half][4 j + e]
        tmem_ld_16x256b_x8(lane_base + b * 128, sr[0]);
        tmem_ld_16x256b_x8(lane_base + b * 128 + 64, sr[1]);
        tmem_ld_wait();
        reg_fence32(sr[0]);
        reg_fence32(sr[1]);
        float mt = neg_inf(), mb = neg_inf();
        if (vrow == kKvTile) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              mt = max3(mt, __uint_as_float(sr[h][4 * jj]), __uint_as_float(sr[h][4 * jj + 1]));
              mb = max3(mb, __uint_as_float(sr[h][4 * jj + 2]), __uint_as_float(sr[h][4 * jj + 3]));
            }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int col = 64 * h + 8 * jj + 2 * c4 + (e & 1);
                const float v = __uint_as_float(sr[h][4 * jj + e]);
                if (col < vrow) {
                  if (e < 2) mt = fmaxf(mt, v);
                  else mb = fmaxf(mb, v);
                }
              }
        }
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        const float tt = mt * p.scale_log2, tb = mb * p.scale_log2;
        if (__any_sync(0xffffffffu, tt > mt_ref + kRescaleLog2 || tb > mb_ref + kRescaleLog2)) {
          const float nt = fmaxf(mt_ref, tt), nb = fmaxf(mb_ref, tb);
          const float rt = ex2(mt_ref - nt), rb = ex2(mb_ref - nb);  // 0 while the reference is -inf
          {
            const float2 a = upk2(lt2), c = upk2(lb2);
            lt2 = pk2(a.x * rt, a.y * rt);
            lb2 = pk2(c.x * rb, c.y * rb);
          }
          if (u > 0) {
            // O holds P.V of the piece's tiles < u: wait for the last of them
            // (the S_j commit already covered tile j-2), rescale my rows.
            const bool done = mbar_wait(bar(bars->o_full), (j - 1) & 1, abort, p.status);
            if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
              uint32_t o[32];
              tmem_ld_16x256b_x8(o_base + c * 64, o);
              tmem_ld_wait();
              reg_fence32(o);
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                o[4 * jj] = __float_as_uint(__uint_as_float(o[4 * jj]) * rt);
                o[4 * jj + 1] = __float_as_uint(__uint_as_float(o[4 * jj + 1]) * rt);
                o[4 * jj + 2] = __float_as_uint(__uint_as_float(o[4 * jj + 2]) * rb);
                o[4 * jj + 3] = __float_as_uint(__uint_as_float(o[4 * jj + 3]) * rb);
              }
              tmem_st_16x256b_x8(o_base + c * 64, o);
            }
            tmem_st_wait();
          }
          mt_ref = nt;
          mb_ref = nb;
        }
        // P_j = exp2(S_j c - m_ref) as 16-bit pairs, stored into the P buffer
        // (once P.V of tile j-1 has read it) with stmatrix: matrices (top,
        // octet jj), (bottom, jj), (top, jj+1), (bottom, jj+1); lane l
        // addresses row l % 8 of matrix l / 8.
        {
          // buffer b was last read by P.V of tile j - 2
          const bool free_now = mbar_wait(bar(bars->p_free[b]), ((j >> 1) & 1) ^ 1, abort, p.status);
          if (!__all_sync(0xffffffffu, free_now)) { ok = false; break; }
        }
        const uint32_t pst = s_p + b * kTileBytes;
        const uint64_t nt2 = pk2(-mt_ref, -mt_ref), nb2 = pk2(-mb_ref, -mb_ref);
        const int mrow = rbase + (lane & 7) + 8 * ((lane >> 3) & 1);  // row this lane addresses
        const uint32_t mrow_addr = pst + mrow * 128;
        const uint32_t mkey = (uint32_t)(mrow & 7), moct = (uint32_t)(lane >> 4);
        auto p_half = [&](auto full_tag, const uint32_t (&v)[32], int h) {
          constexpr bool kFull = decltype(full_tag)::value;
          uint32_t pw[16];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int col = 64 * h + 8 * jj + 2 * c4;
            const float2 xt = upk2(ffma2(pk2(__uint_as_float(v[4 * jj]), __uint_as_float(v[4 * jj + 1])), c2, nt2));
            const float2 xb =
                upk2(ffma2(pk2(__uint_as_float(v[4 * jj + 2]), __uint_as_float(v[4 * jj + 3])), c2, nb2));
            float p0 = ex2(xt.x), p1 = ex2(xt.y), p2 = ex2(xb.x), p3 = ex2(xb.y);
            if (!kFull) {
              p0 = col < vrow ? p0 : 0.f;
              p1 = col + 1 < vrow ? p1 : 0.f;
              p2 = col < vrow ? p2 : 0.f;
              p3 = col + 1 < vrow ? p3 : 0.f;
            }
            lt2 = ffma2(pk2(p0, p1), one2, lt2);
            lb2 = ffma2(pk2(p2, p3), one2, lb2);
            pw[2 * jj] = Elem<T>::from_f2(p0, p1);
            pw[2 * jj + 1] = Elem<T>::from_f2(p2, p3);
          }
#pragma unroll
          for (int jj = 0; jj < 8; jj += 2) {
            const uint32_t chunk = (uint32_t)jj + moct;
            stsm_x4(mrow_addr + h * kSubTile + ((chunk ^ mkey) << 4), pw[2 * jj], pw[2 * jj + 1], pw[2 * jj + 2],
                    pw[2 * jj + 3]);
          }
        };
        if (vrow == kKvTile) {
          p_half(std::true_type{}, sr[0], 0);
          p_half(std::true_type{}, sr[1], 1);
        } else {
          p_half(std::false_type{}, sr[0], 0);
          p_half(std::false_type{}, sr[1], 1);
          if (p.prefix_pages) {
            // A paged prefix's last page may hold anything (even NaN) past the
            // prefix: zero those V rows (once the tile has landed) so that
            // P = 0 meets V = 0 in P.V.
            const int sv = j % kStagesV;
            const bool landed = mbar_wait(bar(bars->v_full[sv]), (j / kStagesV) & 1, abort, p.status);
            if (!__all_sync(0xffffffffu, landed)) { ok = false; break; }
            const uint32_t vst = s_v0 + sv * kTileBytes;
            const int n_chunks = (kKvTile - vrow) * 16;  // 16-byte chunks in both 64-dim halves
            for (int c = (int)threadIdx.x - 64; c < n_chunks; c += 256) {
              const int r = vrow + (c >> 4), half = (c >> 3) & 1, ch16 = c & 7;
              asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vst + half * kSubTile + r * 128 + ch16 * 16),
                           "r"(0u)
                           : "memory");
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(bars->p_full[b]));
        mbar_arrive(bar(bars->s_free[b]));
      }
      g += n_kv;
      // O of the piece is final once its last P.V has completed.
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(bars->o_done), k & 1, abort, p.status));
      float lt, lb;
      {
        const float2 a = upk2(lt2), c = upk2(lb2);
        lt = a.x + a.y;
        lb = c.x + c.y;
      }
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lb += __shfl_xor_sync(0xffffffffu, lb, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      lb += __shfl_xor_sync(0xffffffffu, lb, 2);

      // Epilogue: rows that belong to the piece's group write its state.
      const Piece pc = piece_at(p, x_piece, s1);
      const int b0 = p.req_begin[pc.grp] + pc.mt * (kRows / G);
      const int req_hi = min(p.req_end[pc.grp], p.batch);
      const int rt_row = rbase + g4, rb_row = rt_row + 8;
      const int bt = b0 + rt_row / G, bb = b0 + rb_row / G;
      const bool mine_t = bt < req_hi, mine_b = bb < req_hi;
      const int64_t r_t = (int64_t)bt * p.hq + pc.kvh * G + rt_row % G;
      const int64_t r_b = (int64_t)bb * p.hq + pc.kvh * G + rb_row % G;
      float* out_t = p.out_o + pc.slot * p.split_stride_o + r_t * PKC_HEAD_DIM;
      float* out_b = p.out_o + pc.slot * p.split_stride_o + r_b * PKC_HEAD_DIM;
      const bool has_t = ok && lt > 0.f, has_b = ok && lb > 0.f;
      const float inv_t = has_t ? 1.f / lt : 0.f, inv_b = has_b ? 1.f / lb : 0.f;
      if (ok) tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        if (ok) {  // warp-uniform
          tmem_ld_16x256b_x8(o_base + c * 64, o);
          tmem_ld_wait();
          reg_fence32(o);
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int col = 64 * c + 8 * jj + 2 * c4;
          if (mine_t)
            *reinterpret_cast<float2*>(out_t + col) =
                has_t ? make_float2(__uint_as_float(o[4 * jj]) * inv_t, __uint_as_float(o[4 * jj + 1]) * inv_t)
                      : make_float2(0.f, 0.f);
          if (mine_b)
            *reinterpret_cast<float2*>(out_b + col) =
                has_b ? make_float2(__uint_as_float(o[4 * jj + 2]) * inv_b, __uint_as_float(o[4 * jj + 3]) * inv_b)
                      : make_float2(0.f, 0.f);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(bars->o_free[k & 1]));  // piece k + 2 may overwrite this O buffer
      if (c4 == 0) {
        if (mine_t) p.out_lse[pc.slot * p.split_stride_lse + r_t] = has_t ? (mt_ref + lg2(lt)) * kLn2 : neg_inf();
        if (mine_b) p.out_lse[pc.slot * p.split_stride_lse + r_b] = has_b ? (mb_ref + lg2(lb)) * kLn2 : neg_inf();
      }
      // Fused contraction: the piece is one source of every (request, KV
      // head) pair among the warp's 16 rows (16 / G requests, whose G rows
      // all lie here).  Lane i counts request i; the warp merges the pairs
      // whose count was the last.
      if (kFuse && ok) {
        const int r0 = b0 + rbase / G;
        fuse_arrive_prefix(fuse, r0, max(0, min(16 / G, req_hi - r0)), pc.kvh, lane);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// 3-D tiled map over a row-major [d2][d1][d0] tensor of 16-bit elements
// with a {64, box1, box2} box and 128-byte swizzle (rows of 128 bytes).
bool make_map(CUtensorMap* m, const void* base, int dtype, uint64_t d0, uint64_t d1, uint64_t d2,
              uint32_t box1, uint32_t box2) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const uint32_t box[3] = {64, box1, box2};
  return encode_tiled_map(m, base, dtype, 3, dims, strides, box, true);
}

template <typename T, bool kFuse>
int launch_tf(const PrefixParams& p, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
              cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefix_state_kernel<T, kFuse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return (int)attr_err;
  const dim3 grid(p.n_blocks, 1);  // one block per SM, each over an even share of the KV tiles
  prefix_state_kernel<T, kFuse><<<grid, kThreads, kSmemBytes, st>>>(q, k, v, p);
  return (int)cudaGetLastError();
}

template <typename T>
int launch_t(const PrefixParams& p, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
             cudaStream_t st) {
  return p.fuse.enabled ? launch_tf<T, true>(p, q, k, v, st) : launch_tf<T, false>(p, q, k, v, st);
}

}  // namespace

int launch_prefix(const PrefixParams& p, const void* q, const void* k_prefix, const void* v_prefix,
                  int64_t prefix_tokens, int dtype, void* stream, void* start_event) {
  cudaStream_t st = (cudaStream_t)stream;
  if (p.n_blocks <= 0 || p.total_tiles <= 0) {
    if (start_event) return (int)cudaEventRecord((cudaEvent_t)start_event, st);
    return 0;
  }
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, dtype, PKC_HEAD_DIM, p.hq, p.batch, p.g, kRows / p.g)) return -1;
  if (!p.prefix_pages) {
    if (!make_map(&mk, k_prefix, dtype, PKC_HEAD_DIM, p.hkv, prefix_tokens, 1, kKvTile) ||
        !make_map(&mv, v_prefix, dtype, PKC_HEAD_DIM, p.hkv, prefix_tokens, 1, kKvTile))
      return -1;
  } else {
    // 4-D view (dim, head, slot, page) of the pool [num_pages][page_size][Hkv][128];
    // a box is one head's page_size slots of one page, 64 dims (128 bytes) wide.
    const uint64_t dims[4] = {(uint64_t)PKC_HEAD_DIM, (uint64_t)p.hkv, (uint64_t)p.page_size,
                              (uint64_t)(p.num_pages > 0 ? p.num_pages : 1)};
    const uint64_t strides[3] = {(uint64_t)PKC_HEAD_DIM * 2, (uint64_t)PKC_HEAD_DIM * 2 * p.hkv,
                                 (uint64_t)PKC_HEAD_DIM * 2 * p.hkv * p.page_size};
    const uint32_t box[4] = {64u, 1u, (uint32_t)p.page_size, 1u};
    if (!encode_tiled_map(&mk, k_prefix, dtype, 4, dims, strides, box, true) ||
        !encode_tiled_map(&mv, v_prefix, dtype, 4, dims, strides, box, true))
      return -1;
  }
  if (start_event) {  // recorded after the host work above, right before the launch
    if (const cudaError_t e = cudaEventRecord((cudaEvent_t)start_event, st)) return (int)e;
  }
  return dtype == PKC_BF16 ? launch_t<__nv_bfloat16>(p, mq, mk, mv, st)
                           : launch_t<__half>(p, mq, mk, mv, st);
}

}  // namespace pkc
