// Single-query paged decode with q.k and p.v on the tensor cores.
//
// Same computation as the CUDA-core decode kernel (blog "Cascade Inference",
// algorithm step 2; Hugging Face "Paged attention", decoding path): one
// query per request and head against the request's cached tokens, found
// through the block table, split into KV chunks by the host plan, each
// chunk giving an attention state (MLSys'25 notes, A3 and appendix D).
//
// With grouped query heads the G heads of one KV head form a small dense
// contraction against every K (and V) row.  On the CUDA cores that costs
// 2 G FMAs per loaded element and the kernel runs out of issue slots before
// it runs out of HBM bandwidth.  Here one warp computes, per 16 cached
// tokens of its KV head, S^T = K Q^T and O^T += V^T P^T with m16n8k16
// tensor-core tiles: the tokens (and the head dims) are the M side, the G
// query heads the N = 8 side, so G <= 8 costs the same as G = 1.  The
// query heads fused per KV head follow the MLSys'25 notes, appendix A.
//
// FP8 KV (MLSys'25 notes, appendix F, "FP8-FP16 mixed-precision
// attention"): the cache holds e4m3 codes, queries and outputs stay fp16.
// The tile loader stays byte-wide; each warp converts its fragments to fp16
// in registers (two codes per conversion instruction, exact), and V's
// fragments, which the tensor core wants paired along the token axis, are
// regrouped with one byte permute per register (the "fragment shuffler").
//
// Block = one planned CTA x HG KV heads (HG = 8 when Hkv is a multiple of 8).
//  * Warp 8 (producer): as in the CUDA-core kernel, page slices of up to 16
//    slots are copied by TMA into a shared-memory ring, now as
//    [slice][dim half][head][slot] 128-byte lines with the 128-byte swizzle,
//    so the 8 rows of every 8x8 fragment matrix fall in distinct banks.
//    Each stage carries a header and a mask of its valid slots.
//  * Warps 0..7 (consumers): warp w owns KV head w % HG and 16 slots of
//    every stage.  Softmax is online in base 2 with a lazily moved
//    reference maximum: the reference moves (and O is rescaled) only when a
//    stage's maximum exceeds it by more than 8, so P <= 2^8.  P enters the
//    P.V product as a 16-bit high part plus a 16-bit remainder (two MMAs),
//    which keeps it accurate to about 2^-16 relative.  K and V of slots
//    outside the sequence may hold anything (even NaN): their scores are
//    replaced by -inf and their V fragments are zeroed before the MMA.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <type_traits>

#include "contract_common.cuh"
#include "decode_common.cuh"
#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

constexpr int D = PKC_HEAD_DIM;
constexpr int kWarps = 8;                   // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kRows = 128;                  // (slot, head) rows per stage and tensor
constexpr int kMaxSl = 16;                  // slots per slice
constexpr int kLine = 128;                  // bytes per swizzled shared-memory line
constexpr float kRefFloor = -1e30f;         // reference maximum before the first token
constexpr float kLazy = 8.f;                // log2 of the largest P between rescales

enum : int { kFirst = 1, kLast = 2, kDone = 4 };

struct Hdr {
  int32_t flags, req, slot, hg;
  uint32_t mask[kRows / 32];  // valid stage slots
};

template <int KV> struct KvTraits;
template <> struct KvTraits<kKvF16> {
  using Q = __half;  // query and P operand type
  static constexpr int kBytes = 2;
};
template <> struct KvTraits<kKvBF16> {
  using Q = __nv_bfloat16;
  static constexpr int kBytes = 2;
};
template <> struct KvTraits<kKvE4M3> {
  using Q = __half;
  static constexpr int kBytes = 1;
};

template <int KV, int HG>
struct Cfg {
  static constexpr bool kFp8 = KvTraits<KV>::kBytes == 1;
  static constexpr int kRowBytes = D * KvTraits<KV>::kBytes;  // one token of one head
  static constexpr int kTensor = kRows * kRowBytes;           // K (or V) bytes per stage
  static constexpr int kStages = kFp8 ? (HG == 8 ? 6 : 4) : (HG == 8 ? 3 : 2);
  static constexpr int kWph = kWarps / HG;                    // warps per KV head
  static constexpr int kHdr = kStages * 2 * kTensor;
  static constexpr int kBars = kHdr + kStages * (int)sizeof(Hdr);
  static constexpr int kMergeBars = kBars + 2 * kStages * 8;
  static constexpr int kAbort = kMergeBars + 2 * 8;
  static constexpr int kMerge = (kAbort + 16 + 15) & ~15;
};

// Shared memory: stages, headers, barriers, abort flag, then (warps sharing
// a KV head) two merge buffers of 8 warps x G heads x (D + 2) floats.
template <int KV, int G, int HG>
constexpr int mma_fuse_offset() {  // the block's copy of the fused contraction's parameters
  return (Cfg<KV, HG>::kMerge + (Cfg<KV, HG>::kWph > 1 ? 2 * kWarps * G * (D + 2) * 4 : 0) + 15) & ~15;
}
template <int KV, int G, int HG>
constexpr int mma_smem_bytes() {
  return mma_fuse_offset<KV, G, HG>() + (int)sizeof(FuseParams) + 1024;
}
static_assert(mma_smem_bytes<kKvBF16, 8, 4>() <= 227 * 1024, "shared memory");
static_assert(mma_smem_bytes<kKvE4M3, 8, 4>() <= 227 * 1024, "shared memory");
static_assert(mma_smem_bytes<kKvBF16, 8, 8>() <= 227 * 1024, "shared memory");
static_assert(mma_smem_bytes<kKvE4M3, 8, 8>() <= 227 * 1024, "shared memory");

__device__ __forceinline__ float shfl_max_rows(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
}
__device__ __forceinline__ float shfl_sum_rows(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  return v + __shfl_xor_sync(0xffffffffu, v, 16);
}

// The item's accumulators and query fragments after its state is written:
// the next item's first stage sets them again, so clearing them lets the
// fused contraction's merge reuse their registers.
__device__ __forceinline__ void clear_item_regs(float (&o)[8][4], uint32_t (&qf)[8][2]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    qf[i][0] = qf[i][1] = 0u;
  }
}

template <int KV, int G, int HG, bool kFuse>
__global__ void __launch_bounds__(kThreads, 1)
    paged_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                            const __grid_constant__ DecodeParams p) {
  using C = Cfg<KV, HG>;
  using T = typename KvTraits<KV>::Q;
  constexpr bool kFp8 = C::kFp8;
  constexpr int kStages = C::kStages;
  constexpr int kWph = C::kWph;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_kv = smem_u32(smem);  // stage s: K at s * 2 * kTensor, V at + kTensor
  Hdr* hdrs = reinterpret_cast<Hdr*>(smem + C::kHdr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBars);
  uint64_t* empty = full + kStages;
  uint64_t* merge_bar = reinterpret_cast<uint64_t*>(smem + C::kMergeBars);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kAbort);
  float* merge_buf = reinterpret_cast<float*>(smem + C::kMerge);
  FuseParams* fuse = reinterpret_cast<FuseParams*>(smem + mma_fuse_offset<KV, G, HG>());
  if constexpr (kFuse) fuse_params_to_smem(p.fuse, fuse);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int n_hg_mine = (p.hkv / HG - (int)blockIdx.y + (int)gridDim.y - 1) / (int)gridDim.y;
  const int32_t* pl = p.plan;
  // Word `lane` of the plan's header, one load per lane: the device-plan
  // check and the producer's set-up read the header from here, so a block's
  // first item costs one round trip less.
  const int32_t hw = pl ? pl[lane] : 0;
  if (pl && !device_plan_header_ok(hw, p.plan_words, p.batch)) {  // uniform: before any barrier
    if (threadIdx.x == 0) report(p.status, PKC_ERR_PLAN);
    grid_wait_prerequisites();  // as at every exit of this kernel
    return;
  }
  int w_begin = 0, w_end = 1;
  if (pl && !p.dynamic) {  // the static schedule's CTA list
    const int32_t* cta_indptr = pl + __shfl_sync(0xffffffffu, hw, PKC_PLAN_OFF_CTA_INDPTR);
    w_begin = cta_indptr[cta];
    w_end = cta_indptr[cta + 1];
  }
  const int ps = p.page_size;
  const int sl = ps < kMaxSl ? ps : kMaxSl;             // slots per slice
  const uint32_t half_bytes = (uint32_t)(sl * HG * kLine);  // one 64-dim half (16-bit) of a slice
  const uint32_t slice_bytes = (uint32_t)(sl * HG * C::kRowBytes);

  // A contraction launched after this grid as its programmatic dependent
  // may be scheduled from here on (it waits for this grid to finish before
  // it reads what this grid writes).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kWarps);
    }
    mbar_init(smem_u32(&merge_bar[0]), kWarps);
    mbar_init(smem_u32(&merge_bar[1]), kWarps);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------ producer ------------------------------
    const int spp = (ps + sl - 1) / sl;                 // slices per page
    const int slices_per_stage = kRows / (sl * HG);
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) { prefetch_tmap(&tm_k); prefetch_tmap(&tm_v); }
    int k = 0;  // stage counter
    bool ok = true;
    auto acquire = [&](int kk) -> int {
      const int s = kk % kStages;
      bool got = true;
      if (lane == 0) got = mbar_wait(smem_u32(&empty[s]), ((kk / kStages) & 1) ^ 1, abort, p.status);
      got = __shfl_sync(0xffffffffu, got, 0);
      return got ? s : -1;
    };
    // Items: this CTA's plan list (or its request) for each of its head
    // groups; or, scheduled dynamically, tickets from the shared queue, the
    // next one taken once the current item's last stage is issued (a block
    // holds no second ticket while it works through a long chunk).
    const bool dyn = p.dynamic && pl;
    const int n_w = w_end - w_begin;
    DecodeItemWindow items;
    DecodeQueue queue(p, HG, dyn, hw);
    DecodeItem item{0, 0, 0, -1}, item_n{0, 0, 0, -1};
    int hg = (int)blockIdx.y, hg_n = 0, it = 0;
    bool have = dyn ? queue.take(p, lane, item, hg) : n_hg_mine * n_w > 0;
    if (!dyn && have) item = items.get(p, cta, w_begin, n_w, 0, lane);
    while (ok && have) {
      const int req = item.req, kb = item.kb, ke = item.ke, slot = item.slot;
      bool have_n = false;
      const int32_t* bt_row = p.block_table + (int64_t)req * p.bt_stride;
      const int n_pages_used = (ke + ps - 1) / ps;
      int win_base = -1 << 30;
      int32_t win_pid = -1;
      const int first = kb < ke ? (kb / ps) * spp + (kb % ps) / sl : 0;
      const int last = kb < ke ? ((ke - 1) / ps) * spp + ((ke - 1) % ps) / sl : -1;
      int sl0 = first;
      bool first_stage = true;
      do {
        const int s = acquire(k);
        if (s < 0) { ok = false; break; }
        const int n_sl = min(slices_per_stage, last - sl0 + 1);  // may be <= 0 for empty items
        Hdr& h = hdrs[s];
        const uint32_t kst = s_kv + s * 2 * C::kTensor;
        const uint32_t bar = smem_u32(&full[s]);
        uint32_t maskw[kRows / 32];
#pragma unroll
        for (int q = 0; q < kRows / 32; ++q) maskw[q] = 0;
        for (int i = 0; i < n_sl; ++i) {
          const int sli = sl0 + i;
          const int page_idx = sli / spp;
          const int slot0 = (sli % spp) * sl;
          if (page_idx < win_base || page_idx >= win_base + 32) {
            win_base = page_idx;
            const int pi = win_base + lane;
            win_pid = pi < n_pages_used ? bt_row[pi] : -1;
          }
          const int32_t pid = __shfl_sync(0xffffffffu, win_pid, page_idx - win_base);
          if (pid < 0 || pid >= p.num_pages) {
            if (lane == 0) report(p.status, PKC_ERR_BLOCK_TABLE);
            continue;  // slots stay invalid, nothing is copied
          }
          if (lane == 0) {
            mbar_expect_tx(bar, 2 * slice_bytes);  // before the copies it covers
            const uint32_t kd = kst + i * slice_bytes, vd = kd + C::kTensor;
            tma_load_4d(kd, &tm_k, bar, 0, slot0, hg * HG, pid, pol);
            tma_load_4d(vd, &tm_v, bar, 0, slot0, hg * HG, pid, pol);
            if constexpr (!kFp8) {  // second 64-dim half of each 256-byte row
              tma_load_4d(kd + half_bytes, &tm_k, bar, 64, slot0, hg * HG, pid, pol);
              tma_load_4d(vd + half_bytes, &tm_v, bar, 64, slot0, hg * HG, pid, pol);
            }
          }
          // valid slots: those inside the page and inside [kb, ke)
          const int tok0 = page_idx * ps + slot0;
          mask_range(maskw, i * sl + max(kb - tok0, 0), i * sl + min(min(ke - tok0, sl), ps - slot0));
        }
        sl0 += slices_per_stage;
        const bool last_stage = sl0 > last;
        if (lane == 0) {
          h.flags = (first_stage ? kFirst : 0) | (last_stage ? kLast : 0);
          h.req = req;
          h.slot = slot;
          h.hg = hg;
#pragma unroll
          for (int q = 0; q < kRows / 32; ++q) h.mask[q] = maskw[q];
          mbar_arrive(bar);  // header written; the copies carry their own bytes
        }
        __syncwarp();
        if (dyn && last_stage) have_n = queue.take(p, lane, item_n, hg_n);
        first_stage = false;
        ++k;
      } while (sl0 <= last);
      if (dyn) {
        have = have_n;
        item = item_n;
        hg = hg_n;
      } else {
        ++it;
        have = it < n_hg_mine * n_w;
        hg = (int)blockIdx.y + (int)gridDim.y * (it / max(n_w, 1));
        if (have) item = items.get(p, cta, w_begin, n_w, it % n_w, lane);
      }
    }
    if (ok) {  // no more work
      const int s = acquire(k);
      if (s >= 0 && lane == 0) {
        hdrs[s].flags = kDone;
        mbar_arrive(smem_u32(&full[s]));
      }
    }
    if (*abort && lane == 0) {
      // Let the copies already issued land before the block exits.
      volatile int no_abort = 0;
      for (int kk = k > kStages ? k - kStages : 0; kk < k; ++kk)
        mbar_wait(smem_u32(&full[kk % kStages]), (kk / kStages) & 1, &no_abort, p.status);
    }
    if (dyn) queue.finish(lane);
    // A cascade's decode runs next to the prefix stage (launched as its
    // programmatic dependent): no block of this grid finishes before that
    // grid has, so the contraction that waits for this grid sees the prefix
    // pieces too.  (At once when the decode was launched normally.)
    grid_wait_prerequisites();
    return;
  }

  // ------------------------------ consumers ------------------------------
  // Fused contraction: rows that no kernel will write (empty requests) get
  // the empty state, spread over the blocks' first consumer warps.
  if (kFuse && warp == 0)
    fuse_write_empty(fuse, (int)(blockIdx.x + gridDim.x * blockIdx.y), (int)(gridDim.x * gridDim.y), lane);
  const int hh = warp % HG;   // KV head within the group
  const int cls = warp / HG;  // which 16 slots of each stage
  const int g = lane >> 2, tg = lane & 3;  // fragment row group / thread in group
  const int r8 = lane & 7, mi = lane >> 3;  // ldmatrix: row and matrix this lane addresses
  // Shared-memory line of this warp's token t (stage slot 16 cls + t) for
  // head hh: byte offset within a stage tensor and its swizzle key.
  auto line_of = [&](int t, uint32_t& off, uint32_t& key) {
    const int st = 16 * cls + t;
    const int line = hh * sl + st % sl;
    off = (uint32_t)((st / sl) * slice_bytes + line * kLine);
    key = (uint32_t)(line & 7);
  };
  // K fragments: matrices (tokens 0-7 | 8-15) x (chunk c | c+1).  V: the
  // 16-bit path pairs (tokens 0-7 | 8-15) with (dims lo | hi) of one m-tile;
  // the fp8 path uses the same order as K.
  uint32_t k_off, k_key, v_off, v_key;
  line_of(r8 + 8 * (mi & 1), k_off, k_key);
  line_of(kFp8 ? r8 + 8 * (mi & 1) : r8 + 8 * (mi >> 1), v_off, v_key);
  const uint32_t k_sel = (uint32_t)(mi >> 1);
  const uint32_t v_sel = kFp8 ? (uint32_t)(mi >> 1) : (uint32_t)(mi & 1);

  int kvh = hh, req = 0, out_slot = -1, items_done = 0;
  uint32_t qf[8][2];   // Q^T fragments (B operand), one pair per 16-dim k-step
  float o[8][4];       // O^T fragments: 8 m-tiles of 16 dims x 8 heads
  float m0 = kRefFloor, m1 = kRefFloor, l0 = 0.f, l1 = 0.f;  // heads 2 tg, 2 tg + 1

  for (int k = 0;; ++k) {
    const int s = k % kStages;
    if (!mbar_wait(smem_u32(&full[s]), (k / kStages) & 1, abort, p.status)) break;
    const Hdr& h = hdrs[s];
    const int flags = h.flags;
    if (flags & kDone) break;
    if (flags & kFirst) {
      req = h.req;
      kvh = h.hg * HG + hh;
      out_slot = h.slot;
      const T* qrow = static_cast<const T*>(p.q) + ((int64_t)req * p.hq + kvh * G + (g < G ? g : 0)) * D;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if constexpr (kFp8) {  // dims 16 j + 4 tg .. + 3 (the K bytes' order)
          const uint2 u = *reinterpret_cast<const uint2*>(qrow + 16 * j + 4 * tg);
          qf[j][0] = g < G ? u.x : 0u;
          qf[j][1] = g < G ? u.y : 0u;
        } else {               // dims 16 j + 2 tg (+1) and + 8
          qf[j][0] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * j + 2 * tg) : 0u;
          qf[j][1] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * j + 2 * tg + 8) : 0u;
        }
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      m0 = m1 = kRefFloor;
      l0 = l1 = 0.f;
    }
    const uint32_t wm = (h.mask[(16 * cls) >> 5] >> ((16 * cls) & 31)) & 0xffffu;  // this warp's slots
    // This warp's K and V fragments go to registers first.  With a 16-bit
    // cache the slot is released before the dependent QK -> softmax -> PV
    // chain, so the producer refills it that much earlier (2-3 % on the
    // decode); the fp8 ring, 6 stages deep, was faster releasing after it.
    constexpr int kNf = kFp8 ? 4 : 8;
    uint32_t kf[kNf][4], vf[kNf][4];
    if (wm != 0u) {
      const uint32_t kst = s_kv + s * 2 * C::kTensor, vst = kst + C::kTensor;
#pragma unroll
      for (int j = 0; j < kNf; ++j) {
        const uint32_t c = 2 * j + k_sel;
        if constexpr (!kFp8) ldsm_x4(kst + k_off + (c >> 3) * half_bytes + (((c & 7) ^ k_key) << 4), kf[j]);
        else ldsm_x4(kst + k_off + ((c ^ k_key) << 4), kf[j]);
      }
#pragma unroll
      for (int j = 0; j < kNf; ++j) {
        const uint32_t c = 2 * j + v_sel;
        if constexpr (!kFp8) ldsm_x4_t(vst + v_off + (c >> 3) * half_bytes + (((c & 7) ^ v_key) << 4), vf[j]);
        else ldsm_x4_t(vst + v_off + ((c ^ v_key) << 4), vf[j]);
      }
    }
    if constexpr (!kFp8) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    if (wm != 0u) {
      // ---- S^T = K Q^T (16 tokens x 8 heads) ----
      // two accumulators (even / odd 16-dim steps): half the dependent MMA chain
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (!kFp8) {
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          mma16816<T>(sa, kf[j], qf[j][0], qf[j][1]);
          mma16816<T>(sb, kf[j + 1], qf[j + 1][0], qf[j + 1][1]);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t* r = kf[jj];
          const uint32_t a0[4] = {e4m3x2_lo(r[0]), e4m3x2_lo(r[1]), e4m3x2_hi(r[0]), e4m3x2_hi(r[1])};
          mma16816<T>(sa, a0, qf[2 * jj][0], qf[2 * jj][1]);
          const uint32_t a1[4] = {e4m3x2_lo(r[2]), e4m3x2_lo(r[3]), e4m3x2_hi(r[2]), e4m3x2_hi(r[3])};
          mma16816<T>(sb, a1, qf[2 * jj + 1][0], qf[2 * jj + 1][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) sa[i] += sb[i];
      // ---- online softmax, base 2, lazy reference ----
      const bool ok_lo = (wm >> g) & 1u, ok_hi = (wm >> (g + 8)) & 1u;
      const float s0 = ok_lo ? sa[0] * p.scale_log2 : neg_inf();
      const float s1 = ok_lo ? sa[1] * p.scale_log2 : neg_inf();
      const float s2 = ok_hi ? sa[2] * p.scale_log2 : neg_inf();
      const float s3 = ok_hi ? sa[3] * p.scale_log2 : neg_inf();
      const float t0 = shfl_max_rows(fmaxf(s0, s2)), t1 = shfl_max_rows(fmaxf(s1, s3));
      const bool up0 = t0 > m0 + kLazy, up1 = t1 > m1 + kLazy;
      if (__any_sync(0xffffffffu, up0 || up1)) {
        const float n0 = up0 ? t0 : m0, n1 = up1 ? t1 : m1;
        const float c0 = ex2(m0 - n0), c1 = ex2(m1 - n1);
        m0 = n0;
        m1 = n1;
        l0 *= c0;
        l1 *= c1;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          o[mt][0] *= c0; o[mt][1] *= c1; o[mt][2] *= c0; o[mt][3] *= c1;
        }
      }
      const float p0 = ex2(s0 - m0), p1 = ex2(s1 - m1), p2 = ex2(s2 - m0), p3 = ex2(s3 - m1);
      l0 += p0 + p2;
      l1 += p1 + p3;
      // P^T as a 16-bit high part and remainder, transposed into B fragments
      const uint32_t h01 = Elem<T>::from_f2(p0, p1), h23 = Elem<T>::from_f2(p2, p3);
      const float2 f01 = Elem<T>::to_f2(h01), f23 = Elem<T>::to_f2(h23);
      const uint32_t r01 = Elem<T>::from_f2(p0 - f01.x, p1 - f01.y), r23 = Elem<T>::from_f2(p2 - f23.x, p3 - f23.y);
      const uint32_t bh0 = movm_t(h01), bh1 = movm_t(h23), bl0 = movm_t(r01), bl1 = movm_t(r23);
      // V fragments of slots outside the sequence are zeroed (they may be NaN)
      uint32_t vm_lo = 0xffffffffu, vm_hi = 0xffffffffu;
      if (wm != 0xffffu) {
        vm_lo = (((wm >> (2 * tg)) & 1u) ? 0x0000ffffu : 0u) | (((wm >> (2 * tg + 1)) & 1u) ? 0xffff0000u : 0u);
        vm_hi = (((wm >> (2 * tg + 8)) & 1u) ? 0x0000ffffu : 0u) | (((wm >> (2 * tg + 9)) & 1u) ? 0xffff0000u : 0u);
      }
      // ---- O^T += V^T P^T ----
      if constexpr (!kFp8) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a[4] = {vf[mt][0] & vm_lo, vf[mt][1] & vm_lo, vf[mt][2] & vm_hi, vf[mt][3] & vm_hi};
          mma16816<T>(o[mt], a, bh0, bh1);
          mma16816<T>(o[mt], a, bl0, bl1);
        }
      } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const uint32_t* r = vf[jj];
          // r: [token 2tg: dims d, d+1][token 2tg+1: d, d+1], d = 16 c + 2 g.
          // Regroup by dim: low half (d: tokens 2tg, 2tg+1), high half (d+1).
          const uint32_t x0 = prmt(r[0] & vm_lo, 0u, 0x3120u), x1 = prmt(r[1] & vm_hi, 0u, 0x3120u);
          const uint32_t x2 = prmt(r[2] & vm_lo, 0u, 0x3120u), x3 = prmt(r[3] & vm_hi, 0u, 0x3120u);
          const uint32_t a0[4] = {e4m3x2_lo(x0), e4m3x2_hi(x0), e4m3x2_lo(x1), e4m3x2_hi(x1)};
          mma16816<T>(o[2 * jj], a0, bh0, bh1);
          mma16816<T>(o[2 * jj], a0, bl0, bl1);
          const uint32_t a1[4] = {e4m3x2_lo(x2), e4m3x2_hi(x2), e4m3x2_lo(x3), e4m3x2_hi(x3)};
          mma16816<T>(o[2 * jj + 1], a1, bh0, bh1);
          mma16816<T>(o[2 * jj + 1], a1, bl0, bl1);
        }
      }
    }
    if constexpr (kFp8) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    }
    if (!(flags & kLast)) continue;

    // ---- end of a work item: row sums, then write (or merge warps) ----
    const float ls0 = shfl_sum_rows(l0), ls1 = shfl_sum_rows(l1);
    // Head dims held by this lane: m-tile mt rows g and g + 8.
    auto dim_of = [&](int mt, int hi) -> int { return kFp8 ? 16 * mt + 2 * g + hi : 16 * mt + g + 8 * hi; };
    if constexpr (kWph == 1) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hd = 2 * tg + e;
        if (hd >= G) continue;
        const float l = e ? ls1 : ls0, m = e ? m1 : m0;
        const bool has = l > 0.f;
        const float inv = has ? p.v_scale / l : 0.f;
        const float lse = has ? (m + lg2(l)) * kLn2 : neg_inf();
        const int hq = kvh * G + hd;
        if (out_slot >= 0) {
          float* dst = p.part_o + ((int64_t)out_slot * p.hq + hq) * D;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            dst[dim_of(mt, 0)] = o[mt][e] * inv;
            dst[dim_of(mt, 1)] = o[mt][2 + e] * inv;
          }
          if (g == 0) p.part_lse[(int64_t)out_slot * p.hq + hq] = lse;
        } else {
          const int64_t row = (int64_t)req * p.hq + hq;
          if (p.direct_f32) {
            float* dst = static_cast<float*>(p.o_direct) + row * D;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              dst[dim_of(mt, 0)] = o[mt][e] * inv;
              dst[dim_of(mt, 1)] = o[mt][2 + e] * inv;
            }
          } else {
            T* dst = static_cast<T*>(p.o_direct) + row * D;
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              dst[dim_of(mt, 0)] = Elem<T>::from_f(o[mt][e] * inv);
              dst[dim_of(mt, 1)] = Elem<T>::from_f(o[mt][2 + e] * inv);
            }
          }
          if (g == 0) p.lse_direct[row] = lse;
        }
      }
      // A state that is not the request's final output is one source of the
      // fused contraction: count it; the last source's warp merges the pair.
      if (kFuse && (out_slot >= 0 || p.direct_f32)) {
        clear_item_regs(o, qf);
        fuse_arrive<G>(fuse, req, kvh, lane);
      }
    } else {
      // Warps of the same head meet in shared memory (bounded mbarrier wait;
      // buffers alternate between items).
      const int par = items_done & 1;
      float* mbuf = merge_buf + par * kWarps * G * (D + 2);
      float* mine = mbuf + warp * G * (D + 2);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hd = 2 * tg + e;
        if (hd >= G) continue;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          mine[hd * (D + 2) + dim_of(mt, 0)] = o[mt][e];
          mine[hd * (D + 2) + dim_of(mt, 1)] = o[mt][2 + e];
        }
        if (g == 0) {
          mine[hd * (D + 2) + D] = e ? m1 : m0;
          mine[hd * (D + 2) + D + 1] = e ? ls1 : ls0;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&merge_bar[par]));
      const bool met = mbar_wait(smem_u32(&merge_bar[par]), (items_done >> 1) & 1, abort, p.status);
      ++items_done;
      if (!met) break;
      if (cls != 0) continue;
      for (int hd = 0; hd < G; ++hd) {  // lane owns dims 4 lane .. 4 lane + 3
        float mm = kRefFloor;
        for (int c2 = 0; c2 < kWph; ++c2) mm = fmaxf(mm, mbuf[(hh + HG * c2) * G * (D + 2) + hd * (D + 2) + D]);
        float ll = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c2 = 0; c2 < kWph; ++c2) {
          const float* src = mbuf + (hh + HG * c2) * G * (D + 2) + hd * (D + 2);
          const float w = ex2(src[D] - mm);
          ll += src[D + 1] * w;
          acc.x += src[4 * lane] * w; acc.y += src[4 * lane + 1] * w;
          acc.z += src[4 * lane + 2] * w; acc.w += src[4 * lane + 3] * w;
        }
        const bool has = ll > 0.f;
        const float inv = has ? p.v_scale / ll : 0.f;
        acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
        const float lse = has ? (mm + lg2(ll)) * kLn2 : neg_inf();
        const int hq = kvh * G + hd;
        if (out_slot >= 0) {
          *reinterpret_cast<float4*>(p.part_o + ((int64_t)out_slot * p.hq + hq) * D + 4 * lane) = acc;
          if (lane == 0) p.part_lse[(int64_t)out_slot * p.hq + hq] = lse;
        } else {
          const int64_t row = (int64_t)req * p.hq + hq;
          if (p.direct_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(p.o_direct) + row * D + 4 * lane) = acc;
          } else {
            const uint2 u = make_uint2(Elem<T>::from_f2(acc.x, acc.y), Elem<T>::from_f2(acc.z, acc.w));
            *reinterpret_cast<uint2*>(static_cast<T*>(p.o_direct) + row * D + 4 * lane) = u;
          }
          if (lane == 0) p.lse_direct[row] = lse;
        }
      }
      if (kFuse && (out_slot >= 0 || p.direct_f32)) {
        clear_item_regs(o, qf);
        fuse_arrive<G>(fuse, req, kvh, lane);
      }
    }
  }
  grid_wait_prerequisites();  // see the producer's exit
}

template <int KV, int G, int HG, bool kFuse>
int launch_mma_g(const DecodeParams& p, int grid_x, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t st) {
  constexpr int smem = mma_smem_bytes<KV, G, HG>();
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(paged_decode_mma_kernel<KV, G, HG, kFuse>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (attr != cudaSuccess) return (int)attr;
  const dim3 grid(grid_x, p.dynamic ? 1 : p.hkv / HG);
  if (p.after_prefix)  // next to the prefix stage: see the kernel's exits
    return launch_programmatic(paged_decode_mma_kernel<KV, G, HG, kFuse>, grid, dim3(kThreads), smem, st, mk, mv, p);
  paged_decode_mma_kernel<KV, G, HG, kFuse><<<grid, kThreads, smem, st>>>(mk, mv, p);
  return (int)cudaGetLastError();
}

template <int KV, int HG, bool kFuse>
int launch_mma_hg(const DecodeParams& p, int grid_x, const CUtensorMap& mk, const CUtensorMap& mv, cudaStream_t st) {
  switch (p.hq / p.hkv) {
    case 1: return launch_mma_g<KV, 1, HG, kFuse>(p, grid_x, mk, mv, st);
    case 2: return launch_mma_g<KV, 2, HG, kFuse>(p, grid_x, mk, mv, st);
    case 4: return launch_mma_g<KV, 4, HG, kFuse>(p, grid_x, mk, mv, st);
    case 8: return launch_mma_g<KV, 8, HG, kFuse>(p, grid_x, mk, mv, st);
    default: return (int)cudaErrorInvalidValue;
  }
}

template <int KV, bool kFuse>
int launch_mma_kv(const DecodeParams& p, int grid_x, int hg, const CUtensorMap& mk, const CUtensorMap& mv,
                  cudaStream_t st) {
  switch (hg) {
    case 8: return launch_mma_hg<KV, 8, kFuse>(p, grid_x, mk, mv, st);
    case 4: return launch_mma_hg<KV, 4, kFuse>(p, grid_x, mk, mv, st);
    case 2: return launch_mma_hg<KV, 2, kFuse>(p, grid_x, mk, mv, st);
    default: return launch_mma_hg<KV, 1, kFuse>(p, grid_x, mk, mv, st);
  }
}

// The kernels of one contraction mode (kFuse) for a cache kind.
template <bool kFuse>
int launch_mma_mode(const DecodeParams& p, int grid_x, int kv_kind, int hg, const CUtensorMap& mk,
                    const CUtensorMap& mv, cudaStream_t st) {
  switch (kv_kind) {
    case kKvE4M3: return launch_mma_kv<kKvE4M3, kFuse>(p, grid_x, hg, mk, mv, st);
    case kKvBF16: return launch_mma_kv<kKvBF16, kFuse>(p, grid_x, hg, mk, mv, st);
    default: return launch_mma_kv<kKvF16, kFuse>(p, grid_x, hg, mk, mv, st);
  }
}


}  // namespace
}  // namespace pkc
