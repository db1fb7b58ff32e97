// Single-query paged decode state and the contraction of partial states.
//
// Decode (blog "Cascade Inference", algorithm step 2; Hugging Face "Paged
// attention", decoding path): one query per request attends to its cached
// tokens, found through the block table.  There is no KV reuse across
// queries of different requests, so the kernel is bound by HBM bandwidth
// and runs on the CUDA cores (a query tile of one row is below the tensor
// cores' minimum M; MLSys'25 notes, A3 "micro-kernels of different tile
// sizes").  The query heads of one KV head are fused so every K/V row is
// read once for the whole group (MLSys'25 notes, appendix A).  Long
// sequences are split into KV chunks by the host plan; each chunk yields a
// partial state, merged afterwards by the contraction kernel (MLSys'25
// notes, A3: "the final output is the contraction of the partial outputs";
// appendix D: unsplit requests write the output directly).
//
// One thread block = one planned CTA x one group of HG KV heads (HG = 8 when
// Hkv is a multiple of 8).
//  * Warp 8 (producer) walks the block's work items page slice by page
//    slice.  A slice is up to 16 consecutive slots of one page; the TMA
//    engine copies its K and V rows for the HG heads ([slot][head][128],
//    256 bytes per row) into a 3-stage shared-memory ring, one 4-D tile per
//    slice and tensor.  Page ids come from a 32-entry window of the block
//    table that the warp loads in one go.  Each stage carries a header (work
//    item, first/last flags) and a mask of the rows that belong to the item.
//  * Warps 0..7 (consumers) own one KV head each (several warps share a head
//    when HG < 8).  A half-warp reads one 256-byte row from shared memory (16
//    lanes x 16 bytes).  q.k uses two-wide fp32 FMAs; the 16-lane reduction
//    of the G heads' partial dots is a transposed butterfly, after which
//    each lane owns one head's score.  The online softmax (base 2) updates
//    once per stage; P.V accumulates every head's 8 dims per lane.
//  * At the end of a work item the half-warps (and warps sharing a head)
//    merge their states with (+) and write the chunk's state.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <climits>
#include <mutex>

#include "contract_common.cuh"
#include "decode_common.cuh"
#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

constexpr int D = PKC_HEAD_DIM;
constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageRows = 128;            // (slot, head) rows per stage and tensor
constexpr int kRowBytes = D * 2;           // 256 bytes per 16-bit row
constexpr int kStageHalf = kStageRows * kRowBytes;  // 32 KB of K (and of V)
constexpr int kMaxSliceRows = 16;          // slots per slice

enum : int { kFirst = 1, kLast = 2, kDone = 4 };

// Small-batch cascade: the contiguous prefix tensors [prefix tokens, Hkv,
// 128] seen as pages of the cache (pk, pv: one box per page slice, like the
// cache's maps), and as tokens with one box per stage (pk3, pv3: 128 / HG
// tokens x HG heads, the stage's rows in its (slot, head) order).  A stage
// that lies wholly inside the prefix takes one copy per tensor instead of
// one per page slice: the TMA unit issues 4 KB slices one after another, and
// a one-head stage of 8 slices took it about 0.9 us.
struct PrefixMaps {
  CUtensorMap pk, pv, pk3, pv3;
};

struct StageHdr {
  int32_t flags, req, slot, n_rows, hg, pad0, pad1, pad2;
  uint32_t mask[kStageRows / 32];  // valid rows (row-major: slot, head slot)
};

// Ring depth: three 64 KB stages, or two where the merge buffers of warps
// sharing a KV head (HG < 8) at G = 8 leave no room for a third.
template <int G, int HG>
struct DecodeCfg {
  static constexpr int kWph = kConsumerWarps / HG;  // warps per KV head
  static constexpr int kStages = (HG == 8 || G <= 4) ? 3 : 2;
};

// Shared memory, from a 1024-byte aligned base: the K/V stages, the stage
// headers, the full/empty barriers, the abort flag, then (when several warps
// share a KV head) the buffer where those warps merge their states.
template <int G, int HG>
struct DecodeSmem {
  static constexpr int kStages = DecodeCfg<G, HG>::kStages;
  static constexpr int kHdr = kStages * 2 * kStageHalf;
  static constexpr int kBars = kHdr + kStages * (int)sizeof(StageHdr);
  static constexpr int kMergeBars = kBars + 2 * kStages * 8;  // 2 merge barriers
  static constexpr int kAbort = kMergeBars + 2 * 8;
  static constexpr int kMerge = (kAbort + 16 + 15) & ~15;
};

// Two merge buffers (alternating work items) of 8 warps x G heads x (D + 2).
template <int G, int HG>
constexpr int decode_merge_bytes() {
  return DecodeCfg<G, HG>::kWph > 1 ? 2 * kConsumerWarps * G * (D + 2) * 4 : 0;
}
// ... then the block's copy of the fused contraction's parameters.
template <int G, int HG>
constexpr int decode_fuse_offset() {
  return (DecodeSmem<G, HG>::kMerge + decode_merge_bytes<G, HG>() + 15) & ~15;
}
template <int G, int HG>
constexpr int decode_smem_bytes() {
  return decode_fuse_offset<G, HG>() + (int)sizeof(FuseParams) + 1024;
}
static_assert(decode_smem_bytes<4, 1>() <= 227 * 1024, "shared memory");
static_assert(decode_smem_bytes<8, 1>() <= 227 * 1024, "shared memory");
static_assert(decode_smem_bytes<8, 8>() <= 227 * 1024, "shared memory");

// Transposed butterfly over the 16 lanes of a half-warp: in, v[i] is this
// lane's partial dot of head i; out, v[0] is the full dot of head
// (sub >> (4 - log2 G)).
template <int G>
__device__ __forceinline__ float reduce_heads(float (&v)[G], int sub) {
  float a[G];
#pragma unroll
  for (int i = 0; i < G; ++i) a[i] = v[i];
  int n = G;
#pragma unroll
  for (int m = 8; m >= 1; m >>= 1) {
    if (n > 1) {
      const bool up = (sub & m) != 0;
#pragma unroll
      for (int i = 0; i < G / 2; ++i) {
        if (i < n / 2) {
          const float keep = up ? a[i + n / 2] : a[i];
          const float send = up ? a[i] : a[i + n / 2];
          a[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      n >>= 1;
    } else {
      a[0] += __shfl_xor_sync(0xffffffffu, a[0], m);
    }
  }
  return a[0];
}

template <int G>
struct HeadShift {
  static constexpr int v = G == 1 ? 4 : G == 2 ? 3 : G == 4 ? 2 : 1;
};

template <typename T, int G, int HG, bool kFuse>
__global__ void __launch_bounds__(kDecodeThreads, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ PrefixMaps pm,
                        const __grid_constant__ DecodeParams p) {
  using Cfg = DecodeCfg<G, HG>;
  constexpr int kStages = Cfg::kStages;
  constexpr int kWph = Cfg::kWph;
  constexpr int kShift = HeadShift<G>::v;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_kv = smem_u32(smem);  // stage s: K at s*64KB, V at +32KB
  using L = DecodeSmem<G, HG>;
  StageHdr* hdrs = reinterpret_cast<StageHdr*>(smem + L::kHdr);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* empty = full + kStages;
  uint64_t* merge_bar = reinterpret_cast<uint64_t*>(smem + L::kMergeBars);
  volatile int* abort = reinterpret_cast<volatile int*>(smem + L::kAbort);
  float* merge_buf = reinterpret_cast<float*>(smem + L::kMerge);
  FuseParams* fuse = reinterpret_cast<FuseParams*>(smem + decode_fuse_offset<G, HG>());
  if constexpr (kFuse) fuse_params_to_smem(p.fuse, fuse);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  // Head groups of this block: blockIdx.y, blockIdx.y + gridDim.y, ...
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

  // A contraction launched after this grid as its programmatic dependent
  // may be scheduled from here on (it waits for this grid to finish before
  // it reads what this grid writes).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kConsumerWarps);
    }
    mbar_init(smem_u32(&merge_bar[0]), kConsumerWarps);
    mbar_init(smem_u32(&merge_bar[1]), kConsumerWarps);
    *abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------ producer ------------------------------
    const int ps = p.page_size;
    const int sl = ps < kMaxSliceRows ? ps : kMaxSliceRows;      // slots per slice
    const int spp = (ps + sl - 1) / sl;                           // slices per page
    const int slices_per_stage = kStageRows / (sl * HG);
    const uint32_t slice_bytes = (uint32_t)(sl * HG * kRowBytes);
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      if (p.prefix_as_pages) { prefetch_tmap(&pm.pk); prefetch_tmap(&pm.pv); prefetch_tmap(&pm.pk3); prefetch_tmap(&pm.pv3); }
    }
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
      // Small-batch cascade: the request's first pre_pages pages are its shared
      // prefix, page pre_page0 + i of the prefix tensors; the block table
      // lists the rest.
      int pre_page0;
      const int pre_pages = prefix_pages_of(p, req, pre_page0);
      const int n_pages_used = (ke + ps - 1) / ps - pre_pages;  // block-table entries read
      int win_base = -1 << 30;
      int32_t win_pid = -1;
      if (pre_pages > 0) {
        // The first block-table window, loaded now: the load runs while the
        // prefix pages are copied, and is waited for only at the first suffix page.
        const int bi0 = max(kb / ps - pre_pages, 0);
        win_base = bi0;
        win_pid = bi0 + lane < n_pages_used ? bt_row[bi0 + lane] : -1;
      }
      const int first = kb < ke ? (kb / ps) * spp + (kb % ps) / sl : 0;
      const int last = kb < ke ? ((ke - 1) / ps) * spp + ((ke - 1) % ps) / sl : -1;
      int sl0 = first;
      bool first_stage = true;
      do {
        const int s = acquire(k);
        if (s < 0) { ok = false; break; }
        const int n_sl = min(slices_per_stage, last - sl0 + 1);  // may be <= 0 for empty items
        StageHdr& h = hdrs[s];
        const uint32_t kst = s_kv + s * 2 * kStageHalf;
        // Row validity: row j = i*sl*HG + t*HG + hh belongs to slice i, slot t.
        // Lane l handles slices l, l + 32, ... of the stage: its page id, its
        // two copies (each lane raises the stage's byte count for its own
        // copies before issuing them; lane 0 arrives only after the warp has
        // passed the mask reduction below, so the phase cannot complete
        // early) and its rows of the mask.  One lane per slice instead of a
        // loop over the slices: a stage of 8 one-head slices took 2.5 us to
        // issue one slice after another, which a short request waits for.
        uint32_t maskw[kStageRows / 32];
#pragma unroll
        for (int q = 0; q < kStageRows / 32; ++q) maskw[q] = 0;
        // A full stage wholly inside the prefix: one stage-sized box per
        // tensor from the prefix's token view (its rows are the stage's rows
        // in order; every page of it was checked when the call was set up).
        const bool whole_prefix = n_sl == slices_per_stage && (sl0 + n_sl - 1) / spp < pre_pages;
        if (whole_prefix && lane == 0) {
          const int z = (pre_page0 + sl0 / spp) * ps + (sl0 % spp) * sl;  // its first prefix token
          mbar_expect_tx(smem_u32(&full[s]), 2 * kStageHalf);
          tma_load_3d(kst, &pm.pk3, smem_u32(&full[s]), 0, hg * HG, z, pol);
          tma_load_3d(kst + kStageHalf, &pm.pv3, smem_u32(&full[s]), 0, hg * HG, z, pol);
        }
        for (int i0 = 0; i0 < n_sl; i0 += 32) {
          const int i = i0 + lane;
          const bool mine = i < n_sl;
          const int sli = sl0 + i;
          const int page_idx = sli / spp;
          const int slot0 = (sli % spp) * sl;
          const bool in_prefix = page_idx < pre_pages;
          const int bi = page_idx - pre_pages;  // block-table entry (suffix pages)
          const bool need = mine && !in_prefix;
          // These slices lie on at most 32 consecutive pages: a window that
          // starts at the first suffix page among them covers them all.
          if (__any_sync(0xffffffffu, need && (bi < win_base || bi >= win_base + 32))) {
            win_base = __reduce_min_sync(0xffffffffu, need ? bi : INT_MAX);
            const int pi = win_base + lane;
            win_pid = pi < n_pages_used ? bt_row[pi] : -1;
          }
          int32_t pid = __shfl_sync(0xffffffffu, win_pid, need ? bi - win_base : 0);
          if (in_prefix) pid = pre_page0 + page_idx;
          const bool good = mine && pid >= 0 && pid < (in_prefix ? p.prefix_pages : p.num_pages);
          if (mine && !good) report(p.status, PKC_ERR_BLOCK_TABLE);  // rows stay invalid, nothing is copied
          uint32_t mw[kStageRows / 32];
#pragma unroll
          for (int q = 0; q < kStageRows / 32; ++q) mw[q] = 0;
          if (good) {
            if (!whole_prefix) {
              mbar_expect_tx(smem_u32(&full[s]), 2 * slice_bytes);  // before the copies it covers
              const CUtensorMap* mk = in_prefix ? &pm.pk : &tm_k;
              const CUtensorMap* mv = in_prefix ? &pm.pv : &tm_v;
              tma_load_4d(kst + i * slice_bytes, mk, smem_u32(&full[s]), 0, hg * HG, slot0, pid, pol);
              tma_load_4d(kst + kStageHalf + i * slice_bytes, mv, smem_u32(&full[s]), 0, hg * HG, slot0, pid, pol);
            }
            // valid rows: the HG heads of each slot inside the page and inside [kb, ke)
            const int tok0 = page_idx * ps + slot0;
            mask_range(mw, (i * sl + max(kb - tok0, 0)) * HG, (i * sl + min(min(ke - tok0, sl), ps - slot0)) * HG);
          }
#pragma unroll
          for (int q = 0; q < kStageRows / 32; ++q) maskw[q] |= __reduce_or_sync(0xffffffffu, mw[q]);
        }
        sl0 += slices_per_stage;
        const bool last_stage = sl0 > last;
        if (lane == 0) {
          h.flags = (first_stage ? kFirst : 0) | (last_stage ? kLast : 0);
          h.req = req;
          h.slot = slot;
          h.hg = hg;
          h.n_rows = n_sl > 0 ? n_sl * sl * HG : 0;
#pragma unroll
          for (int q = 0; q < kStageRows / 32; ++q) h.mask[q] = maskw[q];
          mbar_arrive(smem_u32(&full[s]));  // header written; the copies carry their own bytes
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
    // Tell the consumers there is no more work.
    if (ok) {
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
  const int half = lane >> 4, sub = lane & 15;
  const int hh = warp % HG;       // KV head within the group
  const int cls = warp / HG;      // which pairs of rows of the stage
  const int src_base = half << 4;
  int kvh = hh;

  uint64_t q2[G][4];
  uint64_t acc[G][4];
  float m_own = neg_inf(), l_own = 0.f;
  int req = 0, out_slot = -1;
  int items_done = 0;  // work items finished by this warp (merge buffer parity)

  for (int k = 0;; ++k) {
    const int s = k % kStages;
    if (!mbar_wait(smem_u32(&full[s]), (k / kStages) & 1, abort, p.status)) break;
    const StageHdr& h = hdrs[s];
    const int flags = h.flags;
    if (flags & kDone) break;
    if (flags & kFirst) {
      req = h.req;
      kvh = h.hg * HG + hh;
      out_slot = h.slot;
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const T* qp = static_cast<const T*>(p.q) + ((int64_t)req * p.hq + kvh * G + gi) * D + sub * 8;
        const uint4 u = *reinterpret_cast<const uint4*>(qp);
        const uint64_t sc2 = pk2(p.scale_log2, p.scale_log2);
        q2[gi][0] = fmul2(widen2<T>(u.x), sc2);
        q2[gi][1] = fmul2(widen2<T>(u.y), sc2);
        q2[gi][2] = fmul2(widen2<T>(u.z), sc2);
        q2[gi][3] = fmul2(widen2<T>(u.w), sc2);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[gi][c] = 0ull;
      }
      m_own = neg_inf();
      l_own = 0.f;
    }
    const int n_rows = h.n_rows;
    uint32_t mask[kStageRows / 32];
#pragma unroll
    for (int q = 0; q < kStageRows / 32; ++q) mask[q] = h.mask[q];
    const uint32_t kst = s_kv + s * 2 * kStageHalf;
    const uint32_t vst = kst + kStageHalf;

    // Rows of this head in the stage: j = 0 .. rows/HG-1 (slot order);
    // warp class `cls` takes token pairs cls, cls + kWph, ...
    float sc[8];
    bool valid[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int tok_in_stage = 2 * (cls + kWph * u) + half;
      const int row = tok_in_stage * HG + hh;
      const bool v = row < n_rows && ((mask[row >> 5] >> (row & 31)) & 1u);
      valid[u] = v;
      uint4 kr = make_uint4(0, 0, 0, 0);
      if (v) kr = lds128(kst + row * kRowBytes + sub * 16);
      const uint64_t k0 = widen2<T>(kr.x), k1 = widen2<T>(kr.y), k2 = widen2<T>(kr.z), k3 = widen2<T>(kr.w);
      float part[G];
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        uint64_t a = fmul2(q2[gi][0], k0);
        a = ffma2(q2[gi][1], k1, a);
        a = ffma2(q2[gi][2], k2, a);
        a = ffma2(q2[gi][3], k3, a);
        const float2 f = upk2(a);
        part[gi] = f.x + f.y;
      }
      const float d = reduce_heads<G>(part, sub);
      sc[u] = v ? d : neg_inf();
    }
    // Online softmax for this lane's head, once per stage.
    float mx = m_own;
#pragma unroll
    for (int u = 0; u < 8; ++u) mx = fmaxf(mx, sc[u]);
    const float corr = mx == neg_inf() ? 1.f : ex2(m_own - mx);
    m_own = mx;
    float pr[8];
    float lsum = 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      pr[u] = valid[u] ? ex2(sc[u] - mx) : 0.f;
      lsum += pr[u];
    }
    l_own = l_own * corr + lsum;
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const float c = __shfl_sync(0xffffffffu, corr, src_base | (gi << kShift));
      const uint64_t c2 = pk2(c, c);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) acc[gi][cc] = fmul2(acc[gi][cc], c2);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int tok_in_stage = 2 * (cls + kWph * u) + half;
      const int row = tok_in_stage * HG + hh;
      uint4 vr = make_uint4(0, 0, 0, 0);
      if (valid[u]) vr = lds128(vst + row * kRowBytes + sub * 16);
      const uint64_t v0 = widen2<T>(vr.x), v1 = widen2<T>(vr.y), v2 = widen2<T>(vr.z), v3 = widen2<T>(vr.w);
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const float pg = __shfl_sync(0xffffffffu, pr[u], src_base | (gi << kShift));
        const uint64_t p2 = pk2(pg, pg);
        acc[gi][0] = ffma2(p2, v0, acc[gi][0]);
        acc[gi][1] = ffma2(p2, v1, acc[gi][1]);
        acc[gi][2] = ffma2(p2, v2, acc[gi][2]);
        acc[gi][3] = ffma2(p2, v3, acc[gi][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    if (!(flags & kLast)) continue;

    // ---- end of a work item: merge half-warps (and warps), write ----
    float mh[G], lh[G];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const float m_a = __shfl_sync(0xffffffffu, m_own, src_base | (gi << kShift));
      const float l_a = __shfl_sync(0xffffffffu, l_own, src_base | (gi << kShift));
      const float m_b = __shfl_xor_sync(0xffffffffu, m_a, 16);
      const float l_b = __shfl_xor_sync(0xffffffffu, l_a, 16);
      const float mm = fmaxf(m_a, m_b);
      const float wa = mm == neg_inf() ? 0.f : ex2(m_a - mm);
      const float wb = mm == neg_inf() ? 0.f : ex2(m_b - mm);
      mh[gi] = mm;
      lh[gi] = l_a * wa + l_b * wb;
      const uint64_t wa2 = pk2(wa, wa), wb2 = pk2(wb, wb);
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const uint64_t other = __shfl_xor_sync(0xffffffffu, acc[gi][cc], 16);
        acc[gi][cc] = ffma2(acc[gi][cc], wa2, fmul2(other, wb2));
      }
    }
    if (kWph > 1) {
      // Warps of the same head meet in shared memory.  The merge barrier is
      // an mbarrier with a bounded wait, so a warp that gave up earlier
      // cannot leave the others waiting; buffers alternate between items.
      const int par = items_done & 1;
      float* mbuf = merge_buf + par * kConsumerWarps * G * (D + 2);
      float* mine = mbuf + warp * G * (D + 2);
      if (half == 0) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const float2 f = upk2(acc[gi][cc]);
            mine[gi * (D + 2) + sub * 8 + 2 * cc] = f.x;
            mine[gi * (D + 2) + sub * 8 + 2 * cc + 1] = f.y;
          }
          if (sub == 0) { mine[gi * (D + 2) + D] = mh[gi]; mine[gi * (D + 2) + D + 1] = lh[gi]; }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&merge_bar[par]));
      const bool met = mbar_wait(smem_u32(&merge_bar[par]), (items_done >> 1) & 1, abort, p.status);
      ++items_done;
      if (!met) break;
      if (cls == 0) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          float mm = neg_inf();
          for (int c2 = 0; c2 < kWph; ++c2) mm = fmaxf(mm, mbuf[(hh + HG * c2) * G * (D + 2) + gi * (D + 2) + D]);
          float ll = 0.f;
          float o8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o8[e] = 0.f;
          if (mm != neg_inf()) {
            for (int c2 = 0; c2 < kWph; ++c2) {
              const float* src = mbuf + (hh + HG * c2) * G * (D + 2) + gi * (D + 2);
              const float w = ex2(src[D] - mm);
              ll += src[D + 1] * w;
#pragma unroll
              for (int e = 0; e < 8; ++e) o8[e] += src[(sub & 15) * 8 + e] * w;
            }
          }
          mh[gi] = mm;
          lh[gi] = ll;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) acc[gi][cc] = pk2(o8[2 * cc], o8[2 * cc + 1]);
        }
      }
      if (cls != 0) continue;
    }
    if (half == 0) {
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        const bool has = lh[gi] > 0.f;
        const float inv = has ? 1.f / lh[gi] : 0.f;
        float o[8];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const float2 f = upk2(acc[gi][cc]);
          o[2 * cc] = f.x * inv;
          o[2 * cc + 1] = f.y * inv;
        }
        const float lse = has ? (mh[gi] + lg2(lh[gi])) * kLn2 : neg_inf();
        const int hq = kvh * G + gi;
        if (out_slot >= 0) {
          float* dst = p.part_o + ((int64_t)out_slot * p.hq + hq) * D + sub * 8;
          *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
          if (sub == 0) p.part_lse[(int64_t)out_slot * p.hq + hq] = lse;
        } else {
          const int64_t row = (int64_t)req * p.hq + hq;
          if (p.direct_f32) {
            float* dst = static_cast<float*>(p.o_direct) + row * D + sub * 8;
            *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4*>(dst + 4) = make_float4(o[4], o[5], o[6], o[7]);
          } else {
            uint4 w;
            w.x = Elem<T>::from_f2(o[0], o[1]); w.y = Elem<T>::from_f2(o[2], o[3]);
            w.z = Elem<T>::from_f2(o[4], o[5]); w.w = Elem<T>::from_f2(o[6], o[7]);
            *reinterpret_cast<uint4*>(static_cast<T*>(p.o_direct) + row * D + sub * 8) = w;
          }
          if (sub == 0) p.lse_direct[row] = lse;
        }
      }
    }
    // A state that is not the request's final output is one source of the
    // fused contraction: count it; the last source's warp merges the pair.
    // (The next item's first stage sets q2 and acc again: cleared, their
    // registers are free for the merge.)
    if (kFuse && (out_slot >= 0 || p.direct_f32)) {
#pragma unroll
      for (int gi = 0; gi < G; ++gi)
#pragma unroll
        for (int c = 0; c < 4; ++c) q2[gi][c] = acc[gi][c] = 0ull;
      fuse_arrive<G>(fuse, req, kvh, lane);
    }
  }
  grid_wait_prerequisites();  // see the producer's exit
}

template <typename T, int G, int HG, bool kFuse>
int launch_decode_g(const DecodeParams& p, int grid_x, const CUtensorMap& mk, const CUtensorMap& mv,
                    const PrefixMaps& pm, cudaStream_t st) {
  constexpr int smem = decode_smem_bytes<G, HG>();
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(paged_decode_kernel<T, G, HG, kFuse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
  });
  if (attr != cudaSuccess) return (int)attr;
  // one block per (planned CTA, head group); one per planned CTA when the
  // blocks take their items from the shared queue
  const dim3 grid(grid_x, p.dynamic ? 1 : p.hkv / HG);
  if (p.after_prefix)  // next to the prefix stage: see the kernel's exits
    return launch_programmatic(paged_decode_kernel<T, G, HG, kFuse>, grid, dim3(kDecodeThreads), smem, st, mk, mv,
                               pm, p);
  paged_decode_kernel<T, G, HG, kFuse><<<grid, kDecodeThreads, smem, st>>>(mk, mv, pm, p);
  return (int)cudaGetLastError();
}

template <typename T, int HG, bool kFuse>
int launch_decode_hg(const DecodeParams& p, int grid_x, const CUtensorMap& mk, const CUtensorMap& mv,
                     const PrefixMaps& pm, cudaStream_t st) {
  switch (p.hq / p.hkv) {
    case 1: return launch_decode_g<T, 1, HG, kFuse>(p, grid_x, mk, mv, pm, st);
    case 2: return launch_decode_g<T, 2, HG, kFuse>(p, grid_x, mk, mv, pm, st);
    case 4: return launch_decode_g<T, 4, HG, kFuse>(p, grid_x, mk, mv, pm, st);
    case 8: return launch_decode_g<T, 8, HG, kFuse>(p, grid_x, mk, mv, pm, st);
    default: return (int)cudaErrorInvalidValue;
  }
}

template <typename T, bool kFuse>
int launch_decode_t(const DecodeParams& p, int grid_x, int hg, const CUtensorMap& mk, const CUtensorMap& mv,
                    const PrefixMaps& pm, cudaStream_t st) {
  switch (hg) {
    case 8: return launch_decode_hg<T, 8, kFuse>(p, grid_x, mk, mv, pm, st);
    case 4: return launch_decode_hg<T, 4, kFuse>(p, grid_x, mk, mv, pm, st);
    case 2: return launch_decode_hg<T, 2, kFuse>(p, grid_x, mk, mv, pm, st);
    default: return launch_decode_hg<T, 1, kFuse>(p, grid_x, mk, mv, pm, st);
  }
}

// The kernels of one contraction mode (kFuse) for a 16-bit cache.
template <bool kFuse>
int launch_simt_mode(const DecodeParams& p, int grid_x, int dtype, int hg, const CUtensorMap& mk,
                     const CUtensorMap& mv, const PrefixMaps& pm, cudaStream_t st) {
  return dtype == PKC_F16 ? launch_decode_t<__half, kFuse>(p, grid_x, hg, mk, mv, pm, st)
                          : launch_decode_t<__nv_bfloat16, kFuse>(p, grid_x, hg, mk, mv, pm, st);
}

}  // namespace
}  // namespace pkc
