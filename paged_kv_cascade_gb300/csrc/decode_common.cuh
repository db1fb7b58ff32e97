// Work items of the paged-decode kernels, read by the producer warp.
//
// A planned CTA's items are entries w_begin .. w_end-1 of the plan's CTA
// work list (see pkc.h, "Load-balanced plan"); without a plan, block x has
// one item: request x, its whole cache.  Lane j of the producer warp holds
// item base + j, so the warp reads the plan for 32 items with one chain of
// dependent loads instead of one chain per item.
#pragma once
#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {

struct DecodeItem {
  int req, kb, ke, slot;  // request, KV range [kb, ke), partial slot or -1
};

// OR the bits [lo, hi) into a W-word mask.  A stage's valid rows are one
// contiguous range per page slice, so the producer builds the mask with a
// few integer operations in registers.  (Marking rows lane by lane into a
// runtime-indexed array put the array in local memory and took an OR over
// the warp: about 1500 cycles per stage, enough to hold the ring back.)
template <int W>
__device__ __forceinline__ void mask_range(uint32_t (&m)[W], int lo, int hi) {
#pragma unroll
  for (int q = 0; q < W; ++q) {
    const int a = max(lo - 32 * q, 0), b = min(hi - 32 * q, 32);
    if (b > a) m[q] |= (b - a == 32 ? 0xffffffffu : ((1u << (b - a)) - 1u)) << a;
  }
}

// Small-batch cascade: the first page (in the prefix tensors' page view)
// and the number of pages of request req's shared prefix (0 outside every
// group).
__device__ __forceinline__ int prefix_pages_of(const DecodeParams& p, int req, int& page0) {
  page0 = 0;
  if (!p.prefix_as_pages) return 0;
  for (int j = 0; j < p.pre_n; ++j) {
    if (p.pre_req_indptr[j] <= req && req < p.pre_req_indptr[j + 1]) {
      page0 = p.pre_kv_indptr[j] / p.page_size;
      return (p.pre_kv_indptr[j + 1] - p.pre_kv_indptr[j]) / p.page_size;
    }
  }
  return 0;
}

// Checks of a planned item against the cache: a plan whose request length
// (plan_len) no longer matches cache_seqlens is reported (PKC_ERR_PLAN) and
// the range is clamped to the cache; a range past the block table is
// reported (PKC_ERR_BLOCK_TABLE) and clamped to the table.
__device__ __forceinline__ DecodeItem checked_item(const DecodeParams& p, DecodeItem d, int plan_len, bool planned) {
  if (planned) {
    const int len = p.cache_seqlens[d.req];
    if (plan_len != len) {
      report(p.status, PKC_ERR_PLAN);
      d.ke = min(d.ke, len);
      d.kb = min(d.kb, d.ke);
    }
  }
  int page0;
  const int pre = prefix_pages_of(p, d.req, page0) * p.page_size;  // prefix tokens ahead of the cache
  if ((int64_t)d.ke - pre > p.bt_stride * p.page_size) {  // more tokens than table entries
    report(p.status, PKC_ERR_BLOCK_TABLE);
    d.ke = pre + (int)(p.bt_stride * p.page_size);
    d.kb = min(d.kb, d.ke);
  }
  return d;
}

// Item wi of this CTA's plan list (valid = wi < w_end), or request `cta`
// without a plan.
__device__ __forceinline__ DecodeItem load_decode_item(const DecodeParams& p, int cta, int wi, bool valid) {
  DecodeItem d{0, 0, 0, -1};
  if (!valid) return d;
  const int32_t* pl = p.plan;
  if (!pl) {
    d.req = cta;
    int page0;
    d.ke = prefix_pages_of(p, cta, page0) * p.page_size + max(p.cache_seqlens[cta], 0);
    return checked_item(p, d, 0, false);
  }
  const int w = pl[pl[PKC_PLAN_OFF_CTA_WORK] + wi];
  const int unit = pl[pl[PKC_PLAN_OFF_WORK_UNIT] + w];
  d.req = pl[pl[PKC_PLAN_OFF_UNIT_REQ] + unit];
  d.kb = pl[pl[PKC_PLAN_OFF_WORK_KV_BEGIN] + w];
  d.ke = pl[pl[PKC_PLAN_OFF_WORK_KV_END] + w];
  d.slot = pl[pl[PKC_PLAN_OFF_WORK_PARTIAL] + w];
  return checked_item(p, d, pl[pl[PKC_PLAN_OFF_UNIT_KV_LEN] + unit], true);
}

// The warp's copy of item li of the CTA's list (0-based), reloading the
// 32-item window (lane j: item base + j) when li falls outside it.
struct DecodeItemWindow {
  DecodeItem mine{0, 0, 0, -1};
  int base = -64;
  __device__ __forceinline__ DecodeItem get(const DecodeParams& p, int cta, int w_begin, int n_w, int li,
                                            int lane) {
    if (li < base || li >= base + 32) {
      base = li & ~31;
      mine = load_decode_item(p, cta, w_begin + base + lane, base + lane < n_w);
    }
    const int src = li - base;
    DecodeItem d;
    d.req = __shfl_sync(0xffffffffu, mine.req, src);
    d.kb = __shfl_sync(0xffffffffu, mine.kb, src);
    d.ke = __shfl_sync(0xffffffffu, mine.ke, src);
    d.slot = __shfl_sync(0xffffffffu, mine.slot, src);
    return d;
  }
};

// The dynamic schedule: the blocks take tickets from a counter in the
// workspace's status block.  Ticket t is chunk t / n_hg of the plan's
// longest-first order (its 16-byte record) for head group t % n_hg, so the
// blocks that run ahead take the short chunks at the end and the blocks
// finish together.  Block b's first ticket is ticket b, taken without the
// counter; the counter hands out the rest (tickets gridDim + 0, 1, ...).
// Each block counts itself out once the queue is empty; the last one resets
// both counters for the next launch (every block reaches that point, on the
// error paths too).
struct DecodeQueue {
  int32_t* ctr;     // [0] tickets handed out by the counter, [1] blocks finished
  const int4* rec;  // order_rec of the plan
  const int32_t* plan_len;
  int n_total, n_hg;
  bool first;       // the block's own first ticket is still to be taken
  // Warp-collective.  hw: word `lane` of the plan's header, which the warp
  // has loaded (the queue's offsets and sizes are header words).
  __device__ __forceinline__ DecodeQueue(const DecodeParams& p, int hg_per_block, bool active, int32_t hw) {
    ctr = nullptr;
    rec = nullptr;
    plan_len = nullptr;
    n_total = 0;
    n_hg = 1;
    first = true;
    if (!active) return;
    const int32_t* pl = p.plan;
    ctr = p.sched;
    rec = reinterpret_cast<const int4*>(pl + __shfl_sync(0xffffffffu, hw, PKC_PLAN_OFF_ORDER_REC));
    plan_len = pl + __shfl_sync(0xffffffffu, hw, PKC_PLAN_OFF_UNIT_KV_LEN);
    n_hg = p.hkv / hg_per_block;
    n_total = __shfl_sync(0xffffffffu, hw, PKC_PLAN_N_WORK) * n_hg;
  }
  // The next ticket's item (all lanes get it), or false once the queue is
  // empty.  A decode plan's unit is its request.
  __device__ __forceinline__ bool take(const DecodeParams& p, int lane, DecodeItem& d, int& hg) {
    int t;
    if (first) {
      first = false;
      t = (int)(blockIdx.x + gridDim.x * blockIdx.y);
    } else {
      int a = 0;
      if (lane == 0) a = atomicAdd(ctr, 1);
      t = __shfl_sync(0xffffffffu, a, 0) + (int)(gridDim.x * gridDim.y);
    }
    if (t < 0 || t >= n_total) return false;
    const int4 r = rec[t / n_hg];
    hg = t % n_hg;
    d = checked_item(p, DecodeItem{r.x, r.y, r.z, r.w}, plan_len[r.x], true);
    return true;
  }
  __device__ __forceinline__ void finish(int lane) {
    if (lane != 0) return;
    __threadfence();
    const int n_blocks = (int)(gridDim.x * gridDim.y);
    if (atomicAdd(ctr + 1, 1) == n_blocks - 1) {
      atomicExch(ctr, 0);
      atomicExch(ctr + 1, 0);
    }
  }
};

}  // namespace pkc
