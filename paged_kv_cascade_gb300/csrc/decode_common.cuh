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

// Item wi of this CTA (valid = wi < w_end).  A plan whose request length no
// longer matches cache_seqlens is reported (PKC_ERR_PLAN) and its range is
// clamped to the cache; a range past the block table is reported
// (PKC_ERR_BLOCK_TABLE) and clamped to the table.
__device__ __forceinline__ DecodeItem load_decode_item(const DecodeParams& p, int cta, int wi, bool valid) {
  DecodeItem d{0, 0, 0, -1};
  if (!valid) return d;
  const int32_t* pl = p.plan;
  if (pl) {
    const int w = pl[pl[PKC_PLAN_OFF_CTA_WORK] + wi];
    const int unit = pl[pl[PKC_PLAN_OFF_WORK_UNIT] + w];
    d.req = pl[pl[PKC_PLAN_OFF_UNIT_REQ] + unit];
    d.kb = pl[pl[PKC_PLAN_OFF_WORK_KV_BEGIN] + w];
    d.ke = pl[pl[PKC_PLAN_OFF_WORK_KV_END] + w];
    d.slot = pl[pl[PKC_PLAN_OFF_WORK_PARTIAL] + w];
    const int len = p.cache_seqlens[d.req];
    if (pl[pl[PKC_PLAN_OFF_UNIT_KV_LEN] + unit] != len) {
      report(p.status, PKC_ERR_PLAN);
      d.ke = min(d.ke, len);
      d.kb = min(d.kb, d.ke);
    }
  } else {
    d.req = cta;
    d.ke = max(p.cache_seqlens[cta], 0);
  }
  if ((int64_t)d.ke > p.bt_stride * p.page_size) {  // more tokens than table entries
    report(p.status, PKC_ERR_BLOCK_TABLE);
    d.ke = (int)(p.bt_stride * p.page_size);
    d.kb = min(d.kb, d.ke);
  }
  return d;
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

}  // namespace pkc
