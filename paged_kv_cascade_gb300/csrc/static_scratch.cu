// Paged decode for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc when they run the decode:
// code that lives inside another framework's memory pool (an inference
// server that hands out all device memory at start-up and forbids later
// allocations), plug-ins that only receive tensors, and hosts on a fixed,
// pre-reserved memory budget.  They cannot provide the workspace that
// pkc_paged_decode_state needs for the split-KV partial states.  This entry
// point runs the same kernels with the workspace placed in a fixed-size
// array that the library itself declares in device memory:
// kStaticScratchBytes (8 MiB) on every GPU the entry point is first called
// on, held until the process exits.
//
// The array's host-side name is only a stand-in, not a device address, so
// the address is looked up with cudaGetSymbolAddress once per device (on the
// first call made with that device current) and passed to the kernels.
// With CUDA's lazy module loading (the default) that first lookup is also
// when the driver loads this file's module and places the array in device
// memory, so a caller whose memory pool takes the rest of the device later
// makes one call first -- a call with batch 0 does only this.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "pkc.h"
#include "pkc_internal.h"

namespace pkc {
namespace {

constexpr size_t kStaticScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxDevices = 128;

__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of the scratch array on the current device.
int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "paged_decode_state_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(PKC_ERR_UNSUPPORTED, "paged_decode_state_noalloc: device index %d too large", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return cuda_error(e, "paged_decode_state_noalloc: cudaGetSymbolAddress");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKC_OK;
}

}  // namespace
}  // namespace pkc

using namespace pkc;

extern "C" int pkc_paged_decode_state_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table, int block_table_stride,
    const int32_t* cache_seqlens, int batch, int num_qo_heads, int num_kv_heads, int head_dim, int page_size,
    int64_t num_pages, float sm_scale, const int32_t* plan_host, void* o, float* lse, int32_t* device_status,
    int dtype, void* stream) {
  if (batch < 0) return set_error(PKC_ERR_INVALID_ARG, "batch must be >= 0 (got %d)", batch);
  if (head_dim != PKC_HEAD_DIM)
    return set_error(PKC_ERR_UNSUPPORTED, "head_dim %d is not supported (only 128)", head_dim);
  if (num_kv_heads <= 0 || num_qo_heads <= 0 || num_qo_heads % num_kv_heads != 0)
    return set_error(PKC_ERR_INVALID_ARG, "num_qo_heads must be a positive multiple of num_kv_heads");
  const int g = num_qo_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8)
    return set_error(PKC_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", g);
  if (dtype != PKC_F16 && dtype != PKC_BF16)
    return set_error(PKC_ERR_INVALID_ARG, "dtype must be PKC_F16 or PKC_BF16 (got %d)", dtype);
  if (page_size < 1 || block_table_stride < 1 || num_pages < 0)
    return set_error(PKC_ERR_INVALID_ARG, "page_size and block_table_stride must be >= 1, num_pages >= 0");
  int num_ctas = 0;
  size_t plan_bytes = 0;
  if (plan_host) {
    if (plan_host[PKC_PLAN_MAGIC] != PKC_PLAN_MAGIC_VALUE) return set_error(PKC_ERR_PLAN, "plan: bad magic word");
    if (plan_host[PKC_PLAN_N_REQ] != batch || plan_host[PKC_PLAN_TILE_Q] != 1 ||
        plan_host[PKC_PLAN_N_UNITS] != batch || plan_host[PKC_PLAN_NUM_CTAS] < 1)
      return set_error(PKC_ERR_PLAN, "plan does not describe %d single-query decode requests", batch);
    num_ctas = plan_host[PKC_PLAN_NUM_CTAS];
    plan_bytes = 4 * (size_t)plan_host[PKC_PLAN_TOTAL_WORDS];
  }
  // Scratch layout: status word | plan | partial O [2*num_ctas, Hq, D] |
  // partial LSE [2*num_ctas, Hq], each 256-byte aligned.
  const size_t rows = (size_t)2 * num_ctas * num_qo_heads;
  const size_t off_plan = PKC_STATUS_BYTES;
  const size_t off_po = off_plan + al256(plan_bytes);
  const size_t off_pl = off_po + al256(4 * rows * PKC_HEAD_DIM);
  const size_t need = off_pl + al256(4 * rows);
  if (need > kStaticScratchBytes)
    return set_error(PKC_ERR_WORKSPACE,
                     "paged_decode_state_noalloc: needs %zu bytes of scratch for %d CTAs x %d query heads, "
                     "but the built-in scratch holds %zu bytes (use fewer plan CTAs, or "
                     "pkc_paged_decode_state with a caller workspace)",
                     need, num_ctas, num_qo_heads, kStaticScratchBytes);
  // The array is resolved (and, under lazy module loading, placed in device
  // memory) before anything else, so that a batch-0 call pins it.
  void* base = nullptr;
  if (int rc = scratch_address(&base)) return rc;
  if (batch == 0) return PKC_OK;
  if (!q || !k_cache || !v_cache || !block_table || !cache_seqlens || !o || !lse)
    return set_error(PKC_ERR_INVALID_ARG, "paged_decode_state_noalloc: NULL pointer");
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
        reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(o)) & 15) != 0)
    return set_error(PKC_ERR_INVALID_ARG, "paged_decode_state_noalloc: q, caches and o must be 16-byte aligned");

  uint8_t* s = static_cast<uint8_t*>(base);
  cudaStream_t st = (cudaStream_t)stream;
  // The array keeps the previous call's contents: the status word must
  // start at zero; the plan is copied in; every partial slot is written by
  // the decode kernel before the contraction reads it.
  cudaError_t e = cudaMemsetAsync(s, 0, PKC_STATUS_BYTES, st);
  if (e == cudaSuccess && plan_host)
    e = cudaMemcpyAsync(s + off_plan, plan_host, plan_bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_error(e, "paged_decode_state_noalloc: scratch set-up");

  DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.q = q; dp.k_cache = k_cache; dp.v_cache = v_cache;
  dp.block_table = block_table; dp.cache_seqlens = cache_seqlens;
  dp.bt_stride = block_table_stride; dp.num_pages = num_pages;
  dp.batch = batch; dp.hq = num_qo_heads; dp.hkv = num_kv_heads; dp.page_size = page_size;
  dp.scale_log2 = sm_scale * 1.4426950408889634f;
  dp.v_scale = 1.f;
  dp.plan = plan_host ? reinterpret_cast<const int32_t*>(s + off_plan) : nullptr;
  dp.plan_words = plan_host ? plan_host[PKC_PLAN_TOTAL_WORDS] : 0;
  dp.o_direct = o; dp.lse_direct = lse; dp.direct_f32 = 0;
  dp.part_o = reinterpret_cast<float*>(s + off_po);
  dp.part_lse = reinterpret_cast<float*>(s + off_pl);
  dp.status = reinterpret_cast<int32_t*>(s);
  int le = launch_paged_decode(dp, plan_host ? num_ctas : batch, dtype, dtype, stream);
  if (le) return cuda_error(le, "paged_decode_state_noalloc: decode launch");
  if (plan_host) {
    ContractParams cp;
    std::memset(&cp, 0, sizeof(cp));
    cp.batch = batch; cp.hq = num_qo_heads; cp.mode = kContractPlanUnits; cp.plan = dp.plan;
    cp.plan_words = plan_host[PKC_PLAN_TOTAL_WORDS];
    cp.off_unit_list = plan_host[PKC_PLAN_OFF_UNIT_LIST];
    cp.off_unit_req = plan_host[PKC_PLAN_OFF_UNIT_REQ];
    cp.off_unit_n_chunks = plan_host[PKC_PLAN_OFF_UNIT_N_CHUNKS];
    cp.off_unit_partial_begin = plan_host[PKC_PLAN_OFF_UNIT_PARTIAL_BEGIN];
    cp.part_o = dp.part_o; cp.part_lse = dp.part_lse;
    cp.o = o; cp.lse = lse; cp.out_dtype = dtype; cp.status = dp.status;
    le = launch_contract(cp, batch, stream);
    if (le) return cuda_error(le, "paged_decode_state_noalloc: contraction launch");
  }
  if (device_status) {
    e = cudaMemcpyAsync(device_status, s, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return cuda_error(e, "paged_decode_state_noalloc: status copy");
  }
  return PKC_OK;
}
