// CUDA-core paged decode (the kernel is in decode_simt.cuh; its
// instantiations with the fused contraction are compiled in
// decode_fused.cu), the standalone contraction kernel, and the dispatch
// between the decode kernels.
#include <atomic>

#include "decode_simt.cuh"

namespace pkc {
namespace {

// One warp per R query heads of one KV head of a request (R divides the
// query heads per KV head): (+) over every state that belongs to each of its
// rows (contract_rows, the rows in lockstep so that all their loads are in
// flight together), after the stages that wrote them.  More rows per warp
// need more registers, so fewer blocks per SM (kMinBlocks).
template <int R, int kMinBlocks>
__global__ void __launch_bounds__(256, kMinBlocks) contract_kernel(const __grid_constant__ ContractParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int per_row = p.hq / R;  // warps per request
  const int64_t row_idx = gw / per_row;
  const int h0 = (int)(gw % per_row) * R;
  const int32_t* pl = p.plan;
  if (pl && !device_plan_ok(pl, p.plan_words, p.batch)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report(p.status, PKC_ERR_PLAN);
    return;
  }
  // The list length changes with the lengths every step: read it from the
  // device plan (the array offsets depend only on batch and CTA count).
  const int64_t n_rows =
      p.mode == kContractPlanUnits ? (int64_t)pl[PKC_PLAN_N_SPLIT] + pl[PKC_PLAN_N_EMPTY] : p.batch;
  if (row_idx >= n_rows) return;
  int req = (int)row_idx, unit = (int)row_idx;
  if (p.mode == kContractPlanUnits) {
    unit = pl[p.off_unit_list + row_idx];
    req = pl[p.off_unit_req + unit];
  }
  contract_rows<R, ContractParams, true>(p, req, unit, h0, R, lane);
}

}  // namespace

int launch_paged_decode_simt(const DecodeParams& p, int grid_x, int dtype, void* stream) {
  if (grid_x <= 0) return 0;
  // KV heads per block: the largest of 8, 4, 2, 1 that divides Hkv, or the
  // caller's choice (p.hg, which must divide Hkv).
  const int hg = p.hg > 0 ? p.hg : p.hkv % 8 == 0 ? 8 : p.hkv % 4 == 0 ? 4 : p.hkv % 2 == 0 ? 2 : 1;
  const int sl = p.page_size < kMaxSliceRows ? p.page_size : kMaxSliceRows;
  // 4-D view [num_pages][page_size][Hkv][128]; one tile = sl slots x hg heads of a page.
  const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.hkv, (uint64_t)p.page_size,
                            (uint64_t)(p.num_pages > 0 ? p.num_pages : 1)};
  const uint64_t strides[3] = {(uint64_t)D * 2, (uint64_t)D * 2 * p.hkv, (uint64_t)D * 2 * p.hkv * p.page_size};
  const uint32_t box[4] = {(uint32_t)D, (uint32_t)hg, (uint32_t)sl, 1u};
  alignas(64) CUtensorMap mk, mv;
  alignas(64) PrefixMaps pm;
  if (!encode_tiled_map(&mk, p.k_cache, dtype, 4, dims, strides, box, false) ||
      !encode_tiled_map(&mv, p.v_cache, dtype, 4, dims, strides, box, false))
    return -1;
  if (p.prefix_as_pages && p.prefix_pages > 0 && p.prefix_k && p.prefix_v) {
    // the contiguous prefix tensors [prefix_pages * page_size, Hkv, 128] in the same page view
    const uint64_t pdims[4] = {(uint64_t)D, (uint64_t)p.hkv, (uint64_t)p.page_size,
                               (uint64_t)(p.prefix_pages > 0 ? p.prefix_pages : 1)};
    // ... and as tokens, one box per stage: 128 / hg tokens x hg heads
    const uint64_t tdims[3] = {(uint64_t)D, (uint64_t)p.hkv, (uint64_t)p.prefix_pages * (uint64_t)p.page_size};
    const uint64_t tstrides[2] = {(uint64_t)D * 2, (uint64_t)D * 2 * p.hkv};
    const uint32_t tbox[3] = {(uint32_t)D, (uint32_t)hg, (uint32_t)(kStageRows / hg)};
    if (!encode_tiled_map(&pm.pk, p.prefix_k, dtype, 4, pdims, strides, box, false) ||
        !encode_tiled_map(&pm.pv, p.prefix_v, dtype, 4, pdims, strides, box, false) ||
        !encode_tiled_map(&pm.pk3, p.prefix_k, dtype, 3, tdims, tstrides, tbox, false) ||
        !encode_tiled_map(&pm.pv3, p.prefix_v, dtype, 3, tdims, tstrides, tbox, false))
      return -1;
  } else {
    pm.pk = pm.pk3 = mk;  // not read
    pm.pv = pm.pv3 = mv;
  }
  cudaStream_t st = (cudaStream_t)stream;
  if (p.fuse.enabled) return launch_paged_decode_simt_fused(p, grid_x, dtype, hg, &mk, &mv, &pm, st);
  return launch_simt_mode<false>(p, grid_x, dtype, hg, mk, mv, pm, st);
}

// Kernel choice for a 16-bit cache: 0 = automatic, 1 = CUDA-core kernel,
// 2 = tensor-core kernel (pkc_set_decode_kernel).
static std::atomic<int> g_decode_kernel{0};

int set_decode_kernel(int which) {
  if (which < 0 || which > 2) return -1;
  g_decode_kernel.store(which);
  return 0;
}

// Planned decodes: 1 = blocks take the plan's chunks from a shared queue in
// the plan's longest-first order (default), 0 = each block runs its CTA's
// list of the plan (pkc_set_decode_schedule).
static std::atomic<int> g_decode_dynamic{1};

int decode_schedule_dynamic() { return g_decode_dynamic.load(); }

int set_decode_schedule(int dynamic) {
  if (dynamic != 0 && dynamic != 1) return -1;
  g_decode_dynamic.store(dynamic);
  return 0;
}

// An fp8 cache always takes the tensor-core kernel.  A 16-bit cache takes it
// for grouped heads (G >= 2), where the CUDA-core kernel runs out of issue
// slots before HBM bandwidth, and the CUDA-core kernel for G = 1, unless
// the choice is forced.
int launch_paged_decode(const DecodeParams& p_in, int grid_x, int dtype, int kv_dtype, void* stream) {
  DecodeParams p = p_in;
  // The queue's counters: words 16 and 17 of the status block, which every
  // workspace starts with (zeroed by pkc_workspace_init).
  p.dynamic = p.plan != nullptr && g_decode_dynamic.load() != 0;
  p.sched = p.status + 16;
  const bool mma_ok = mma_decode_heads_per_block(p.hkv, p.page_size) > 0;
  if (kv_dtype == PKC_E4M3) {
    if (dtype != PKC_F16 || !mma_ok) return (int)cudaErrorInvalidValue;
    return launch_paged_decode_mma(p, grid_x, kKvE4M3, stream);
  }
  const int forced = g_decode_kernel.load();
  const bool use_mma = mma_ok && !p.prefix_as_pages && (forced == 2 || (forced == 0 && p.hq / p.hkv >= 2));
  if (use_mma) return launch_paged_decode_mma(p, grid_x, dtype == PKC_BF16 ? kKvBF16 : kKvF16, stream);
  return launch_paged_decode_simt(p, grid_x, dtype, stream);
}

// The contraction follows the suffix decode on the stream (after_decode).
// Launched with programmatic stream serialization (the default), it may
// start once every
// decode block has signalled (griddepcontrol.launch_dependents, at each
// decode block's start): its blocks take the SM room the decode leaves,
// load the plan words (and, unless the decode itself follows the prefix
// kernel as a dependent, the prefix pieces), and wait at griddepcontrol.wait
// for the decode grid to finish before reading the suffix states.  The
// dependency on everything else before the decode on the stream (the plan
// upload, and the prefix grid, which every decode block waits for before it
// exits) stays complete.
static std::atomic<int> g_contract_pdl{1};
int set_contract_pdl(int on) {
  g_contract_pdl.store(on ? 1 : 0);
  return 0;
}

template <int R, int kMinBlocks>
int launch_contract_r(const ContractParams& p, int n_rows, cudaStream_t st, bool programmatic) {
  const int64_t warps = (int64_t)n_rows * (p.hq / R);
  if (warps <= 0) return 0;
  const int blocks = (int)((warps + 7) / 8);
  if (!programmatic) {
    contract_kernel<R, kMinBlocks><<<blocks, 256, 0, st>>>(p);
    return (int)cudaGetLastError();
  }
  return launch_programmatic(contract_kernel<R, kMinBlocks>, dim3(blocks), dim3(256), 0, st, p);
}

int launch_contract(const ContractParams& p, int n_rows, void* stream, bool after_decode) {
  const bool programmatic = after_decode && g_contract_pdl.load();
  cudaStream_t st = (cudaStream_t)stream;
  // The rows in flight per SM, not the loads per warp, set the kernel's
  // time: 4 rows per warp at 2 blocks per SM took longer than 1 row at 4
  // blocks (gqa_cascade_lb contraction 12.8 -> 15.2 us), while 2 rows at 4
  // blocks fit the headline's rows in one wave of resident blocks (step
  // 290.1 -> 288.5 us).  The two rows are query heads of one KV head
  // (G >= 2), which share their prefix pieces; G = 1 keeps one row per warp.
  if (p.g >= 2 && p.hq % 2 == 0) return launch_contract_r<2, 4>(p, n_rows, st, programmatic);
  return launch_contract_r<1, 4>(p, n_rows, st, programmatic);
}

}  // namespace pkc
