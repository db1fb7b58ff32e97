// Multi-query prefix state on the 5th-generation tensor cores.
//
// Blog "Cascade Inference", algorithm step 1 and section "Multi-query vs
// single-query kernels": every request in a group shares the same prefix
// KV, so one thread block loads each KV tile into shared memory once and
// computes all the group's queries against it on the tensor cores.  The
// query rows of a tile are (request, query head) pairs of one KV head, GQA
// heads fused with the request dimension (MLSys'25 notes, appendix A), 128
// rows per tile.  The prefix KV is split into `splits` chunks per group so
// the grid fills the SMs; each (row tile, chunk) writes a partial state
// that the contraction kernel merges with (+).
//
// Per 128-token KV tile j (FlashAttention-style online softmax, blog
// section "Recursive Attention"):
//   S_j = Q K_j^T            tcgen05.mma, M=N=128, K=128, fp32 in TMEM
//   P_j = exp2(S_j*c - m_j)  softmax warps: TMEM -> registers -> smem (16b)
//   O_j = P_j V_j            tcgen05.mma, P K-major, V MN-major, into TMEM
//   O  <- O * exp2(m_{j-1} - m_j) + O_j   in registers of the row's thread
// Roles: warp 0 issues TMA loads (Q once, K/V into a 3-stage ring), warp 1
// allocates TMEM and issues MMAs, warps 2..5 own one query row per thread.
// TMEM: S double buffer (2 x 128 columns) + O double buffer (2 x 128).
// P_j overwrites K_j's shared memory once S_j is complete.  All waits are
// bounded (2 s) and set PKC_ERR_TIMEOUT when they run out.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

constexpr int kRows = 128;       // query rows per tile (MMA M)
constexpr int kKvTile = 128;     // tokens per KV tile (MMA N of S, K of PV)
constexpr int kStages = 3;
constexpr int kSubTile = 16384;  // 128 rows x 128 bytes (64 elements)
constexpr int kQBytes = 2 * kSubTile;
constexpr int kStageBytes = 4 * kSubTile;  // K (2 sub-tiles) + V (2 sub-tiles)
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

struct __align__(8) Barriers {
  uint64_t q_full;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2], o_full[2], o_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kSmemBytes = kQBytes + kStages * kStageBytes + 256 + 1024;

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
    prefix_state_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefixParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_q = smem_u32(smem);
  const uint32_t s_stage0 = s_q + kQBytes;
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kQBytes + kStages * kStageBytes);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.g;
  const int kvh = blockIdx.y;
  const int tile = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
  int grp = 0;
  while (grp + 1 < p.n_prefix && p.tile_indptr[grp + 1] <= tile) ++grp;
  const int mt = tile - p.tile_indptr[grp];
  const int req_hi = p.req_indptr[grp + 1];
  const int b0 = p.req_indptr[grp] + mt * (kRows / G);
  const int kv_lo = p.kv_indptr[grp] + split * p.chunk[grp];
  const int kv_hi = min(p.kv_indptr[grp + 1], kv_lo + p.chunk[grp]);
  const int n_tiles = kv_hi > kv_lo ? (kv_hi - kv_lo + kKvTile - 1) / kKvTile : 0;

  auto bar = [&](uint64_t& b) { return smem_u32(&b); };
  if (threadIdx.x == 0) {
    mbar_init(bar(bars->q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(bars->kv_full[s]), 1);
      mbar_init(bar(bars->kv_empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(bars->s_full[b]), 1);
      mbar_init(bar(bars->s_free[b]), 128);
      mbar_init(bar(bars->p_full[b]), 128);
      mbar_init(bar(bars->o_full[b]), 1);
      mbar_init(bar(bars->o_free[b]), 128);
    }
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

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && n_tiles > 0) {
      const uint64_t pol = l2_policy_evict_first();
      const uint64_t pol_q = l2_policy_evict_last();
      mbar_arrive_expect_tx(bar(bars->q_full), kQBytes);
      tma_load_3d(s_q, &tm_q, bar(bars->q_full), 0, kvh * G, b0, pol_q);
      tma_load_3d(s_q + kSubTile, &tm_q, bar(bars->q_full), 64, kvh * G, b0, pol_q);
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(bar(bars->kv_empty[s]), ((j / kStages) & 1) ^ 1, abort, p.status)) break;
        const uint32_t st = s_stage0 + s * kStageBytes;
        const int t0 = kv_lo + j * kKvTile;
        mbar_arrive_expect_tx(bar(bars->kv_full[s]), kStageBytes);
        tma_load_3d(st, &tm_k, bar(bars->kv_full[s]), 0, kvh, t0, pol);
        tma_load_3d(st + kSubTile, &tm_k, bar(bars->kv_full[s]), 64, kvh, t0, pol);
        tma_load_3d(st + 2 * kSubTile, &tm_v, bar(bars->kv_full[s]), 0, kvh, t0, pol);
        tma_load_3d(st + 3 * kSubTile, &tm_v, bar(bars->kv_full[s]), 64, kvh, t0, pol);
        issued = j + 1;
      }
      if (*abort) {
        // Let the copies already issued land before the block exits.
        volatile int no_abort = 0;
        mbar_wait(bar(bars->q_full), 0, &no_abort, p.status);
        for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
          mbar_wait(bar(bars->kv_full[j % kStages]), (j / kStages) & 1, &no_abort, p.status);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value ? 1 : 0;
      constexpr uint32_t idesc_qk = idesc_f16(128, 128, kBf16, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16(128, 128, kBf16, 0, 1);
      bool ok = mbar_wait(bar(bars->q_full), 0, abort, p.status);
      tc_fence_after();
      for (int j = 0; ok && j <= n_tiles; ++j) {
        if (j < n_tiles) {
          const int s = j % kStages, b = j & 1;
          ok = mbar_wait(bar(bars->kv_full[s]), (j / kStages) & 1, abort, p.status) &&
               mbar_wait(bar(bars->s_free[b]), ((j >> 1) & 1) ^ 1, abort, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kb = s_stage0 + s * kStageBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kSubTile + (kk & 3) * 32;
            tc_mma_f16(tmem + b * 128, smem_desc_sw128(s_q + off, 16, 1024),
                       smem_desc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0);
          }
          tc_commit(bar(bars->s_full[b]));
        }
        if (j >= 1) {
          const int jp = j - 1, sp = jp % kStages, bp = jp & 1;
          ok = mbar_wait(bar(bars->p_full[bp]), (jp >> 1) & 1, abort, p.status) &&
               mbar_wait(bar(bars->o_free[bp]), ((jp >> 1) & 1) ^ 1, abort, p.status);
          if (!ok) break;
          tc_fence_after();
          const uint32_t pb = s_stage0 + sp * kStageBytes;  // P overwrote K
          const uint32_t vb = pb + 2 * kSubTile;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a_off = (kk >> 2) * kSubTile + (kk & 3) * 32;
            tc_mma_f16(tmem + 256 + bp * 128, smem_desc_sw128(pb + a_off, 16, 1024),
                       smem_desc_sw128(vb + kk * 2048, kSubTile, 1024), idesc_pv, kk > 0);
          }
          tc_commit(bar(bars->o_full[bp]));
          tc_commit(bar(bars->kv_empty[sp]));
        }
      }
      // Drain: every MMA issued above completes before TMEM is released.
      tc_commit(bar(bars->drain));
      volatile int no_abort = 0;
      mbar_wait(bar(bars->drain), 0, &no_abort, p.status);
    }
  } else {
    // ---------------- softmax / correction: one query row per thread ----------------
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int row = quad * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(quad * 32) << 16);
    float o_acc[128];
#pragma unroll
    for (int i = 0; i < 128; ++i) o_acc[i] = 0.f;
    float m_run = neg_inf(), l_run = 0.f, corr_prev = 1.f;
    bool ok = true;
    auto fold = [&](int jp) {
      const int bp = jp & 1;
      if (!mbar_wait(bar(bars->o_full[bp]), (jp >> 1) & 1, abort, p.status)) { ok = false; return; }
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_addr + 256 + bp * 128 + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) o_acc[c * 32 + i] = fmaf(o_acc[c * 32 + i], corr_prev, __uint_as_float(r[i]));
      }
      tc_fence_before();
      mbar_arrive(bar(bars->o_free[bp]));
    };
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int b = j & 1, s = j % kStages;
      if (!mbar_wait(bar(bars->s_full[b]), (j >> 1) & 1, abort, p.status)) { ok = false; break; }
      tc_fence_after();
      const int valid = min(kKvTile, kv_hi - (kv_lo + j * kKvTile));
      float mx = neg_inf();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_addr + b * 128 + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c * 32 + i < valid) mx = fmaxf(mx, __uint_as_float(r[i]));
      }
      const float m_new = fmaxf(m_run, mx * p.scale_log2);
      const float corr = m_new == neg_inf() ? 1.f : ex2(m_run - m_new);
      l_run *= corr;
      const uint32_t pbase = s_stage0 + s * kStageBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_addr + b * 128 + c * 32, r);
        tmem_ld_wait();
        float pv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          pv[i] = c * 32 + i < valid ? ex2(fmaf(__uint_as_float(r[i]), p.scale_log2, -m_new)) : 0.f;
          l_run += pv[i];
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t chunk = (uint32_t)((c & 1) * 4 + k);
          const uint32_t addr = pbase + (c >> 1) * kSubTile + row * 128 + ((chunk ^ (row & 7)) << 4);
          const uint32_t w0 = Elem<T>::from_f2(pv[8 * k + 0], pv[8 * k + 1]);
          const uint32_t w1 = Elem<T>::from_f2(pv[8 * k + 2], pv[8 * k + 3]);
          const uint32_t w2 = Elem<T>::from_f2(pv[8 * k + 4], pv[8 * k + 5]);
          const uint32_t w3 = Elem<T>::from_f2(pv[8 * k + 6], pv[8 * k + 7]);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                       : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar(bars->p_full[b]));
      mbar_arrive(bar(bars->s_free[b]));
      m_run = m_new;
      if (j >= 1) fold(j - 1);
      corr_prev = corr;
    }
    if (ok && n_tiles > 0) fold(n_tiles - 1);

    // Epilogue: rows that belong to this group write their state.
    const int rb = b0 + row / G;
    if (rb < req_hi && rb < p.batch) {
      const int h = kvh * G + row % G;
      const int64_t r = (int64_t)rb * p.hq + h;
      float* out = p.out_o + split * p.split_stride_o + r * PKC_HEAD_DIM;
      const bool has = ok && l_run > 0.f;
      const float inv = has ? 1.f / l_run : 0.f;
#pragma unroll
      for (int i = 0; i < 128; i += 4)
        *reinterpret_cast<float4*>(out + i) =
            make_float4(o_acc[i] * inv, o_acc[i + 1] * inv, o_acc[i + 2] * inv, o_acc[i + 3] * inv);
      p.out_lse[split * p.split_stride_lse + r] = has ? (m_run + lg2(l_run)) * kLn2 : neg_inf();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D tiled map over a row-major [d2][d1][d0] tensor of 16-bit elements
// with a {64, box1, box2} box and 128-byte swizzle (rows of 128 bytes).
bool make_map(CUtensorMap* m, const void* base, int dtype, uint64_t d0, uint64_t d1, uint64_t d2,
              uint32_t box1, uint32_t box2) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  const cuuint32_t box[3] = {64, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType t =
      dtype == PKC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return enc(m, t, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
int launch_t(const PrefixParams& p, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
             int n_tiles, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(prefix_state_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return (int)attr_err;
  const dim3 grid(n_tiles * p.splits, p.hkv);
  prefix_state_kernel<T><<<grid, kThreads, kSmemBytes, st>>>(q, k, v, p);
  return (int)cudaGetLastError();
}

}  // namespace

int launch_prefix(const PrefixParams& p, const void* q, const void* k_prefix, const void* v_prefix,
                  int64_t prefix_tokens, int n_tiles, int dtype, void* stream) {
  if (n_tiles <= 0) return 0;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, dtype, PKC_HEAD_DIM, p.hq, p.batch, p.g, kRows / p.g) ||
      !make_map(&mk, k_prefix, dtype, PKC_HEAD_DIM, p.hkv, prefix_tokens, 1, kKvTile) ||
      !make_map(&mv, v_prefix, dtype, PKC_HEAD_DIM, p.hkv, prefix_tokens, 1, kKvTile))
    return -1;
  cudaStream_t st = (cudaStream_t)stream;
  return dtype == PKC_BF16 ? launch_t<__nv_bfloat16>(p, mq, mk, mv, n_tiles, st)
                           : launch_t<__half>(p, mq, mk, mv, n_tiles, st);
}

}  // namespace pkc
