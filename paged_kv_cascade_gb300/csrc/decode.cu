// Single-query paged decode state and the contraction of partial states.
//
// Decode (blog "Cascade Inference", algorithm step 2; Hugging Face "Paged
// attention", decoding path): one query per request attends to its cached
// tokens, found through the block table.  There is no KV reuse across
// queries of different requests, so the kernel is bound by HBM bandwidth
// and runs on the CUDA cores (a query tile of one row is below the tensor
// cores' minimum M; MLSys'25 notes, A3 "micro-kernels of different tile
// sizes").  The query heads of one KV head are fused into one thread block
// so every K/V row is loaded once for the whole group (MLSys'25 notes,
// appendix A).  Long sequences are split into KV chunks by the host plan;
// each chunk yields a partial state, merged afterwards by the contraction
// kernel (MLSys'25 notes, A3: "the final output is the contraction of the
// partial outputs"; appendix D: unsplit requests write the output
// directly).
//
// Thread layout: 4 warps per block; a half-warp (16 lanes x 8 dims) holds
// one 128-dim K or V row, so a warp consumes two tokens per step.  Loads
// are 16-byte vectors straight from HBM, U steps in flight per warp.  Each
// half-warp keeps its own online-softmax state (running max m, running sum
// l, accumulator); the halves and the warps are merged at the end with the
// same (+) operator.
#include <cuda_runtime.h>

#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

constexpr int D = PKC_HEAD_DIM;
constexpr int kWarps = 4;

struct WorkItem {
  int req, kv_begin, kv_end, slot;
};

template <typename T, int G>
__global__ void __launch_bounds__(128) paged_decode_kernel(const DecodeParams p) {
  constexpr int U = G >= 4 ? 4 : 8;  // steps (token pairs) in flight per warp
  __shared__ float s_m[kWarps][G], s_l[kWarps][G];
  __shared__ __align__(16) float s_acc[kWarps][G][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int half = lane >> 4, sub = lane & 15;
  const int kvh = blockIdx.y;
  const int cta = blockIdx.x;
  const T* __restrict__ kc = static_cast<const T*>(p.k_cache);
  const T* __restrict__ vc = static_cast<const T*>(p.v_cache);
  const int ps = p.page_size;
  const int ps_shift = (ps & (ps - 1)) == 0 ? __ffs(ps) - 1 : -1;

  int w_begin = 0, w_end = 1;
  const int32_t* pl = p.plan;
  if (pl) {
    w_begin = pl[pl[PKC_PLAN_OFF_CTA_INDPTR] + cta];
    w_end = pl[pl[PKC_PLAN_OFF_CTA_INDPTR] + cta + 1];
  }
  for (int wi = w_begin; wi < w_end; ++wi) {
    WorkItem it;
    if (pl) {
      const int w = pl[pl[PKC_PLAN_OFF_CTA_WORK] + wi];
      const int unit = pl[pl[PKC_PLAN_OFF_WORK_UNIT] + w];
      it.req = pl[pl[PKC_PLAN_OFF_UNIT_REQ] + unit];
      it.kv_begin = pl[pl[PKC_PLAN_OFF_WORK_KV_BEGIN] + w];
      it.kv_end = pl[pl[PKC_PLAN_OFF_WORK_KV_END] + w];
      it.slot = pl[pl[PKC_PLAN_OFF_WORK_PARTIAL] + w];
      const int len = p.cache_seqlens[it.req];
      if (pl[pl[PKC_PLAN_OFF_UNIT_KV_LEN] + unit] != len) {
        if (threadIdx.x == 0) report(p.status, PKC_ERR_PLAN);
        it.kv_end = min(it.kv_end, len);
        it.kv_begin = min(it.kv_begin, it.kv_end);
      }
    } else {
      it.req = cta;
      it.kv_begin = 0;
      it.kv_end = max(p.cache_seqlens[cta], 0);
      it.slot = -1;
    }
    if ((int64_t)it.kv_end > p.bt_stride * ps) {  // more tokens than table entries
      if (threadIdx.x == 0) report(p.status, PKC_ERR_BLOCK_TABLE);
      it.kv_end = (int)(p.bt_stride * ps);
      it.kv_begin = min(it.kv_begin, it.kv_end);
    }

    // Query rows of the G heads of this KV head, pre-scaled to log2 units.
    float q[G][8];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const T* qp = static_cast<const T*>(p.q) + ((int64_t)it.req * p.hq + kvh * G + gi) * D + sub * 8;
      uint4 u = *reinterpret_cast<const uint4*>(qp);
      float2 a = Elem<T>::to_f2(u.x), b = Elem<T>::to_f2(u.y), c = Elem<T>::to_f2(u.z), d = Elem<T>::to_f2(u.w);
      q[gi][0] = a.x * p.scale_log2; q[gi][1] = a.y * p.scale_log2;
      q[gi][2] = b.x * p.scale_log2; q[gi][3] = b.y * p.scale_log2;
      q[gi][4] = c.x * p.scale_log2; q[gi][5] = c.y * p.scale_log2;
      q[gi][6] = d.x * p.scale_log2; q[gi][7] = d.y * p.scale_log2;
    }

    float m[G], l[G], acc[G][8];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      m[gi] = neg_inf();
      l[gi] = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[gi][k] = 0.f;
    }

    // Contiguous token range of this warp (whole token pairs).
    const int n = it.kv_end - it.kv_begin;
    const int pairs = (n + 1) >> 1;
    const int ppw = (pairs + kWarps - 1) / kWarps;
    const int wb = it.kv_begin + 2 * warp * ppw;
    const int we = min(it.kv_end, wb + 2 * ppw);
    const int nsteps = we > wb ? (we - wb + 1) >> 1 : 0;
    const int32_t* bt_row = p.block_table + (int64_t)it.req * p.bt_stride;

    for (int s0 = 0; s0 < nsteps; s0 += U) {
      uint4 kr[U], vr[U];
      bool valid[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = wb + 2 * (s0 + u) + half;
        bool ok = t < we;
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
        if (ok) {
          int pi, slot;
          if (ps_shift >= 0) { pi = t >> ps_shift; slot = t & (ps - 1); }
          else { pi = t / ps; slot = t - pi * ps; }
          const int32_t page = bt_row[pi];
          if (page < 0 || page >= p.num_pages) {
            report(p.status, PKC_ERR_BLOCK_TABLE);
            ok = false;
          } else {
            const int64_t off = (((int64_t)page * ps + slot) * p.hkv + kvh) * D + sub * 8;
            kr[u] = ldg_stream(kc + off);
            vr[u] = ldg_stream(vc + off);
          }
        }
        valid[u] = ok;
      }
      // Scores s = q . k (log2 units), reduced over the 16 lanes of a half.
      float sc[U][G];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float2 k0 = Elem<T>::to_f2(kr[u].x), k1 = Elem<T>::to_f2(kr[u].y);
        float2 k2 = Elem<T>::to_f2(kr[u].z), k3 = Elem<T>::to_f2(kr[u].w);
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          float d = q[gi][0] * k0.x;
          d = fmaf(q[gi][1], k0.y, d); d = fmaf(q[gi][2], k1.x, d); d = fmaf(q[gi][3], k1.y, d);
          d = fmaf(q[gi][4], k2.x, d); d = fmaf(q[gi][5], k2.y, d); d = fmaf(q[gi][6], k3.x, d);
          d = fmaf(q[gi][7], k3.y, d);
          sc[u][gi] = d;
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          float d = sc[u][gi];
          d += __shfl_xor_sync(0xffffffffu, d, 8);
          d += __shfl_xor_sync(0xffffffffu, d, 4);
          d += __shfl_xor_sync(0xffffffffu, d, 2);
          d += __shfl_xor_sync(0xffffffffu, d, 1);
          sc[u][gi] = valid[u] ? d : neg_inf();
        }
      // Online softmax update, once per U steps.
      float pr[U][G];
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        float mx = m[gi];
#pragma unroll
        for (int u = 0; u < U; ++u) mx = fmaxf(mx, sc[u][gi]);
        const float corr = mx == neg_inf() ? 1.f : ex2(m[gi] - mx);
        m[gi] = mx;
        l[gi] *= corr;
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[gi][k] *= corr;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          pr[u][gi] = valid[u] ? ex2(sc[u][gi] - mx) : 0.f;
          l[gi] += pr[u][gi];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float2 v0 = Elem<T>::to_f2(vr[u].x), v1 = Elem<T>::to_f2(vr[u].y);
        float2 v2 = Elem<T>::to_f2(vr[u].z), v3 = Elem<T>::to_f2(vr[u].w);
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
          const float pw = pr[u][gi];
          acc[gi][0] = fmaf(pw, v0.x, acc[gi][0]); acc[gi][1] = fmaf(pw, v0.y, acc[gi][1]);
          acc[gi][2] = fmaf(pw, v1.x, acc[gi][2]); acc[gi][3] = fmaf(pw, v1.y, acc[gi][3]);
          acc[gi][4] = fmaf(pw, v2.x, acc[gi][4]); acc[gi][5] = fmaf(pw, v2.y, acc[gi][5]);
          acc[gi][6] = fmaf(pw, v3.x, acc[gi][6]); acc[gi][7] = fmaf(pw, v3.y, acc[gi][7]);
        }
      }
    }

    // Merge the two halves of the warp ((+) with log2-domain maxima).
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[gi], 16);
      const float lo = __shfl_xor_sync(0xffffffffu, l[gi], 16);
      const float mm = fmaxf(m[gi], mo);
      const float a = mm == neg_inf() ? 0.f : ex2(m[gi] - mm);
      const float b = mm == neg_inf() ? 0.f : ex2(mo - mm);
      l[gi] = l[gi] * a + lo * b;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float ao = __shfl_xor_sync(0xffffffffu, acc[gi][k], 16);
        acc[gi][k] = acc[gi][k] * a + ao * b;
      }
      m[gi] = mm;
    }
    if (half == 0) {
#pragma unroll
      for (int gi = 0; gi < G; ++gi) {
        if (sub == 0) { s_m[warp][gi] = m[gi]; s_l[warp][gi] = l[gi]; }
        *reinterpret_cast<float4*>(&s_acc[warp][gi][sub * 8]) = make_float4(acc[gi][0], acc[gi][1], acc[gi][2], acc[gi][3]);
        *reinterpret_cast<float4*>(&s_acc[warp][gi][sub * 8 + 4]) = make_float4(acc[gi][4], acc[gi][5], acc[gi][6], acc[gi][7]);
      }
    }
    __syncthreads();
    // Merge the warps and write the state of this chunk.
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
      const int gi = idx / D, d = idx % D;
      float mm = neg_inf();
#pragma unroll
      for (int w = 0; w < kWarps; ++w) mm = fmaxf(mm, s_m[w][gi]);
      float den = 0.f, num = 0.f;
      if (mm != neg_inf()) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float e = ex2(s_m[w][gi] - mm);
          den += s_l[w][gi] * e;
          num += s_acc[w][gi][d] * e;
        }
      }
      const float o = den > 0.f ? num / den : 0.f;
      const float lse = den > 0.f ? (mm + lg2(den)) * kLn2 : neg_inf();
      const int h = kvh * G + gi;
      if (it.slot >= 0) {
        p.part_o[((int64_t)it.slot * p.hq + h) * D + d] = o;
        if (d == 0) p.part_lse[(int64_t)it.slot * p.hq + h] = lse;
      } else {
        const int64_t row = (int64_t)it.req * p.hq + h;
        if (p.direct_f32) static_cast<float*>(p.o_direct)[row * D + d] = o;
        else static_cast<T*>(p.o_direct)[row * D + d] = Elem<T>::from_f(o);
        if (d == 0) p.lse_direct[row] = lse;
      }
    }
    __syncthreads();
  }
}

// One warp per (row, head): (+) over every state that belongs to the row,
// lane i owning dims 4i..4i+3.
__global__ void __launch_bounds__(256) contract_kernel(const ContractParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t row_idx = gw / p.hq;
  const int h = (int)(gw % p.hq);
  const int32_t* pl = p.plan;
  int64_t n_rows = p.batch;
  if (p.mode == kContractPlanUnits) n_rows = pl[PKC_PLAN_N_SPLIT] + pl[PKC_PLAN_N_EMPTY];
  if (row_idx >= n_rows) return;
  int req = (int)row_idx, unit = (int)row_idx;
  if (p.mode == kContractPlanUnits) {
    unit = pl[pl[PKC_PLAN_OFF_UNIT_LIST] + row_idx];
    req = pl[pl[PKC_PLAN_OFF_UNIT_REQ] + unit];
  }
  // Sources: prefix splits of the request's group, then the suffix.
  int group = -1;
  if (p.prefix_o) {
    for (int j = 0; j < p.n_prefix; ++j)
      if (p.req_indptr[j] <= req && req < p.req_indptr[j + 1]) { group = j; break; }
  }
  int n_pref = group >= 0 ? p.prefix_splits : 0;
  int suf_kind = 0, suf_begin = 0, suf_n = 0;  // 1: direct state, 2: partial slots
  if (pl) {
    const int nch = pl[pl[PKC_PLAN_OFF_UNIT_N_CHUNKS] + unit];
    if (nch >= 2) { suf_kind = 2; suf_begin = pl[pl[PKC_PLAN_OFF_UNIT_PARTIAL_BEGIN] + unit]; suf_n = nch; }
    else if (nch == 1 && p.suffix_o) { suf_kind = 1; suf_n = 1; }
  } else if (p.suffix_o) {
    suf_kind = 1; suf_n = 1;
  }
  const int n_src = n_pref + suf_n;
  auto src_lse = [&](int i) -> float {
    if (i < n_pref) return p.prefix_lse[i * p.prefix_stride_lse + (int64_t)req * p.hq + h];
    if (suf_kind == 1) return p.suffix_lse[(int64_t)req * p.hq + h];
    return p.part_lse[(int64_t)(suf_begin + i - n_pref) * p.hq + h];
  };
  auto src_o = [&](int i) -> const float* {
    if (i < n_pref) return p.prefix_o + i * p.prefix_stride_o + ((int64_t)req * p.hq + h) * D;
    if (suf_kind == 1) return p.suffix_o + ((int64_t)req * p.hq + h) * D;
    return p.part_o + ((int64_t)(suf_begin + i - n_pref) * p.hq + h) * D;
  };
  float m = neg_inf();
  for (int i = 0; i < n_src; ++i) m = fmaxf(m, src_lse(i));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  if (m != neg_inf()) {
    for (int i = 0; i < n_src; ++i) {
      const float w = ex2((src_lse(i) - m) * kLog2e);
      const float4 x = *reinterpret_cast<const float4*>(src_o(i) + lane * 4);
      den += w;
      acc.x = fmaf(w, x.x, acc.x); acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z); acc.w = fmaf(w, x.w, acc.w);
    }
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

template <typename T>
int launch_decode_t(const DecodeParams& p, int grid_x, cudaStream_t st) {
  const dim3 grid(grid_x, p.hkv);
  switch (p.hq / p.hkv) {
    case 1: paged_decode_kernel<T, 1><<<grid, 128, 0, st>>>(p); break;
    case 2: paged_decode_kernel<T, 2><<<grid, 128, 0, st>>>(p); break;
    case 4: paged_decode_kernel<T, 4><<<grid, 128, 0, st>>>(p); break;
    case 8: paged_decode_kernel<T, 8><<<grid, 128, 0, st>>>(p); break;
    default: return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

}  // namespace

int launch_paged_decode(const DecodeParams& p, int grid_x, int dtype, void* stream) {
  if (grid_x <= 0) return 0;
  cudaStream_t st = (cudaStream_t)stream;
  return dtype == PKC_F16 ? launch_decode_t<__half>(p, grid_x, st)
                          : launch_decode_t<__nv_bfloat16>(p, grid_x, st);
}

int launch_contract(const ContractParams& p, int n_rows, void* stream) {
  const int64_t warps = (int64_t)n_rows * p.hq;
  if (warps <= 0) return 0;
  const int blocks = (int)((warps + 7) / 8);
  contract_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace pkc
