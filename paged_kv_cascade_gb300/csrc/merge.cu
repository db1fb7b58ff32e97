// Merge operator kernels: binary and n-ary (+) over attention states
// ("Attention States and Recursive Attention", binary and n-ary merge
// equations).  Pure streaming work: each (token, head) row is read once and
// written once with 16-byte vector accesses; a row's LSE values are read by
// every lane that handles the row, then written by one lane.
#include <cuda_runtime.h>

#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

template <typename T> struct Vec;  // 16 bytes of T <-> 4 or 8 floats
template <> struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const void* p, float* f) {
    uint4 u = ldg_stream(p);
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
  static __device__ __forceinline__ void store(void* p, const float* f) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <typename H> struct Vec16 {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const void* p, float* f) {
    uint4 u = ldg_stream(p);
    float2 a = Elem<H>::to_f2(u.x), b = Elem<H>::to_f2(u.y);
    float2 c = Elem<H>::to_f2(u.z), d = Elem<H>::to_f2(u.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
  static __device__ __forceinline__ void store(void* p, const float* f) {
    uint4 u;
    u.x = Elem<H>::from_f2(f[0], f[1]); u.y = Elem<H>::from_f2(f[2], f[3]);
    u.z = Elem<H>::from_f2(f[4], f[5]); u.w = Elem<H>::from_f2(f[6], f[7]);
    *reinterpret_cast<uint4*>(p) = u;
  }
};
template <> struct Vec<__half> : Vec16<__half> {};
template <> struct Vec<__nv_bfloat16> : Vec16<__nv_bfloat16> {};

// Binary weights of one row: (wa, wb) normalised, s the merged LSE.
__device__ __forceinline__ void merge2_weights(float a, float b, float& wa, float& wb, float& s) {
  const float m = fmaxf(a, b);
  wa = 0.f;
  wb = 0.f;
  s = neg_inf();
  if (m != neg_inf()) {
    wa = ex2((a - m) * kLog2e);
    wb = ex2((b - m) * kLog2e);
    const float den = wa + wb;
    s = m + lg2(den) * kLn2;
    const float inv = 1.f / den;
    wa *= inv;
    wb *= inv;
  }
}

// Rows are (token, head) pairs.  A warp covers `32 / cpr` rows at a time
// when a row has cpr <= 32 16-byte chunks, else one row in 32-chunk steps.
// With at most one chunk per lane (head_dim 128 in any dtype) a warp step
// takes two row groups, a grid stride apart, and issues both groups'
// vector and LSE loads before any arithmetic: two rows' bytes in flight per
// warp and one memory round trip per step.
template <typename T>
__global__ void __launch_bounds__(256) merge2_kernel(const T* __restrict__ va, const float* sa,
                                                     const T* __restrict__ vb, const float* sb,
                                                     T* vo, float* so, int64_t rows, int cpr) {
  using V = Vec<T>;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (gridDim.x * (int64_t)blockDim.x) >> 5;
  const int rpw = cpr >= 32 ? 1 : 32 / cpr;          // rows per warp step
  const int sub_row = cpr >= 32 ? 0 : lane / cpr;
  const int chunk0 = cpr >= 32 ? lane : lane % cpr;
  const int cstep = cpr >= 32 ? 32 : cpr;
  const int64_t stride = nwarps * rpw;
  if (cpr <= 32) {
    for (int64_t r0 = warp * rpw; r0 < rows; r0 += 2 * stride) {
      const int64_t row0 = r0 + sub_row, row1 = row0 + stride;
      const bool act0 = row0 < rows, act1 = row1 < rows;
      const int64_t off0 = (row0 * cpr + chunk0) * V::N, off1 = (row1 * cpr + chunk0) * V::N;
      float x0[V::N], y0[V::N], x1[V::N], y1[V::N];
      if (act0) {
        V::load(va + off0, x0);
        V::load(vb + off0, y0);
      }
      if (act1) {
        V::load(va + off1, x1);
        V::load(vb + off1, y1);
      }
      const float a0 = act0 ? sa[row0] : 0.f, b0 = act0 ? sb[row0] : 0.f;
      const float a1 = act1 ? sa[row1] : 0.f, b1 = act1 ? sb[row1] : 0.f;
      float wa0, wb0, s0, wa1, wb1, s1;
      merge2_weights(a0, b0, wa0, wb0, s0);
      merge2_weights(a1, b1, wa1, wb1, s1);
      if (act0) {
#pragma unroll
        for (int i = 0; i < V::N; ++i) x0[i] = x0[i] * wa0 + y0[i] * wb0;
        V::store(vo + off0, x0);
        if (chunk0 == 0) so[row0] = s0;
      }
      if (act1) {
#pragma unroll
        for (int i = 0; i < V::N; ++i) x1[i] = x1[i] * wa1 + y1[i] * wb1;
        V::store(vo + off1, x1);
        if (chunk0 == 0) so[row1] = s1;
      }
    }
    return;
  }
  for (int64_t r0 = warp * rpw; r0 < rows; r0 += stride) {
    const int64_t row = r0 + sub_row;
    if (row >= rows) continue;
    float wa, wb, s;
    merge2_weights(sa[row], sb[row], wa, wb, s);
    for (int c = chunk0; c < cpr; c += cstep) {
      const int64_t off = (row * cpr + c) * V::N;
      float x[V::N], y[V::N];
      V::load(va + off, x);
      V::load(vb + off, y);
#pragma unroll
      for (int i = 0; i < V::N; ++i) x[i] = x[i] * wa + y[i] * wb;
      V::store(vo + off, x);
    }
    if (chunk0 == 0) so[row] = s;
  }
}

// N floats of a row written to an output of type TO at element offset off
// (N = the input vector's width: 4 for fp32 inputs, 8 for 16-bit ones).
template <typename TO, int N> struct Out;
template <int N> struct Out<float, N> {
  static __device__ __forceinline__ void store(float* o, int64_t off, const float* f) {
#pragma unroll
    for (int i = 0; i < N; i += 4) *reinterpret_cast<float4*>(o + off + i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
  }
};
template <typename H, int N> struct Out16 {
  static __device__ __forceinline__ void store(H* o, int64_t off, const float* f) {
    if constexpr (N == 8) {
      uint4 u;
      u.x = Elem<H>::from_f2(f[0], f[1]); u.y = Elem<H>::from_f2(f[2], f[3]);
      u.z = Elem<H>::from_f2(f[4], f[5]); u.w = Elem<H>::from_f2(f[6], f[7]);
      *reinterpret_cast<uint4*>(o + off) = u;
    } else {
      static_assert(N == 4, "row vector width");
      *reinterpret_cast<uint2*>(o + off) = make_uint2(Elem<H>::from_f2(f[0], f[1]), Elem<H>::from_f2(f[2], f[3]));
    }
  }
};
template <int N> struct Out<__half, N> : Out16<__half, N> {};
template <int N> struct Out<__nv_bfloat16, N> : Out16<__nv_bfloat16, N> {};

// n-ary: v [T, n, H, D], s [T, n, H] -> [T, H, D], [T, H]; the output may
// have another element type than the states (TO: fp32 states merged into
// a 16-bit result, rounded once).
template <typename T, typename TO = T>
__global__ void __launch_bounds__(256) mergen_kernel(const T* __restrict__ v, const float* s,
                                                     TO* vo, float* so, int64_t n_tokens,
                                                     int n_states, int n_heads, int cpr) {
  using V = Vec<T>;
  using W = Out<TO, V::N>;
  const int lane = threadIdx.x & 31;
  const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (gridDim.x * (int64_t)blockDim.x) >> 5;
  const int64_t rows = n_tokens * n_heads;
  const int rpw = cpr >= 32 ? 1 : 32 / cpr;
  const int sub_row = cpr >= 32 ? 0 : lane / cpr;
  const int chunk0 = cpr >= 32 ? lane : lane % cpr;
  const int cstep = cpr >= 32 ? 32 : cpr;
  // Fast path: one chunk per lane and at most one state per lane of the
  // row's lane group (cstep lanes, a power of two).  The group's lanes load
  // the row's LSEs in parallel and reduce their maximum and sum with
  // shuffles, while the first four states' vector loads are in flight;
  // each lane then takes the weights from the lanes that own them.
  const bool fast = cpr <= 32 && n_states <= cstep && (cstep & (cstep - 1)) == 0;
  if (fast) {
    const int base = lane - chunk0;  // first lane of this row's group
    const unsigned gmask = cstep == 32 ? 0xffffffffu : (((1u << cstep) - 1u) << base);
    for (int64_t r0 = warp * rpw; r0 < rows; r0 += nwarps * rpw) {
      const int64_t row = r0 + sub_row;
      const bool active = row < rows;
      const int64_t t = active ? row / n_heads : 0;
      const int h = active ? (int)(row % n_heads) : 0;
      const T* vrow = v + ((t * n_states * n_heads + h) * cpr + chunk0) * V::N;
      const int64_t vstride = (int64_t)n_heads * cpr * V::N;  // one state further
      float x[4][V::N];
      if (active) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (u < n_states) V::load(vrow + u * vstride, x[u]);
      }
      const float lse = active && chunk0 < n_states ? s[(t * n_states + chunk0) * n_heads + h] : neg_inf();
      float m = lse;
      for (int o = 1; o < cstep; o <<= 1) m = fmaxf(m, __shfl_xor_sync(gmask, m, o));
      const float e = m == neg_inf() ? 0.f : ex2((lse - m) * kLog2e);
      float den = e;
      for (int o = 1; o < cstep; o <<= 1) den += __shfl_xor_sync(gmask, den, o);
      const float w_mine = den > 0.f ? e / den : 0.f;
      float acc[V::N];
#pragma unroll
      for (int k = 0; k < V::N; ++k) acc[k] = 0.f;
      for (int i = 0; i < n_states; i += 4) {
        if (i > 0 && active) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (i + u < n_states) V::load(vrow + (i + u) * vstride, x[u]);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = __shfl_sync(gmask, w_mine, base + ((i + u) & (cstep - 1)));
          if (i + u < n_states && m != neg_inf()) {  // an all-empty row stays 0
#pragma unroll
            for (int k = 0; k < V::N; ++k) acc[k] += w * x[u][k];
          }
        }
      }
      if (active) {
        W::store(vo, (row * cpr + chunk0) * V::N, acc);
        if (chunk0 == 0) so[row] = m == neg_inf() ? neg_inf() : m + lg2(den) * kLn2;
      }
    }
    return;
  }
  for (int64_t r0 = warp * rpw; r0 < rows; r0 += nwarps * rpw) {
    const int64_t row = r0 + sub_row;
    const bool active = row < rows;
    const int64_t t = active ? row / n_heads : 0;
    const int h = active ? (int)(row % n_heads) : 0;
    const float* srow = s + t * n_states * n_heads + h;
    float m = neg_inf();
    if (active)
      for (int i = 0; i < n_states; ++i) m = fmaxf(m, srow[(int64_t)i * n_heads]);
    float den = 0.f;
    if (active && m != neg_inf())
      for (int i = 0; i < n_states; ++i) den += ex2((srow[(int64_t)i * n_heads] - m) * kLog2e);
    const float inv = den > 0.f ? 1.f / den : 0.f;
    if (active) {
      for (int c = chunk0; c < cpr; c += cstep) {
        float acc[V::N];
#pragma unroll
        for (int k = 0; k < V::N; ++k) acc[k] = 0.f;
        if (m != neg_inf()) {
          int i = 0;
          for (; i + 4 <= n_states; i += 4) {
            float x[4][V::N], w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int64_t off = (((t * n_states + i + u) * n_heads + h) * cpr + c) * V::N;
              V::load(v + off, x[u]);
              w[u] = ex2((srow[(int64_t)(i + u) * n_heads] - m) * kLog2e) * inv;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
              for (int k = 0; k < V::N; ++k) acc[k] += w[u] * x[u][k];
          }
          for (; i < n_states; ++i) {
            float x[V::N];
            const int64_t off = (((t * n_states + i) * n_heads + h) * cpr + c) * V::N;
            V::load(v + off, x);
            const float w = ex2((srow[(int64_t)i * n_heads] - m) * kLog2e) * inv;
#pragma unroll
            for (int k = 0; k < V::N; ++k) acc[k] += w * x[k];
          }
        }
        W::store(vo, (row * cpr + c) * V::N, acc);
      }
    }
    __syncwarp();
    if (active && chunk0 == 0) so[row] = (m == neg_inf()) ? neg_inf() : m + lg2(den) * kLn2;
  }
}

int grid_for(int64_t warps_needed) {
  const int64_t per_block = 8;  // 256 threads
  int64_t blocks = (warps_needed + per_block - 1) / per_block;
  const int64_t cap = (int64_t)num_sms() * 8;  // 8 x 256-thread blocks per SM resident
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace

int launch_merge_state(const void* va, const float* sa, const void* vb, const float* sb, void* vo,
                       float* so, int64_t rows, int head_dim, int dtype, void* stream) {
  const int esz = dtype == PKC_F32 ? 4 : 2;
  const int cpr = head_dim * esz / 16;
  const int rpw = cpr >= 32 ? 1 : 32 / cpr;
  const int grid = grid_for((rows + rpw - 1) / rpw);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == PKC_F32)
    merge2_kernel<float><<<grid, 256, 0, st>>>((const float*)va, sa, (const float*)vb, sb, (float*)vo, so, rows, cpr);
  else if (dtype == PKC_F16)
    merge2_kernel<__half><<<grid, 256, 0, st>>>((const __half*)va, sa, (const __half*)vb, sb, (__half*)vo, so, rows, cpr);
  else
    merge2_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)va, sa, (const __nv_bfloat16*)vb, sb,
                                                       (__nv_bfloat16*)vo, so, rows, cpr);
  return (int)cudaGetLastError();
}

int launch_merge_states_to(const void* v, const float* s, void* vo, float* so, int64_t n_tokens, int n_states,
                           int n_heads, int head_dim, int dtype, int out_dtype, void* stream) {
  if (out_dtype == dtype) return launch_merge_states(v, s, vo, so, n_tokens, n_states, n_heads, head_dim, dtype, stream);
  if (dtype != PKC_F32) return (int)cudaErrorInvalidValue;  // 16-bit states are merged into their own type
  const int cpr = head_dim * 4 / 16;
  const int rpw = cpr >= 32 ? 1 : 32 / cpr;
  const int64_t rows = n_tokens * n_heads;
  const int grid = grid_for((rows + rpw - 1) / rpw);
  cudaStream_t st = (cudaStream_t)stream;
  if (out_dtype == PKC_F16)
    mergen_kernel<float, __half><<<grid, 256, 0, st>>>((const float*)v, s, (__half*)vo, so, n_tokens, n_states,
                                                       n_heads, cpr);
  else
    mergen_kernel<float, __nv_bfloat16><<<grid, 256, 0, st>>>((const float*)v, s, (__nv_bfloat16*)vo, so, n_tokens,
                                                              n_states, n_heads, cpr);
  return (int)cudaGetLastError();
}

int launch_merge_states(const void* v, const float* s, void* vo, float* so, int64_t n_tokens,
                        int n_states, int n_heads, int head_dim, int dtype, void* stream) {
  const int esz = dtype == PKC_F32 ? 4 : 2;
  const int cpr = head_dim * esz / 16;
  const int rpw = cpr >= 32 ? 1 : 32 / cpr;
  const int64_t rows = n_tokens * n_heads;
  const int grid = grid_for((rows + rpw - 1) / rpw);
  cudaStream_t st = (cudaStream_t)stream;
  if (dtype == PKC_F32)
    mergen_kernel<float><<<grid, 256, 0, st>>>((const float*)v, s, (float*)vo, so, n_tokens, n_states, n_heads, cpr);
  else if (dtype == PKC_F16)
    mergen_kernel<__half><<<grid, 256, 0, st>>>((const __half*)v, s, (__half*)vo, so, n_tokens, n_states, n_heads, cpr);
  else
    mergen_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)v, s, (__nv_bfloat16*)vo, so, n_tokens,
                                                       n_states, n_heads, cpr);
  return (int)cudaGetLastError();
}

}  // namespace pkc
