// In-place append of one decoded token's K and V to the paged cache.
//
// Hugging Face "Paged attention", decoding path: the new token of request b
// goes to the slot after its cached tokens, page block_table[b][len / ps],
// slot len % ps with len = cache_seqlens[b], and the length grows by one.
// One block per request: its threads copy the Hkv rows of K and V (16 bytes
// per thread and step), then one thread bumps the length.  A page id that
// is negative or past the pool is reported in the status word and nothing
// of that request is written.
#include <cuda_runtime.h>

#include "pkc_device.cuh"
#include "pkc_internal.h"

namespace pkc {
namespace {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads) append_kv_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  if (p.mask && p.mask[b] == 0) return;
  const int len = p.cache_seqlens[b];
  const int64_t page_idx = len / p.page_size;
  int32_t page = -1;
  if (len >= 0 && page_idx < p.bt_stride) page = p.block_table[(int64_t)b * p.bt_stride + page_idx];
  if (page < 0 || page >= p.num_pages) {
    if (threadIdx.x == 0) report(p.status, PKC_ERR_BLOCK_TABLE);
    return;  // uniform over the block: nothing written, length unchanged
  }
  const int slot = len % p.page_size;
  const int64_t row_bytes = (int64_t)p.hkv * p.row_bytes;  // one token, all KV heads
  const int64_t dst = ((int64_t)page * p.page_size + slot) * row_bytes;
  const int64_t src = (int64_t)b * row_bytes;
  const int n16 = (int)(row_bytes / 16);
  for (int i = threadIdx.x; i < n16; i += blockDim.x) {
    reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_cache) + dst)[i] =
        reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.k_new) + src)[i];
    reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_cache) + dst)[i] =
        reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.v_new) + src)[i];
  }
  __syncthreads();  // every thread has read len before it changes
  if (threadIdx.x == 0) p.cache_seqlens[b] = len + 1;
}

}  // namespace

int launch_append_kv(const AppendParams& p, int batch, void* stream) {
  if (batch <= 0) return 0;
  append_kv_kernel<<<batch, kAppendThreads, 0, (cudaStream_t)stream>>>(p);
  return (int)cudaGetLastError();
}

}  // namespace pkc
