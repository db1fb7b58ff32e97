// Tensor-core paged decode: launch set-up and the kernels without the fused
// contraction (the kernel itself is in decode_mma.cuh; the instantiations
// with the fused contraction are compiled in decode_mma_fused.cu).
#include "decode_mma.cuh"

namespace pkc {

int mma_decode_heads_per_block(int hkv, int page_size) {
  const int hg = hkv % 8 == 0 ? 8 : hkv % 4 == 0 ? 4 : hkv % 2 == 0 ? 2 : 1;
  const int sl = page_size < kMaxSl ? page_size : kMaxSl;
  // A slice of sl slots x hg heads must fill whole 1024-byte swizzle atoms
  // (sl hg >= 8) and a stage a whole number of slices (sl a power of two),
  // so every fragment address stays inside its stage.
  const bool pow2 = (sl & (sl - 1)) == 0;
  return pow2 && (sl * hg) % 8 == 0 ? hg : 0;
}

int launch_paged_decode_mma(const DecodeParams& p, int grid_x, int kv_kind, void* stream) {
  if (grid_x <= 0) return 0;
  const int hg = mma_decode_heads_per_block(p.hkv, p.page_size);
  if (hg == 0) return (int)cudaErrorInvalidValue;
  const int sl = p.page_size < kMaxSl ? p.page_size : kMaxSl;
  const uint64_t es = kv_kind == kKvE4M3 ? 1 : 2;
  // 4-D view (dim, slot, head, page) of [num_pages][page_size][Hkv][128];
  // a box is sl slots x hg heads of one page, 128 bytes of each row.
  const uint64_t dims[4] = {(uint64_t)D, (uint64_t)p.page_size, (uint64_t)p.hkv,
                            (uint64_t)(p.num_pages > 0 ? p.num_pages : 1)};
  const uint64_t strides[3] = {D * es * p.hkv, D * es, D * es * p.hkv * p.page_size};
  const uint32_t box[4] = {(uint32_t)(kLine / es), (uint32_t)sl, (uint32_t)hg, 1u};
  const int tdt = kv_kind == kKvE4M3 ? PKC_E4M3 : kv_kind == kKvBF16 ? PKC_BF16 : PKC_F16;
  alignas(64) CUtensorMap mk, mv;
  if (!encode_tiled_map(&mk, p.k_cache, tdt, 4, dims, strides, box, true) ||
      !encode_tiled_map(&mv, p.v_cache, tdt, 4, dims, strides, box, true))
    return -1;
  cudaStream_t st = (cudaStream_t)stream;
  if (p.fuse.enabled) return launch_paged_decode_mma_fused(p, grid_x, kv_kind, hg, &mk, &mv, st);
  return launch_mma_mode<false>(p, grid_x, kv_kind, hg, mk, mv, st);
}

}  // namespace pkc
