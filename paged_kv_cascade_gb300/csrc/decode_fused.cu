// CUDA-core paged decode with the contraction fused in (the instantiations
// with kFuse = true, compiled apart from the others to halve each build step).
#include "decode_simt.cuh"

namespace pkc {

int launch_paged_decode_simt_fused(const DecodeParams& p, int grid_x, int dtype, int hg, const void* mk,
                                   const void* mv, const void* prefix_maps, void* stream) {
  return launch_simt_mode<true>(p, grid_x, dtype, hg, *static_cast<const CUtensorMap*>(mk),
                                *static_cast<const CUtensorMap*>(mv), *static_cast<const PrefixMaps*>(prefix_maps),
                                (cudaStream_t)stream);
}

}  // namespace pkc
