// CUDA-core paged decode with the contraction fused in (the instantiations
// with kFuse = true, compiled apart from the others to halve each build step).
#include "decode_simt.cuh"

namespace pkc {

int launch_paged_decode_simt_fused(const DecodeParams& p, int grid_x, int dtype, int hg, const void* mk,
                                   const void* mv, void* stream) {
  return launch_simt_mode<true>(p, grid_x, dtype, hg, *static_cast<const CUtensorMap*>(mk),
                                *static_cast<const CUtensorMap*>(mv), (cudaStream_t)stream);
}

}  // namespace pkc
