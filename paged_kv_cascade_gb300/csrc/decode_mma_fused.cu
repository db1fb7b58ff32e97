// Tensor-core paged decode with the contraction fused in (the instantiations
// with kFuse = true, compiled apart from the others to halve each build step).
#include "decode_mma.cuh"

namespace pkc {

int launch_paged_decode_mma_fused(const DecodeParams& p, int grid_x, int kv_kind, int hg, const void* mk,
                                  const void* mv, void* stream) {
  return launch_mma_mode<true>(p, grid_x, kv_kind, hg, *static_cast<const CUtensorMap*>(mk),
                               *static_cast<const CUtensorMap*>(mv), (cudaStream_t)stream);
}

}  // namespace pkc
