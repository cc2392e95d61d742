// Instantiations of the tensor-core split-KV decode kernel for the bf16 KV cache
// over several layer caches in one launch (kvattn_decode_layers); the
// single-layer kernels of decode_bf16.cu leave the layer arithmetic out.
#include "decode_mma.cuh"

namespace kvattn {

cudaError_t launch_decode_bf16_layers(const DecodeParams &p, int head_dim, int gs, int grid,
                                      cudaStream_t stream, int *ctas_per_sm, bool launch) {
  if (head_dim == 64) {
    if (gs == 4) return launch_decode_mma_t<64, 4, false, true>(p, grid, stream, ctas_per_sm, launch);
    if (gs == 2) return launch_decode_mma_t<64, 2, false, true>(p, grid, stream, ctas_per_sm, launch);
    return launch_decode_mma_t<64, 1, false, true>(p, grid, stream, ctas_per_sm, launch);
  }
  if (gs == 4) return launch_decode_mma_t<128, 4, false, true>(p, grid, stream, ctas_per_sm, launch);
  if (gs == 2) return launch_decode_mma_t<128, 2, false, true>(p, grid, stream, ctas_per_sm, launch);
  return launch_decode_mma_t<128, 1, false, true>(p, grid, stream, ctas_per_sm, launch);
}

}  // namespace kvattn
