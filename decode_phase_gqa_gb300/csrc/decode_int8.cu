// Instantiations of the tensor-core split-KV decode kernel for the int8 KV cache.
#include "decode_mma.cuh"

namespace kvattn {

cudaError_t launch_decode_int8(const DecodeParams &p, int head_dim, int gs, int grid,
                               cudaStream_t stream, int *ctas_per_sm, bool launch) {
  if (p.n_layers > 1)  // several layer caches: the instantiations of decode_int8_layers.cu
    return launch_decode_int8_layers(p, head_dim, gs, grid, stream, ctas_per_sm, launch);
  if (head_dim == 64) {
    if (gs == 4) return launch_decode_mma_t<64, 4, true, false>(p, grid, stream, ctas_per_sm, launch);
    if (gs == 2) return launch_decode_mma_t<64, 2, true, false>(p, grid, stream, ctas_per_sm, launch);
    return launch_decode_mma_t<64, 1, true, false>(p, grid, stream, ctas_per_sm, launch);
  }
  if (gs == 4) return launch_decode_mma_t<128, 4, true, false>(p, grid, stream, ctas_per_sm, launch);
  if (gs == 2) return launch_decode_mma_t<128, 2, true, false>(p, grid, stream, ctas_per_sm, launch);
  return launch_decode_mma_t<128, 1, true, false>(p, grid, stream, ctas_per_sm, launch);
}

}  // namespace kvattn
