// decode_shrink.cu -- the MODE_SHRINK instantiations of the decode kernel (see decode_impl.cuh).
#include "decode_impl.cuh"

namespace mlora {

cudaError_t launch_decode_shrink(int dtype, const DecodeParams &p, unsigned grid, size_t smem, int cluster,
                             bool pdl, cudaStream_t stream) {
  if (dtype == MLORA_BF16) return decode::dispatch<MLORA_BF16, MODE_SHRINK>(p, grid, smem, cluster, pdl, stream);
  return decode::dispatch<MLORA_FP16, MODE_SHRINK>(p, grid, smem, cluster, pdl, stream);
}

}  // namespace mlora
