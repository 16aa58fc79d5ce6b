// kernel_tma_nn.cu -- instantiations of the TMA-fed SIMT kernel for op(A) = A, op(B) = B.
// (One translation unit per operand layout so the build compiles them in parallel.)
#include "kernel_tma.cuh"

namespace sgemm_impl {

cudaError_t launch_tma_op_nn(TmaTile tile, const CUtensorMap& mapA, const CUtensorMap& mapB,
                             const GemmParams& p, int split, cudaStream_t stream) {
  if (tile == TmaTile::k128x128) return tma::launch<4, 2, false, false>(mapA, mapB, p, split, stream);
  return tma::launch<2, 4, false, false>(mapA, mapB, p, split, stream);
}

cudaError_t prepare_tma_op_nn() {
  cudaError_t e = tma::set_attributes<4, 2, false, false>();
  if (e != cudaSuccess) return e;
  return tma::set_attributes<2, 4, false, false>();
}

}  // namespace sgemm_impl
