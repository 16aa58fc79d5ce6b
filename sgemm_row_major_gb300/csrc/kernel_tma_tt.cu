// kernel_tma_tt.cu -- instantiations of the TMA-fed SIMT kernel for op(A) = A^T, op(B) = B^T.
// (One translation unit per operand layout so the build compiles them in parallel.)
#include "kernel_tma.cuh"

namespace sgemm_impl {

cudaError_t launch_tma_op_tt(TmaTile tile, const CUtensorMap& mapA, const CUtensorMap& mapB,
                             const GemmParams& p, int split, cudaStream_t stream) {
  if (tile == TmaTile::k128x128) return tma::launch<4, 2, true, true>(mapA, mapB, p, split, stream);
  return tma::launch<2, 4, true, true>(mapA, mapB, p, split, stream);
}

cudaError_t prepare_tma_op_tt() {
  cudaError_t e = tma::set_attributes<4, 2, true, true>();
  if (e != cudaSuccess) return e;
  return tma::set_attributes<2, 4, true, true>();
}

}  // namespace sgemm_impl
