// sgemm_internal.h -- host-side declarations shared by the translation units of libsgemm.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sgemm_impl {

// Everything a GEMM kernel needs besides its tensor maps.
struct GemmParams {
  int M, N, K;
  float alpha, beta;
  const float* A;  // used by the generic kernel (the TMA kernel reads through tensor maps)
  const float* B;
  float* C;        // final output (split == 1) ...
  float* ws;       // ... or the partial-sum workspace [split][M][ws_ld] (split > 1)
  int64_t lda, ldb, ldc, ws_ld;
  int k_tiles_per_split;  // K tiles (of the kernel's BK) per slice
  int tiles_m, tiles_n;   // output tiles
  int c_vec;              // 1: C is 16-byte aligned and ldc % 4 == 0
  uint64_t timeout_ns;    // limit of every in-kernel wait
  unsigned* fault;        // device fault word (bits of FaultBits), see fault_word()
};

// Shapes of the TMA-fed SIMT kernel.
enum class TmaTile { k128x128, k64x256 };

struct GenericTileShape {
  int bm, bn, bk, threads;
};
GenericTileShape generic_tile_shape();

// Launchers: enqueue one kernel on `stream`, return the launch error.
// TMA-fed kernel, one entry per operand layout (kernel_tma_{nn,nt,tn,tt}.cu).
#define SGEMM_DECLARE_TMA_OP(op)                                                                   \
  cudaError_t launch_tma_op_##op(TmaTile tile, const CUtensorMap& mapA, const CUtensorMap& mapB, \
                                 const GemmParams& p, int split, cudaStream_t stream);            \
  cudaError_t prepare_tma_op_##op();
SGEMM_DECLARE_TMA_OP(nn)
SGEMM_DECLARE_TMA_OP(nt)
SGEMM_DECLARE_TMA_OP(tn)
SGEMM_DECLARE_TMA_OP(tt)
#undef SGEMM_DECLARE_TMA_OP
// 3xTF32 tensor-core kernel (kernel_tf32x3.cu), 128x128x32 tiles, any op, optional K split.
cudaError_t prepare_tf32x3();
cudaError_t launch_tf32x3(bool transA, bool transB, const CUtensorMap& mapA, const CUtensorMap& mapB,
                          const GemmParams& p, int split, cudaStream_t stream);
cudaError_t launch_generic_gemm(bool transA, bool transB, const GemmParams& p, int split,
                                cudaStream_t stream);
cudaError_t launch_splitk_reduce(const GemmParams& p, int split, cudaStream_t stream);
cudaError_t launch_scale(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint64_t timeout_ns, unsigned* fault, cudaStream_t stream);

// Device address of the current device's fault word (looked up once per device).
cudaError_t fault_word(unsigned** ptr);
// Reads and clears the current device's fault word (synchronous).
cudaError_t take_faults(unsigned* bits);

}  // namespace sgemm_impl
