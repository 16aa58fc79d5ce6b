// kernel_small.h -- launcher of the small-product kernel (kernel_small.cu).
#pragma once

#include <cuda_runtime.h>

#include "sgemm_internal.h"

namespace sgemm_impl {

// Persistent grid of `grid` CTAs (1 <= grid <= p.batch; four fit on an SM),
// 64 threads each, products dealt round-robin; M <= 64 and N <= 64, any K.
// The planner guarantees the kernel's copy rules: A and B 16-byte aligned,
// lda, ldb and the batch strides multiples of 4, and K (op 'N' of A, op 'T'
// of B), M (op 'T' of A) and N (op 'N' of B) multiples of 4.
cudaError_t launch_small_gemm(bool transA, bool transB, const GemmParams& p, int grid, cudaStream_t stream);

// Sets the kernels' dynamic shared-memory size (32 KB); once per device.
cudaError_t prepare_small_gemm();

}  // namespace sgemm_impl
