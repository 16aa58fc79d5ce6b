// kernel_small.h -- launcher of the small-product kernel (kernel_small.cu).
#pragma once

#include <cuda_runtime.h>

#include "sgemm_internal.h"

namespace sgemm_impl {

// One CTA of 128 threads per product (grid = p.batch), M <= 64 and N <= 64,
// any K.  The planner guarantees the kernel's load rules: A and B 16-byte
// aligned, lda, ldb and the batch strides multiples of 4, and K (op 'N' of A,
// op 'T' of B), M (op 'T' of A) and N (op 'N' of B) multiples of 4.
cudaError_t launch_small_gemm(bool transA, bool transB, const GemmParams& p, cudaStream_t stream);

}  // namespace sgemm_impl
