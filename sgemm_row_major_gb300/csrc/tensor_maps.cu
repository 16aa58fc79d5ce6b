// tensor_maps.cu -- TMA tensor maps of the GEMM operands (host code).
//
// Every TMA-fed kernel reads A and B through 3-D float32 maps {contiguous
// elements of a stored row, stored rows, product index}.  A single product
// (sgemm) is the case of a product extent of 1; a strided batch gives the
// third dimension the batch count and the batch stride, so one map serves
// every product of the call and a kernel only changes the third coordinate.
#include <mutex>

#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encode_fn(EncodeTiledFn* out) {
  static EncodeTiledFn fn = nullptr;
  static cudaError_t err = cudaSuccess;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (err == cudaSuccess && (q != cudaDriverEntryPointSuccess || !p)) err = cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  *out = fn;
  return err;
}

// Map over `products` row-major matrices of `outer` rows x `inner` contiguous
// floats, row stride `ld`, product stride `stride` (elements); box
// {box_inner, box_outer, 1}.
cudaError_t encode_3d(const float* base, int64_t inner, int64_t outer, int64_t ld, int64_t products,
                      int64_t stride, int box_inner, int box_outer, bool swizzle128, CUtensorMap* map) {
  EncodeTiledFn fn = nullptr;
  cudaError_t e = encode_fn(&fn);
  if (e != cudaSuccess) return e;
  if (products <= 1) {
    products = 1;
    stride = outer * ld;  // unused with one product, but must be a valid stride
  }
  const cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)products};
  const cuuint64_t strides[2] = {(cuuint64_t)ld * 4u, (cuuint64_t)stride * 4u};
  const cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// cuTensorMapEncodeTiled fails with CUDA_ERROR_INVALID_CONTEXT on a thread
// that has no current context: a host thread whose first CUDA call is into
// this library has none yet (cudaGetDevice does not bind one).  cudaSetDevice
// makes the device's primary context current; once per thread and device.
cudaError_t bind_primary_context() {
  thread_local int bound = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || bound == dev) return e;
  e = cudaSetDevice(dev);
  if (e == cudaSuccess) bound = dev;
  return e;
}

}  // namespace

cudaError_t encode_split_map(const float* base, int64_t K, int64_t rows, int64_t ldk, int64_t products,
                             CUtensorMap* map, int box_rows) {
  cudaError_t e = bind_primary_context();
  if (e != cudaSuccess) return e;
  return encode_3d(base, K, rows, ldk, products, rows * ldk, 32, box_rows, true, map);
}

cudaError_t encode_bf16_map(const void* base, int64_t K, int64_t rows, int64_t ldk, CUtensorMap* map) {
  cudaError_t e = bind_primary_context();
  if (e != cudaSuccess) return e;
  EncodeTiledFn fn = nullptr;
  e = encode_fn(&fn);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, 1};
  const cuuint64_t strides[2] = {(cuuint64_t)ldk * 2u, (cuuint64_t)(rows * ldk) * 2u};
  const cuuint32_t box[3] = {64u, 128u, 1u};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_matrix_map(const float* base, int64_t inner, int64_t outer, int64_t ld, int box_inner,
                              int box_outer, CUtensorMap* map) {
  cudaError_t e = bind_primary_context();
  if (e != cudaSuccess) return e;
  return encode_3d(base, inner, outer, ld, 1, 0, box_inner, box_outer, box_inner == 32, map);
}

cudaError_t encode_operand_maps(bool ta, bool tb, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                int64_t stride_a, const float* B, int64_t ldb, int64_t stride_b, int batch,
                                int bm, int bn, int bk, CUtensorMap* mapA, CUtensorMap* mapB, int* za, int* zb) {
  const int64_t pa = (batch > 1 && stride_a != 0) ? batch : 1;
  const int64_t pb = (batch > 1 && stride_b != 0) ? batch : 1;
  cudaError_t e = bind_primary_context();
  if (e != cudaSuccess) return e;
  *za = pa > 1 ? 1 : 0;
  *zb = pb > 1 ? 1 : 0;
  // op(A): 'N' -> stored M x K, K contiguous (swizzled K-major tile);
  //        'T' -> stored K x M, M contiguous.
  e = ta ? encode_3d(A, M, K, lda, pa, stride_a, bm, bk, false, mapA)
         : encode_3d(A, K, M, lda, pa, stride_a, bk, bm, true, mapA);
  if (e != cudaSuccess) return e;
  // op(B): 'N' -> stored K x N, N contiguous; 'T' -> stored N x K, K contiguous (swizzled).
  return tb ? encode_3d(B, K, N, ldb, pb, stride_b, bk, bn, true, mapB)
            : encode_3d(B, N, K, ldb, pb, stride_b, bn, bk, false, mapB);
}

}  // namespace sgemm_impl
