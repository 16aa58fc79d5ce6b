// kernel_small.cu -- many small products (M <= 64, N <= 64; a strided batch of
// them): one CTA computes a product's whole output tile, then moves on to the
// next product, whose copies are already in flight.
//
// For such products the tensor-core kernel's 128x128 tile is three quarters
// padding, and its pipeline (TMA ring, split, MMA issue, fold) is set up for
// long K loops.  Here the work of a CTA is a list of (product, 64-k chunk)
// items; each item's op(A) and op(B) chunks (16 KB each) are copied into one
// of two shared-memory stages with 16-byte cp.async copies, as they are
// stored in global memory (no transposition), and the next item's copies are
// issued before the current item is computed.  128 threads each accumulate a
// 4x8 block of the 64x64 tile with packed FP32 FMAs (fma.rn.f32x2, IEEE
// round-to-nearest); a chunk's partial sums are added into a second set of
// registers after every chunk, so no accumulator sums more than 64 products.
// The grid is persistent (three CTAs per SM, products dealt round-robin), so
// HBM traffic and FMA work overlap within a CTA and across the CTAs of an SM.
//
// Shared layout of a stage: the A chunk, then the B chunk, each 64 rows of 64
// floats (16 groups of 16 bytes).  A stored K-contiguous (op 'N') is kept as
// [m][k] and B stored K-contiguous (op 'T') as [n][k]; in both, group g of row
// r sits at g XOR ((r / 4) % 8), which puts the rows a warp reads together in
// distinct bank groups.  A stored M-contiguous ('T') and B stored
// N-contiguous ('N') are kept as [k][m] and [k][n], unswizzled: a warp reads
// contiguous groups of one row.
//
// Requirements (checked by the planner): A, B 16-byte aligned, lda, ldb and
// the batch strides multiples of 4 floats, and the extent copied along a row
// a multiple of 4: K for op(A) 'N' and op(B) 'T', M for op(A) 'T', N for
// op(B) 'N'.  Groups outside the matrix are zero-filled, never read.
#include <cstdint>

#include "kernel_small.h"

namespace sgemm_impl {
namespace {

constexpr int SM_T = 64;                              // output tile and K chunk
constexpr int SM_THREADS = 128;                       // 16 x 8 threads, 4 rows x 8 columns each
constexpr int SM_CHUNK_FLOATS = SM_T * SM_T;          // one operand chunk
constexpr int SM_STAGE_FLOATS = 2 * SM_CHUNK_FLOATS;  // A chunk + B chunk
constexpr int SM_SMEM_BYTES = 2 * SM_STAGE_FLOATS * 4;
static_assert(SM_SMEM_BYTES == 65536, "two 32 KB stages");
static_assert(3 * (SM_SMEM_BYTES + 1024) <= 228 * 1024, "three CTAs per SM");

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros and reads nothing.
__device__ __forceinline__ void cp_async16(uint32_t dst, const float* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;\n" ::: "memory"); }

__device__ __forceinline__ float4 lds4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Copy one operand chunk, 64 rows of 16 groups: row r is matrix row r0 + r and
// group g its columns c0 + 4g .. +3; rows >= rows_valid and columns >=
// cols_valid (a multiple of 4) are zero.  `swizzle` places group g of row r at
// g ^ ((r / 4) % 8).
__device__ __forceinline__ void copy_chunk(float* dst, const float* base, int64_t ld, int r0, int rows_valid,
                                           int c0, int cols_valid, bool swizzle, int tid) {
  const uint32_t d0 = smem_addr(dst);
#pragma unroll
  for (int q = 0; q < SM_CHUNK_FLOATS / 4 / SM_THREADS; ++q) {
    const int e = tid + SM_THREADS * q;  // 0 .. 1023
    const int r = e >> 4, g = e & 15;
    const int row = r0 + r, col = c0 + 4 * g;
    const bool ok = row < rows_valid && col < cols_valid;
    const float* src = ok ? base + (int64_t)row * ld + col : base;
    const int gs = swizzle ? (g ^ ((r >> 2) & 7)) : g;
    cp_async16(d0 + (uint32_t)((r * SM_T + 4 * gs) * 4), src, ok ? 16 : 0);
  }
}

template <bool TA, bool TB>
__global__ void __launch_bounds__(SM_THREADS, 3) small_gemm_kernel(const GemmParams p) {
  extern __shared__ __align__(16) float smem[];
  const int tid = threadIdx.x;
  const int ty = tid >> 3, tx = tid & 7;  // rows 4ty .. +3, columns 4tx .. +3 and 32 + 4tx .. +3
  const int chunks = (p.K + SM_T - 1) / SM_T;
  // items of this CTA: products blockIdx.x, blockIdx.x + gridDim.x, ..., `chunks` K chunks each
  const int my_products = (p.batch - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int items = my_products * chunks;

  const auto issue = [&](int item) {
    const int64_t prod = (int64_t)blockIdx.x + (int64_t)(item / chunks) * gridDim.x;
    const int k0 = (item % chunks) * SM_T;
    float* st = smem + (item & 1) * SM_STAGE_FLOATS;
    const float* A = p.A + prod * p.stride_a;
    const float* B = p.B + prod * p.stride_b;
    if (!TA) copy_chunk(st, A, p.lda, 0, p.M, k0, p.K, true, tid);   // [m][k]
    else copy_chunk(st, A, p.lda, k0, p.K, 0, p.M, false, tid);      // [k][m]
    if (!TB) copy_chunk(st + SM_CHUNK_FLOATS, B, p.ldb, k0, p.K, 0, p.N, false, tid);  // [k][n]
    else copy_chunk(st + SM_CHUNK_FLOATS, B, p.ldb, 0, p.N, k0, p.K, true, tid);       // [n][k]
  };

  float2 acc[4][4], mst[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = mst[i][j] = make_float2(0.0f, 0.0f);

  if (items > 0) issue(0);
  cp_async_commit();
  for (int it = 0; it < items; ++it) {
    // the stage of item it + 1 was last read by item it - 1, which every
    // thread finished before the barrier at the end of the previous pass
    if (it + 1 < items) issue(it + 1);
    cp_async_commit();
    cp_async_wait_one();  // this thread's copies of item it have landed ...
    __syncthreads();      // ... and every thread's
    const float* As = smem + (it & 1) * SM_STAGE_FLOATS;
    const float* Bs = As + SM_CHUNK_FLOATS;
#pragma unroll 2
    for (int k4 = 0; k4 < SM_T / 4; ++k4) {
      float a[4][4];  // a[i][kk] = op(A)[4ty + i][4k4 + kk]
      float b[8][4];  // b[j][kk] = op(B)[4k4 + kk][column j of the thread]
      if (!TA) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 v = lds4(As + (4 * ty + i) * SM_T + 4 * (k4 ^ (ty & 7)));
          a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 v = lds4(As + (4 * k4 + kk) * SM_T + 4 * ty);
          a[0][kk] = v.x; a[1][kk] = v.y; a[2][kk] = v.z; a[3][kk] = v.w;
        }
      }
      if (!TB) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 v0 = lds4(Bs + (4 * k4 + kk) * SM_T + 4 * tx);
          const float4 v1 = lds4(Bs + (4 * k4 + kk) * SM_T + 32 + 4 * tx);
          b[0][kk] = v0.x; b[1][kk] = v0.y; b[2][kk] = v0.z; b[3][kk] = v0.w;
          b[4][kk] = v1.x; b[5][kk] = v1.y; b[6][kk] = v1.z; b[7][kk] = v1.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int n = (j < 4 ? 0 : 28) + 4 * tx + j;  // 4tx + j, then 32 + 4tx + j - 4; (n / 4) % 8 == tx
          const float4 v = lds4(Bs + n * SM_T + 4 * (k4 ^ tx));
          b[j][0] = v.x; b[j][1] = v.y; b[j][2] = v.z; b[j][3] = v.w;
        }
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 ai = make_float2(a[i][kk], a[i][kk]);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            acc[i][j] = __ffma2_rn(ai, make_float2(b[2 * j][kk], b[2 * j + 1][kk]), acc[i][j]);
        }
    }
    // fold the chunk's partial sums (round-to-nearest adds)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mst[i][j] = __fadd2_rn(mst[i][j], acc[i][j]);
        acc[i][j] = make_float2(0.0f, 0.0f);
      }

    if ((it + 1) % chunks == 0) {
      // ---- last chunk of the product: C = alpha * sum + beta * C (C not read when
      // beta == 0); a warp stores 128 contiguous bytes of each of 4 rows per instruction
      const int64_t prod = (int64_t)blockIdx.x + (int64_t)(it / chunks) * gridDim.x;
      float* Cp = p.C + prod * p.stride_c;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int row = 4 * ty + i;
        if (row < p.M) {
          float* crow = Cp + (int64_t)row * p.ldc;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int col = 32 * q + 4 * tx;
            const float v[4] = {mst[i][2 * q].x, mst[i][2 * q].y, mst[i][2 * q + 1].x, mst[i][2 * q + 1].y};
            if (p.c_vec && col + 3 < p.N) {
              float4* cp = reinterpret_cast<float4*>(crow + col);
              if (p.beta == 0.0f) {
                *cp = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
              } else {
                const float4 c = *cp;
                *cp = make_float4(fmaf(p.alpha, v[0], p.beta * c.x), fmaf(p.alpha, v[1], p.beta * c.y),
                                  fmaf(p.alpha, v[2], p.beta * c.z), fmaf(p.alpha, v[3], p.beta * c.w));
              }
            } else {
#pragma unroll
              for (int h = 0; h < 4; ++h)
                if (col + h < p.N)
                  crow[col + h] = p.beta == 0.0f ? p.alpha * v[h] : fmaf(p.alpha, v[h], p.beta * crow[col + h]);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) mst[i][j] = make_float2(0.0f, 0.0f);
      }
    }
    __syncthreads();  // every thread is done with this stage before it is refilled
  }
}

template <bool TA, bool TB>
cudaError_t launch_one(const GemmParams& p, int grid, cudaStream_t stream) {
  small_gemm_kernel<TA, TB><<<(unsigned)grid, SM_THREADS, SM_SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <bool TA, bool TB>
cudaError_t allow_smem() {
  return cudaFuncSetAttribute(small_gemm_kernel<TA, TB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SM_SMEM_BYTES);
}

}  // namespace

cudaError_t prepare_small_gemm() {
  cudaError_t e = allow_smem<false, false>();
  if (e == cudaSuccess) e = allow_smem<false, true>();
  if (e == cudaSuccess) e = allow_smem<true, false>();
  if (e == cudaSuccess) e = allow_smem<true, true>();
  return e;
}

cudaError_t launch_small_gemm(bool transA, bool transB, const GemmParams& p, int grid, cudaStream_t stream) {
  if (grid < 1 || grid > p.batch) return cudaErrorInvalidValue;
  if (!transA && !transB) return launch_one<false, false>(p, grid, stream);
  if (!transA && transB) return launch_one<false, true>(p, grid, stream);
  if (transA && !transB) return launch_one<true, false>(p, grid, stream);
  return launch_one<true, true>(p, grid, stream);
}

}  // namespace sgemm_impl
