// kernel_small.cu -- many small products (M <= 64, N <= 64; a strided batch of
// them): one CTA computes a product's whole 64x64 output tile, then moves on
// to the next product, whose copies are already in flight.
//
// For such products the tensor-core kernel's 128x128 tile is three quarters
// padding, and its pipeline (TMA ring, split, MMA issue, fold) is set up for
// long K loops.  Here the work of a CTA is a list of (product, 32-k chunk)
// items; each item's op(A) and op(B) chunks (8 KB each) are copied into one
// of two shared-memory stages with 16-byte cp.async copies, in the operands'
// stored orientation, and the next item's copies are issued before the
// current item is computed.  Two warps share the tile, 32 rows each; a
// thread accumulates an 8x8 block with packed FP32 FMAs (fma.rn.f32x2, IEEE
// round-to-nearest, k ascending), so each 128-bit shared load feeds 16 FMAs,
// and loads the fragments of the next group of 4 k while the current group's
// FMAs issue.  The grid is persistent (four CTAs per SM, products dealt
// round-robin), so HBM traffic and FMA work overlap within a CTA and across
// the CTAs of an SM.
//
// Shared layout of a stage: the A chunk, then the B chunk.  An operand stored
// K-contiguous (A 'N' as [m][k], B 'T' as [n][k]) is kept as 64 rows of 32
// floats with 16-byte group g of row r at g XOR (r % 8); one stored
// M/N-contiguous (A 'T' as [k][m], B 'N' as [k][n]) as 32 rows of 64 floats.
// The thread-to-row and thread-to-column maps depend on the orientation so
// that every shared load of a warp touches distinct banks (rows 4 apart for a
// K-contiguous A, 4 adjacent rows otherwise; columns 8 apart for a
// K-contiguous B, 4 adjacent columns otherwise).
//
// Requirements (checked by the planner): A, B 16-byte aligned, lda, ldb and
// the batch strides multiples of 4 floats, and the extent copied along a row
// a multiple of 4: K for op(A) 'N' and op(B) 'T', M for op(A) 'T', N for
// op(B) 'N'.  Groups outside the matrix are zero-filled, never read.
#include <cstdint>

#include "bounds.cuh"
#include "kernel_small.h"

namespace sgemm_impl {
namespace {

constexpr int SM_T = 64;                              // output tile
constexpr int SM_KC = 32;                             // K chunk
constexpr int SM_THREADS = 64;                        // 2 warps, 8x8 results per thread
constexpr int SM_CTAS = 4;                            // CTAs per SM
constexpr int SM_CHUNK_FLOATS = SM_T * SM_KC;         // one operand chunk (8 KB)
constexpr int SM_STAGE_FLOATS = 2 * SM_CHUNK_FLOATS;  // A chunk + B chunk
constexpr int SM_SMEM_BYTES = 2 * SM_STAGE_FLOATS * 4;
static_assert(SM_SMEM_BYTES == 32768, "two 16 KB stages");
static_assert(SM_CTAS * (SM_SMEM_BYTES + 1024) <= 228 * 1024, "CTAs per SM");

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

// One operand chunk stored K-contiguous: 64 rows (matrix rows 0..63, valid
// below `rows`) of 8 groups (columns k0 + 4g, valid below K), swizzled.
// (chk: the bounds check of the debug build on the operand, `off` the chunk base's element offset)
template <class Chk>
__device__ __forceinline__ void copy_k_rows(float* dst, const float* base, int64_t ld, int rows, int k0, int K,
                                            int tid, const Chk& chk, int64_t off) {
  const uint32_t d0 = smem_addr(dst);
#pragma unroll
  for (int q = 0; q < SM_CHUNK_FLOATS / 4 / SM_THREADS; ++q) {
    const int e = tid + SM_THREADS * q;  // 0 .. 511
    const int r = e >> 3, g = e & 7;
    const int col = k0 + 4 * g;
    const bool ok = r < rows && col < K && chk(off + (int64_t)r * ld + col, 4);
    cp_async16(d0 + (uint32_t)((r * SM_KC + 4 * (g ^ (r & 7))) * 4), ok ? base + (int64_t)r * ld + col : base,
               ok ? 16 : 0);
  }
}

// One operand chunk stored M/N-contiguous: 32 rows (matrix rows k0 .. k0+31,
// valid below K) of 16 groups (columns 4g, valid below `cols`), unswizzled.
template <class Chk>
__device__ __forceinline__ void copy_mn_rows(float* dst, const float* base, int64_t ld, int cols, int k0, int K,
                                             int tid, const Chk& chk, int64_t off) {
  const uint32_t d0 = smem_addr(dst);
#pragma unroll
  for (int q = 0; q < SM_CHUNK_FLOATS / 4 / SM_THREADS; ++q) {
    const int e = tid + SM_THREADS * q;
    const int r = e >> 4, g = e & 15;
    const int row = k0 + r;
    const bool ok = row < K && 4 * g < cols && chk(off + (int64_t)row * ld + 4 * g, 4);
    cp_async16(d0 + (uint32_t)((r * SM_T + 4 * g) * 4), ok ? base + (int64_t)row * ld + 4 * g : base, ok ? 16 : 0);
  }
}

// Tile row of the thread's i-th accumulator row, tile column of its j-th column.
template <bool TA>
__device__ __forceinline__ int row_of(int i, int wm, int ty) {
  return TA ? 32 * wm + 16 * (i >> 2) + 4 * ty + (i & 3) : 32 * wm + ty + 4 * i;
}
template <bool TB>
__device__ __forceinline__ int col_of(int j, int tx) {
  return TB ? tx + 8 * j : 32 * (j >> 2) + 4 * tx + (j & 3);
}

// Fragments of group g (k 4g .. 4g+3 of the chunk) for the thread's 8 rows and 8 columns.
template <bool TA, bool TB>
__device__ __forceinline__ void load_group(const float* As, const float* Bs, int g, int wm, int ty, int tx,
                                           const int (&a_off)[2], const int (&b_off)[8], float (&a)[4][8],
                                           float (&b)[4][8]) {
  if (!TA) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = row_of<TA>(i, wm, ty);
      const float4 v = lds4(As + r * SM_KC + 4 * (g ^ (r & 7)));
      a[0][i] = v.x; a[1][i] = v.y; a[2][i] = v.z; a[3][i] = v.w;
    }
  } else {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 v = lds4(As + (4 * g + kk) * SM_T + a_off[h]);
        a[kk][4 * h] = v.x; a[kk][4 * h + 1] = v.y; a[kk][4 * h + 2] = v.z; a[kk][4 * h + 3] = v.w;
      }
  }
  if (!TB) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 v = lds4(Bs + (4 * g + kk) * SM_T + b_off[4 * h]);
        b[kk][4 * h] = v.x; b[kk][4 * h + 1] = v.y; b[kk][4 * h + 2] = v.z; b[kk][4 * h + 3] = v.w;
      }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v = lds4(Bs + b_off[j] + 4 * (g ^ tx));  // row tx + 8j: (row % 8) == tx
      b[0][j] = v.x; b[1][j] = v.y; b[2][j] = v.z; b[3][j] = v.w;
    }
  }
}

// 4 rank-1 updates of the thread's 8x8 block, k ascending.
__device__ __forceinline__ void fma_group(const float (&a)[4][8], const float (&b)[4][8], float2 (&acc)[8][4]) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 ai = make_float2(a[kk][i], a[kk][i]);
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][q] = __ffma2_rn(ai, make_float2(b[kk][2 * q], b[kk][2 * q + 1]), acc[i][q]);
    }
}

template <bool TA, bool TB>
__global__ void __launch_bounds__(SM_THREADS, SM_CTAS) small_gemm_kernel(const GemmParams p) {
  extern __shared__ __align__(16) float smem[];
  const int tid = threadIdx.x;
  const int wm = tid >> 5, lane = tid & 31;
  const int ty = lane >> 3, tx = lane & 7;
  const int chunks = (p.K + SM_KC - 1) / SM_KC;
  // items of this CTA: products blockIdx.x, blockIdx.x + gridDim.x, ..., `chunks` K chunks each
  const int my_products = (p.batch - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  const int items = my_products * chunks;

  const auto issue = [&](int item) {
    const int64_t prod = (int64_t)blockIdx.x + (int64_t)(item / chunks) * gridDim.x;
    const int k0 = (item % chunks) * SM_KC;
    float* st = smem + (item & 1) * SM_STAGE_FLOATS;
    const float* A = p.A + prod * p.stride_a;
    const float* B = p.B + prod * p.stride_b;
    const auto achk = [&](int64_t o, int64_t n) { return a_ok(p, o, n); };
    const auto bchk = [&](int64_t o, int64_t n) { return b_ok(p, o, n); };
    if (!TA) copy_k_rows(st, A, p.lda, p.M, k0, p.K, tid, achk, prod * p.stride_a);
    else copy_mn_rows(st, A, p.lda, p.M, k0, p.K, tid, achk, prod * p.stride_a);
    if (!TB) copy_mn_rows(st + SM_CHUNK_FLOATS, B, p.ldb, p.N, k0, p.K, tid, bchk, prod * p.stride_b);
    else copy_k_rows(st + SM_CHUNK_FLOATS, B, p.ldb, p.N, k0, p.K, tid, bchk, prod * p.stride_b);
  };

  // per-thread float offsets of the M/N-contiguous fragments (first column of 4) and of the
  // K-contiguous B rows
  int a_off[2], b_off[8];
#pragma unroll
  for (int h = 0; h < 2; ++h) a_off[h] = row_of<TA>(4 * h, wm, ty);
#pragma unroll
  for (int j = 0; j < 8; ++j) b_off[j] = TB ? col_of<TB>(j, tx) * SM_KC : col_of<TB>(j, tx);

  float2 acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

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
    // fragments of group g + 1 are loaded while group g's FMAs issue
    float a[2][4][8], b[2][4][8];  // a[.][kk][i] = op(A)(row i, 4g + kk), b[.][kk][j] = op(B)(4g + kk, column j)
    load_group<TA, TB>(As, Bs, 0, wm, ty, tx, a_off, b_off, a[0], b[0]);
#pragma unroll
    for (int g = 0; g < SM_KC / 4; ++g) {
      if (g + 1 < SM_KC / 4) load_group<TA, TB>(As, Bs, g + 1, wm, ty, tx, a_off, b_off, a[(g + 1) & 1], b[(g + 1) & 1]);
      fma_group(a[g & 1], b[g & 1], acc);
    }

    if ((it + 1) % chunks == 0) {
      // ---- last chunk of the product: C = alpha * sum + beta * C (C not read when beta == 0)
      const int64_t prod = (int64_t)blockIdx.x + (int64_t)(it / chunks) * gridDim.x;
      float* Cp = p.C + prod * p.stride_c;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = row_of<TA>(i, wm, ty);
        if (row < p.M) {
          const int64_t roff = prod * p.stride_c + (int64_t)row * p.ldc;
          float* crow = Cp + (int64_t)row * p.ldc;
          const float v[8] = {acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y,
                              acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y};
          if (!TB) {
            // columns 4tx .. +3 and 32 + 4tx .. +3: a warp stores 128 contiguous bytes per row
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int col = 32 * h + 4 * tx;
              if (col >= p.N || !c_ok(p, roff + col, min(4, p.N - col))) continue;
              if (p.c_vec && col + 3 < p.N) {
                float4* cp = reinterpret_cast<float4*>(crow + col);
                if (p.beta == 0.0f) {
                  *cp = make_float4(p.alpha * v[4 * h], p.alpha * v[4 * h + 1], p.alpha * v[4 * h + 2],
                                    p.alpha * v[4 * h + 3]);
                } else {
                  const float4 c = *cp;
                  *cp = make_float4(fmaf(p.alpha, v[4 * h], p.beta * c.x), fmaf(p.alpha, v[4 * h + 1], p.beta * c.y),
                                    fmaf(p.alpha, v[4 * h + 2], p.beta * c.z),
                                    fmaf(p.alpha, v[4 * h + 3], p.beta * c.w));
                }
              } else {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (col + e < p.N)
                    crow[col + e] = p.beta == 0.0f ? p.alpha * v[4 * h + e]
                                                   : fmaf(p.alpha, v[4 * h + e], p.beta * crow[col + e]);
              }
            }
          } else {
            // columns tx + 8j: a warp stores 32 contiguous bytes of 4 rows per instruction
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const int col = tx + 8 * j;
              if (col < p.N && c_ok(p, roff + col, 1))
                crow[col] = p.beta == 0.0f ? p.alpha * v[j] : fmaf(p.alpha, v[j], p.beta * crow[col]);
            }
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.0f, 0.0f);
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
