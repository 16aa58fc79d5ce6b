// kernel_generic.cu -- SGEMM kernel for operands of any alignment and leading
// dimension (the edge path): 128x128x16 tiles, 256 threads, 8x8 results per
// thread, operands copied element by element with cp.async (4 bytes each: any
// address is aligned for them) into a double-buffered shared-memory tile, so
// the next K tile's copies run while the current one's FMAs issue.
//
// Edge handling follows the zero-fill reading of the shared-memory kernel in
// klklkl10086.github.io "Sgemm单精度矩阵乘法" (更优雅的实现): elements outside
// op(A) or op(B) are filled with 0 by the copy itself (source size 0), so
// ragged M, N and K need no special case in the inner loop, and only in-range
// elements of C are written.  Both operands are stored in shared memory as
// [k][m] / [k][n] rows whatever their layout in memory (each 4-byte copy
// picks its own destination), so a thread reads its 8 rows and 8 columns of
// a k with four 128-bit loads and runs 32 packed fma.rn.f32x2.
#include "bounds.cuh"
#include "device_utils.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

constexpr int GBM = 128, GBN = 128, GBK = 16, GTHREADS = 256, GPAD = 4;
// Partial sums are folded into a second accumulator every GFLUSH K tiles, so
// no float accumulator ever sums more than GFLUSH*GBK = 128 products.
constexpr int GFLUSH = 8;
constexpr int kCopies = GBM * GBK / GTHREADS;  // elements of each operand a thread copies per K tile
static_assert(GBM == GBN && kCopies == 8, "the copy mapping below assumes 128 x 16 operand tiles");

__device__ __forceinline__ float epilogue(float alpha, float beta, float v, const float* c) {
  return beta == 0.0f ? alpha * v : fmaf(alpha, v, beta * *c);
}

// 4-byte asynchronous copy global -> shared; `ok` false fills the destination with 0 and reads
// nothing (source size 0; the source is then any valid address).
__device__ __forceinline__ void cp_async4(uint32_t dst, const float* src, bool ok) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(ok ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <bool TA, bool TB, bool SPLIT>
__global__ void __launch_bounds__(GTHREADS) generic_gemm_kernel(const GemmParams p) {
  __shared__ __align__(16) float As[2][GBK][GBM + GPAD];  // [k][m]
  __shared__ __align__(16) float Bs[2][GBK][GBN + GPAD];  // [k][n]

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int tiles = p.tiles_m * p.tiles_n;
  const int prod = (int)(blockIdx.x / (unsigned)tiles);  // product of a strided batch
  const int tile = (int)(blockIdx.x - (unsigned)(prod * tiles));
  const int tm = tile / p.tiles_n, tn = tile % p.tiles_n;
  const float* __restrict__ Ab = p.A + (int64_t)prod * p.stride_a;
  const float* __restrict__ Bb = p.B + (int64_t)prod * p.stride_b;
  const int m0 = tm * GBM, n0 = tn * GBN;
  const int kt_total = (p.K + GBK - 1) / GBK;
  const int kt0 = blockIdx.y * p.k_tiles_per_split;
  const int kt1 = min(kt_total, kt0 + p.k_tiles_per_split);

  // Copies of K tile kt into stage `buf`: consecutive threads walk the operand's contiguous axis.
  auto copy_tile = [&](int kt, int buf) {
    const int k0 = kt * GBK;
#pragma unroll
    for (int r = 0; r < kCopies; ++r) {
      int mm, kk;
      if (!TA) { kk = tid & 15; mm = (tid >> 4) + 16 * r; }   // K contiguous: 16 k of a row
      else     { mm = tid & 127; kk = (tid >> 7) + 2 * r; }   // M contiguous: 128 m of a k
      const int gm = m0 + mm, gk = k0 + kk;
      const int64_t ai = TA ? (int64_t)gk * p.lda + gm : (int64_t)gm * p.lda + gk;
      const bool aok = gm < p.M && gk < p.K && a_ok(p, (int64_t)prod * p.stride_a + ai, 1);
      cp_async4(smem_addr(&As[buf][kk][mm]), aok ? Ab + ai : p.A, aok);
      int nn;
      if (!TB) { nn = tid & 127; kk = (tid >> 7) + 2 * r; }   // N contiguous: 128 n of a k
      else     { kk = tid & 15; nn = (tid >> 4) + 16 * r; }   // K contiguous: 16 k of a column
      const int gn = n0 + nn, gk2 = k0 + kk;
      const int64_t bi = TB ? (int64_t)gn * p.ldb + gk2 : (int64_t)gk2 * p.ldb + gn;
      const bool bok = gn < p.N && gk2 < p.K && b_ok(p, (int64_t)prod * p.stride_b + bi, 1);
      cp_async4(smem_addr(&Bs[buf][kk][nn]), bok ? Bb + bi : p.B, bok);
    }
    cp_async_commit();
  };

  // this thread's results: rows 4ty + (0..3) and 64 + 4ty + (0..3), columns 4tx + (0..3) and
  // 64 + 4tx + (0..3); acc[i][j2] holds columns 2 j2, 2 j2 + 1 of that list
  float2 acc[8][4], mst[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = mst[i][j] = make_float2(0.0f, 0.0f);

  if (kt0 < kt1) copy_tile(kt0, 0);
  for (int kt = kt0; kt < kt1; ++kt) {
    const int buf = (kt - kt0) & 1;
    if (kt + 1 < kt1) {
      copy_tile(kt + 1, buf ^ 1);  // the next tile's copies overlap this tile's math
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < GBK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][k][4 * ty]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][k][64 + 4 * ty]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][k][4 * tx]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][k][64 + 4 * tx]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float2 b[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                           make_float2(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(make_float2(a[i], a[i]), b[j], acc[i][j]);
    }
    __syncthreads();  // every thread is done with `buf` before the next iteration refills it
    if ((kt - kt0) % GFLUSH == GFLUSH - 1) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mst[i][j] = __fadd2_rn(mst[i][j], acc[i][j]);
          acc[i][j] = make_float2(0.0f, 0.0f);
        }
    }
  }

#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = m0 + (i < 4 ? 4 * ty + i : 64 + 4 * ty + i - 4);
    if (row >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int col = n0 + (j < 4 ? 4 * tx + j : 64 + 4 * tx + j - 4);
      if (col >= p.N) continue;
      const float2 s = __fadd2_rn(mst[i][j >> 1], acc[i][j >> 1]);
      const float v = (j & 1) ? s.y : s.x;
      if (SPLIT) {
        const int64_t wi = (((int64_t)prod * gridDim.y + blockIdx.y) * p.M + row) * p.ws_ld + col;
        if (ws_ok(p, wi, 1)) p.ws[wi] = v;
      } else {
        const int64_t ci = (int64_t)prod * p.stride_c + (int64_t)row * p.ldc + col;
        if (c_ok(p, ci, 1)) p.C[ci] = epilogue(p.alpha, p.beta, v, p.C + ci);
      }
    }
  }
}

template <bool TA, bool TB>
cudaError_t launch_one(const GemmParams& p, int split, cudaStream_t stream) {
  dim3 grid((unsigned)((int64_t)p.batch * p.tiles_m * p.tiles_n), (unsigned)split);
  if (split > 1)
    generic_gemm_kernel<TA, TB, true><<<grid, GTHREADS, 0, stream>>>(p);
  else
    generic_gemm_kernel<TA, TB, false><<<grid, GTHREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

GenericTileShape generic_tile_shape() { return {GBM, GBN, GBK, GTHREADS}; }

cudaError_t launch_generic_gemm(bool transA, bool transB, const GemmParams& p, int split,
                                cudaStream_t stream) {
  if (!transA && !transB) return launch_one<false, false>(p, split, stream);
  if (!transA && transB) return launch_one<false, true>(p, split, stream);
  if (transA && !transB) return launch_one<true, false>(p, split, stream);
  return launch_one<true, true>(p, split, stream);
}

}  // namespace sgemm_impl
