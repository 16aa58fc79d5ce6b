// kernel_generic.cu -- SGEMM kernel for operands of any alignment and leading
// dimension (the edge path): 64x64x16 tiles, 256 threads, 4x4 results per
// thread, predicated zero-filling global loads staged through registers into a
// double-buffered shared-memory tile.
//
// Edge handling follows the zero-fill reading of the shared-memory kernel in
// klklkl10086.github.io "Sgemm单精度矩阵乘法" (更优雅的实现): elements outside
// op(A) or op(B) load as 0, so ragged M, N and K need no special case in the
// inner loop, and only in-range elements of C are written.
#include "bounds.cuh"
#include "device_utils.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

constexpr int GBM = 64, GBN = 64, GBK = 16, GTHREADS = 256, GPAD = 4;
// Partial sums are folded into a second accumulator every GFLUSH K tiles, so
// no float accumulator ever sums more than GFLUSH*GBK = 128 products.
constexpr int GFLUSH = 8;

__device__ __forceinline__ float epilogue(float alpha, float beta, float v, const float* c) {
  return beta == 0.0f ? alpha * v : fmaf(alpha, v, beta * *c);
}

template <bool TA, bool TB, bool SPLIT>
__global__ void __launch_bounds__(GTHREADS) generic_gemm_kernel(const GemmParams p) {
  __shared__ float As[2][GBK][GBM + GPAD];  // [k][m]
  __shared__ float Bs[2][GBK][GBN + GPAD];  // [k][n]

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

  float ra[4], rb[4];
  auto load = [&](int kt) {
    const int k0 = kt * GBK;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      int mm, kk;
      if (!TA) { kk = tid & 15; mm = (tid >> 4) + 16 * r; }   // consecutive threads walk k
      else     { mm = tid & 63; kk = (tid >> 6) + 4 * r; }    // consecutive threads walk m
      const int gm = m0 + mm, gk = k0 + kk;
      const int64_t ai = TA ? (int64_t)gk * p.lda + gm : (int64_t)gm * p.lda + gk;
      ra[r] = (gm < p.M && gk < p.K && a_ok(p, (int64_t)prod * p.stride_a + ai, 1)) ? Ab[ai] : 0.0f;
      int nn;
      if (!TB) { nn = tid & 63; kk = (tid >> 6) + 4 * r; }
      else     { kk = tid & 15; nn = (tid >> 4) + 16 * r; }
      const int gn = n0 + nn, gk2 = k0 + kk;
      const int64_t bi = TB ? (int64_t)gn * p.ldb + gk2 : (int64_t)gk2 * p.ldb + gn;
      rb[r] = (gn < p.N && gk2 < p.K && b_ok(p, (int64_t)prod * p.stride_b + bi, 1)) ? Bb[bi] : 0.0f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (!TA) As[buf][tid & 15][(tid >> 4) + 16 * r] = ra[r];
      else     As[buf][(tid >> 6) + 4 * r][tid & 63] = ra[r];
      if (!TB) Bs[buf][(tid >> 6) + 4 * r][tid & 63] = rb[r];
      else     Bs[buf][tid & 15][(tid >> 4) + 16 * r] = rb[r];
    }
  };

  float acc[4][4], mst[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = mst[i][j] = 0.0f;

  if (kt0 < kt1) {
    load(kt0);
    store(0);
  }
  __syncthreads();
  for (int kt = kt0; kt < kt1; ++kt) {
    const int buf = (kt - kt0) & 1;
    if (kt + 1 < kt1) load(kt + 1);  // next tile's global loads overlap this tile's math
#pragma unroll
    for (int k = 0; k < GBK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[buf][k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[buf][k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    if (kt + 1 < kt1) store(buf ^ 1);
    __syncthreads();
    if ((kt - kt0) % GFLUSH == GFLUSH - 1) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          mst[i][j] += acc[i][j];
          acc[i][j] = 0.0f;
        }
    }
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = m0 + ty + 16 * i;
    if (row >= p.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = n0 + tx + 16 * j;
      if (col >= p.N) continue;
      const float v = mst[i][j] + acc[i][j];
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
