// kernel_small.cu -- many small products (M <= 64, N <= 64; a strided batch of
// them): one CTA per product computes the whole 64x64 output tile.
//
// For such products the tensor-core kernel's 128x128 tile is three quarters
// padding, and its pipeline (TMA ring, split, MMA issue, fold) is set up for
// long K loops; here a CTA stages 64-k chunks of op(A) and op(B) in shared
// memory with 128-bit loads, and 128 threads each accumulate a 4x8 block with
// packed FP32 FMAs (fma.rn.f32x2, IEEE round-to-nearest).  A chunk's partial
// sums are added into a second set of registers after every chunk, so no
// accumulator sums more than 64 products.  Several CTAs share an SM, so one
// CTA's loads overlap another's arithmetic.
//
// Requirements (checked by the planner): A, B 16-byte aligned, lda, ldb and
// the batch strides multiples of 4 floats, and the extent read along a row
// with 128-bit loads a multiple of 4: K for op(A) 'N' and op(B) 'T', M for
// op(A) 'T', N for op(B) 'N'.
#include "kernel_small.h"

namespace sgemm_impl {
namespace {

constexpr int SM_T = 64;           // output tile and K chunk
constexpr int SM_THREADS = 128;    // 16 x 8 threads, 4 rows x 8 columns each

__device__ __forceinline__ float4 ld4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }

// Shared tiles are [k][64 columns]; column c of row k is stored at c XOR 4*((k/4) % 8).  The XOR
// keeps each aligned group of 4 columns together (128-bit reads and writes stay whole) and spreads
// the transposing scalar stores (16 k of one column per warp) over 8 bank groups instead of 1.
__device__ __forceinline__ int swz(int k, int c) { return c ^ (((k >> 2) & 7) << 2); }

template <bool TA, bool TB>
__global__ void __launch_bounds__(SM_THREADS) small_gemm_kernel(const GemmParams p) {
  __shared__ __align__(16) float As[SM_T][SM_T];  // [k][m], swizzled columns
  __shared__ __align__(16) float Bs[SM_T][SM_T];  // [k][n], swizzled columns
  const int tid = threadIdx.x;
  const int ty = tid >> 3, tx = tid & 7;  // rows 4ty .. +3, columns 4tx .. +3 and 32 + 4tx .. +3
  const int64_t prod = blockIdx.x;
  const float* __restrict__ A = p.A + prod * p.stride_a;
  const float* __restrict__ B = p.B + prod * p.stride_b;

  float2 acc[4][4], mst[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = mst[i][j] = make_float2(0.0f, 0.0f);

  for (int k0 = 0; k0 < p.K; k0 += SM_T) {
    // ---- stage op(A)[0:64, k0:k0+64] as As[k][m] and op(B)[k0:k0+64, 0:64] as Bs[k][n], zero-filled
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int e = tid + SM_THREADS * r;  // 0 .. 1023: one float4 each
      if (!TA) {
        // stored M x K: a float4 along k of row m, transposed into As
        const int m = e >> 4, kq = (e & 15) * 4, k = k0 + kq;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m < p.M && k < p.K) v = ld4(A + (int64_t)m * p.lda + k);
        As[kq + 0][swz(kq + 0, m)] = v.x; As[kq + 1][swz(kq + 1, m)] = v.y;
        As[kq + 2][swz(kq + 2, m)] = v.z; As[kq + 3][swz(kq + 3, m)] = v.w;
      } else {
        // stored K x M: a float4 along m of row k
        const int kk = e >> 4, mq = (e & 15) * 4, k = k0 + kk;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < p.K && mq < p.M) v = ld4(A + (int64_t)k * p.lda + mq);
        *reinterpret_cast<float4*>(&As[kk][swz(kk, mq)]) = v;
      }
      if (!TB) {
        // stored K x N: a float4 along n of row k
        const int kk = e >> 4, nq = (e & 15) * 4, k = k0 + kk;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < p.K && nq < p.N) v = ld4(B + (int64_t)k * p.ldb + nq);
        *reinterpret_cast<float4*>(&Bs[kk][swz(kk, nq)]) = v;
      } else {
        // stored N x K: a float4 along k of row n, transposed into Bs
        const int n = e >> 4, kq = (e & 15) * 4, k = k0 + kq;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n < p.N && k < p.K) v = ld4(B + (int64_t)n * p.ldb + k);
        Bs[kq + 0][swz(kq + 0, n)] = v.x; Bs[kq + 1][swz(kq + 1, n)] = v.y;
        Bs[kq + 2][swz(kq + 2, n)] = v.z; Bs[kq + 3][swz(kq + 3, n)] = v.w;
      }
    }
    __syncthreads();
    // ---- 64 rank-1 updates of the thread's 4 x 8 block (column pairs packed)
#pragma unroll 8
    for (int k = 0; k < SM_T; ++k) {
      const float4 a = *reinterpret_cast<const float4*>(&As[k][swz(k, 4 * ty)]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[k][swz(k, 4 * tx)]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[k][swz(k, 32 + 4 * tx)]);
      const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                            make_float2(b1.z, b1.w)};
      const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 ai = make_float2(av[i], av[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(ai, bp[j], acc[i][j]);
      }
    }
    // fold the chunk's partial sums (round-to-nearest adds), then reuse the stage
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        mst[i][j] = __fadd2_rn(mst[i][j], acc[i][j]);
        acc[i][j] = make_float2(0.0f, 0.0f);
      }
    __syncthreads();
  }

  // ---- epilogue: C = alpha * sum + beta * C (C not read when beta == 0); a warp stores 128
  // contiguous bytes of each of 4 rows per instruction
  float* Cp = p.C + prod * p.stride_c;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = 4 * ty + i;
    if (row >= p.M) continue;
    float* crow = Cp + (int64_t)row * p.ldc;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int col = 32 * q + 4 * tx;
      float v[4] = {mst[i][2 * q].x, mst[i][2 * q].y, mst[i][2 * q + 1].x, mst[i][2 * q + 1].y};
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
}

template <bool TA, bool TB>
cudaError_t launch_one(const GemmParams& p, cudaStream_t stream) {
  small_gemm_kernel<TA, TB><<<(unsigned)p.batch, SM_THREADS, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_small_gemm(bool transA, bool transB, const GemmParams& p, cudaStream_t stream) {
  if (!transA && !transB) return launch_one<false, false>(p, stream);
  if (!transA && transB) return launch_one<false, true>(p, stream);
  if (transA && !transB) return launch_one<true, false>(p, stream);
  return launch_one<true, true>(p, stream);
}

}  // namespace sgemm_impl
