// kernel_tma.cuh -- the main SGEMM kernel for sm_103a: a SIMT FFMA kernel fed
// by a TMA + mbarrier shared-memory ring.
//
// Structure (one CTA per output tile, 8 warps, 256 threads):
//   * thread 0 also acts as the producer: it issues 2-D TMA tile loads of
//     op(A) and op(B) for K tile t into stage t % kStages.  A stage is refilled
//     one iteration after it was consumed, once all 256 threads released it
//     ("empty" mbarrier), so loads run kStages-1 tiles ahead.  The copy engine
//     zero-fills any part of a box outside the matrix, which gives ragged M,
//     N and K for free.  (A separate producer warp would put 3 warps on one
//     SM sub-partition and cap every thread at 168 registers.)
//   * all threads wait for a stage ("full" mbarrier), run the register outer
//     products out of shared memory and release the stage.  Shared-memory
//     fragments are double-buffered in registers: the loads of k-group g+1
//     (across a stage boundary, the next tile's first group) issue while
//     group g's FMAs run, so the two warps of an SM sub-partition do not
//     stall together on shared-memory latency.
//   * each thread owns an 8x8 block of C (warp tile 32x64) and accumulates
//     with packed fma.rn.f32x2 (two IEEE fp32 FMAs per issue, a broadcast
//     A value times a pair of adjacent B values).
//   * every kFlushTiles K tiles the register sums are folded into running
//     sums kept in tensor memory (TMEM, otherwise unused by this SIMT kernel),
//     so no float accumulator adds more than 128 products; this keeps the
//     relative Frobenius error near 3e-7 at K = 4096 instead of the ~1.2e-6 a
//     single accumulator over all of K gives, and costs no registers.
//   * every bounded wait is voted across the warp, so a warp leaves the loop
//     as a whole and the warp-collective TMEM instructions stay converged.
//   * epilogue C = alpha*acc + beta*C fused, 128-bit where C allows it; C is
//     not read when beta == 0.  With a K split, the raw partial sums go to a
//     workspace instead and a reduction kernel applies the epilogue.
//
// Shared-memory tiles (per stage):
//   op(A) 'N' (K contiguous): [BM rows][32 floats], TMA 128-byte swizzle: the
//       16-byte chunk c of row r sits at chunk c ^ (r & 7), so the 8 rows a
//       warp reads in one 128-bit load hit 8 different bank groups.
//   op(A) 'T' (M contiguous): [32 k][BM floats], no swizzle needed.
//   op(B) 'N' (N contiguous): [32 k][BN floats].
//   op(B) 'T' (K contiguous): [BN rows][32 floats], 128-byte swizzle.
// These replace the hand transposition of A and the +1 padding used against
// bank conflicts on the pages (itan.pw "CUDA NVIDIA 4090 高性能計算", §3.5 and
// §3.8; youngju.dev "CUDA architecture visualized", 共有メモリのバンクコンフリクト):
// the TMA engine cannot transpose 4-byte elements, so each layout is read
// along its contiguous axis instead.
#pragma once

#include "bounds.cuh"
#include "device_utils.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace tma {

constexpr int kBK = 32;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers;
constexpr int kFlushTiles = 4;
constexpr uint32_t kTmemCols = 128;  // 2 warp columns x 64 running sums per thread
constexpr int kGroupM = 8;  // tile rows per raster group (L2 reuse of B)

template <int WM, int WN>
struct Tile {
  static_assert(WM * WN == kConsumerWarps, "8 consumer warps");
  static constexpr int BM = WM * 32;
  static constexpr int BN = WN * 64;
  static constexpr int A_BYTES = BM * kBK * 4;
  static constexpr int B_BYTES = BN * kBK * 4;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM_BYTES = kStages * STAGE_BYTES + 1024;  // + alignment slack
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzle atoms are 1024-byte aligned");
};

// Output tile of CTA `bid`: groups of kGroupM tile rows are walked column by
// column, so the CTAs resident at one time share a few B column panels.
__device__ __forceinline__ void tile_coords(int bid, int tiles_m, int tiles_n, int& tm, int& tn) {
  const int span = kGroupM * tiles_n;
  const int group = bid / span;
  const int first = group * kGroupM;
  const int rows = min(tiles_m - first, kGroupM);
  const int local = bid - group * span;
  tm = first + local % rows;
  tn = local / rows;
}

__device__ __forceinline__ float4 lds128(const uint8_t* base, uint32_t off) {
  return *reinterpret_cast<const float4*>(base + off);
}

__device__ __forceinline__ float2 ffma2(float a, float2 b, float2 c) {
  return __ffma2_rn(make_float2(a, a), b, c);
}

// Row (within the CTA tile) of the thread's i-th accumulator row.
template <bool TA>
__device__ __forceinline__ int row_of(int i, int wm, int ty) {
  return TA ? wm * 32 + 16 * (i >> 2) + 4 * ty + (i & 3)  // 2 groups of 4 adjacent rows
            : wm * 32 + ty + 4 * i;                        // rows ty, ty+4, ..., ty+28
}

// Column (within the CTA tile) of the thread's j-th accumulator column.
template <bool TB>
__device__ __forceinline__ int col_of(int j, int wn, int tx) {
  return TB ? wn * 64 + tx + 8 * j                         // columns tx, tx+8, ..., tx+56
            : wn * 64 + 32 * (j >> 2) + 4 * tx + (j & 3);  // 2 groups of 4 adjacent columns
}

// Per-thread byte offsets into a stage's tiles (see load_group).
struct Offsets {
  uint32_t xa_even, xa_odd;  // K-major A: rows of even / odd i, with their swizzle phase
  uint32_t xa_mn;            // M-major A
  uint32_t xb_k;             // K-major B
  uint32_t xb_mn;            // N-major B
};

// Fragments of one group of 4 k: a[kk][i] = op(A)(row_i, k), b[kk][j] = op(B)(k, col_j).
// Each operand takes 8 128-bit shared-memory loads per group, whatever its layout.
template <int WM, int WN, bool TA, bool TB>
__device__ __forceinline__ void load_group(const uint8_t* a_tile, const uint8_t* b_tile, int g, const Offsets& o,
                                           float (&a)[4][8], float (&b)[4][8]) {
  using T = Tile<WM, WN>;
  if (!TA) {
    // K-contiguous rows, 128-byte swizzle: one load = 4 k of one row.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t off = (((i & 1) ? o.xa_odd : o.xa_even) ^ (uint32_t)(g << 4)) + (uint32_t)(i >> 1) * 1024u;
      const float4 v = lds128(a_tile, off);
      a[0][i] = v.x; a[1][i] = v.y; a[2][i] = v.z; a[3][i] = v.w;
    }
  } else {
    // M-contiguous: one load = 4 adjacent rows at one k.
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 v = lds128(a_tile, o.xa_mn + (uint32_t)((4 * g + kk) * T::BM * 4 + h * 64));
        a[kk][4 * h + 0] = v.x; a[kk][4 * h + 1] = v.y; a[kk][4 * h + 2] = v.z; a[kk][4 * h + 3] = v.w;
      }
  }
  if (!TB) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 v = lds128(b_tile, o.xb_mn + (uint32_t)((4 * g + kk) * T::BN * 4 + h * 128));
        b[kk][4 * h + 0] = v.x; b[kk][4 * h + 1] = v.y; b[kk][4 * h + 2] = v.z; b[kk][4 * h + 3] = v.w;
      }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float4 v = lds128(b_tile, (o.xb_k ^ (uint32_t)(g << 4)) + (uint32_t)j * 1024u);
      b[0][j] = v.x; b[1][j] = v.y; b[2][j] = v.z; b[3][j] = v.w;
    }
  }
}

// 4 rank-1 updates of the 8x8 accumulator block: 128 packed FMAs, k ascending.
__device__ __forceinline__ void fma_group(const float (&a)[4][8], const float (&b)[4][8], float2 (&acc)[8][4]) {
#pragma unroll
  for (int kk = 0; kk < 4; ++kk)
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int p = 0; p < 4; ++p)
        acc[i][p] = ffma2(a[kk][i], make_float2(b[kk][2 * p], b[kk][2 * p + 1]), acc[i][p]);
}

// The thread's 64 running sums live in 64 consecutive TMEM columns of its own
// lane (warps 0-3: columns 0-63 of lanes 0-127; warps 4-7: columns 64-127).
// Element (i, 2p + h) of the 8x8 block is column 8i + 2p + h.
__device__ __forceinline__ void fold_into_tmem(uint32_t taddr, float2 (&acc)[8][4]) {
  float m[4][16];
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld16(taddr + 16u * c, m[c]);
  tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld_ready(m[c]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int i = 2 * c + (e >> 2), p = e & 3;
      m[c][2 * e] += acc[i][p].x;
      m[c][2 * e + 1] += acc[i][p].y;
      acc[i][p] = make_float2(0.0f, 0.0f);
    }
    tmem_st16(taddr + 16u * c, m[c]);
  }
  tmem_wait_st();
}

// C = alpha * v + beta * C for the thread's 8x8 block (v[8i + j] is row i,
// column j of the block), or the raw sums into this CTA's slice of the
// split-K workspace.  `cm` is this product's C, `wm_base` its workspace slice
// (both row 0).  C is not read when beta == 0; 128-bit accesses where the 4
// columns are in range and C allows it.
template <int WM, int WN, bool TA, bool TB, bool SPLIT>
__device__ __forceinline__ void epilogue(const GemmParams& p, float* cm, float* wm_base, int m0, int n0, int wm,
                                         int wn, int ty, int tx, const float (&v)[64]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = m0 + row_of<TA>(i, wm, ty);
    if (row >= p.M) continue;
    if (!TB) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int col = n0 + col_of<false>(4 * h, wn, tx);
        const float* x = &v[8 * i + 4 * h];
        if (SPLIT) {
          if (col < p.N) {
            float* w = wm_base + (int64_t)row * p.ws_ld + col;
            if (ws_ok(p, w - p.ws, 4)) *reinterpret_cast<float4*>(w) = make_float4(x[0], x[1], x[2], x[3]);
          }
          continue;
        }
        float* c = cm + (int64_t)row * p.ldc + col;
        if (col >= p.N || !c_ok(p, c - p.C, min(4, p.N - col))) continue;
        if (p.c_vec && col + 3 < p.N) {
          float4 o;
          if (p.beta == 0.0f) {
            o = make_float4(p.alpha * x[0], p.alpha * x[1], p.alpha * x[2], p.alpha * x[3]);
          } else {
            const float4 old = *reinterpret_cast<const float4*>(c);
            o = make_float4(fmaf(p.alpha, x[0], p.beta * old.x), fmaf(p.alpha, x[1], p.beta * old.y),
                            fmaf(p.alpha, x[2], p.beta * old.z), fmaf(p.alpha, x[3], p.beta * old.w));
          }
          *reinterpret_cast<float4*>(c) = o;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (col + q < p.N) c[q] = p.beta == 0.0f ? p.alpha * x[q] : fmaf(p.alpha, x[q], p.beta * c[q]);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int col = n0 + col_of<true>(j, wn, tx);
        if (col >= p.N) continue;
        const float x = v[8 * i + j];
        if (SPLIT) {
          float* w = wm_base + (int64_t)row * p.ws_ld + col;
          if (ws_ok(p, w - p.ws, 1)) *w = x;
        } else {
          float* c = cm + (int64_t)row * p.ldc + col;
          if (c_ok(p, c - p.C, 1)) *c = p.beta == 0.0f ? p.alpha * x : fmaf(p.alpha, x, p.beta * *c);
        }
      }
    }
  }
}

template <int WM, int WN, bool TA, bool TB, bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    tma_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const GemmParams p) {
  using T = Tile<WM, WN>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ uint32_t tmem_slot;

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  const uint8_t* smem = smem_raw + pad;  // 1024-byte aligned: 128-byte swizzle atoms
  const uint32_t sbase = raw + pad;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int tiles = p.tiles_m * p.tiles_n;
  const int prod = (int)(blockIdx.x / (unsigned)tiles);  // product of a strided batch
  int tm, tn;
  tile_coords((int)(blockIdx.x - (unsigned)(prod * tiles)), p.tiles_m, p.tiles_n, tm, tn);
  const int m0 = tm * T::BM;
  const int n0 = tn * T::BN;
  const int za = prod * p.za, zb = prod * p.zb;
  const int kt_total = (p.K + kBK - 1) / kBK;
  const int kt0 = blockIdx.y * p.k_tiles_per_split;
  const int nkt = min(kt_total, kt0 + p.k_tiles_per_split) - kt0;  // >= 1 by construction

  if (warp == 0) tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kConsumers);
    }
    fence_mbar_init();
  }
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t taddr = tmem_slot + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)(64 * (warp >> 2));

  // Producer side (thread 0): load K tile t into stage t % kStages.
  auto issue = [&](int t) {
    const int s = t % kStages;
    const uint32_t fb = smem_addr(&full_bar[s]);
    const uint32_t a_dst = sbase + (uint32_t)(s * T::STAGE_BYTES);
    const uint32_t b_dst = a_dst + (uint32_t)T::A_BYTES;
    const int k0 = (kt0 + t) * kBK;
    mbar_arrive_expect_tx(fb, (uint32_t)T::STAGE_BYTES);
    if (!TA) tma_load_3d(a_dst, &mapA, fb, k0, m0, za);
    else     tma_load_3d(a_dst, &mapA, fb, m0, k0, za);
    if (!TB) tma_load_3d(b_dst, &mapB, fb, n0, k0, zb);
    else     tma_load_3d(b_dst, &mapB, fb, k0, n0, zb);
  };
  const bool producer = threadIdx.x == 0;
  int issued = 0;  // K tiles whose loads thread 0 has issued
  if (producer) {
    prefetch_tensormap(&mapA);
    prefetch_tensormap(&mapB);
    for (; issued < nkt && issued < kStages; ++issued) issue(issued);
  }

  const int wm = warp / WN, wn = warp % WN;
  const int ty = lane >> 3, tx = lane & 7;
  Offsets o;
  {
    const uint32_t ra_even = (uint32_t)(wm * 32 + ty);  // rows of even i: & 7 == ty
    const uint32_t ra_odd = ra_even + 4;                 // rows of odd i:  & 7 == ty + 4
    o.xa_even = ra_even * 128u + ((ra_even & 7u) << 4);
    o.xa_odd = ra_odd * 128u + ((ra_odd & 7u) << 4);
    o.xa_mn = (uint32_t)(wm * 32 + 4 * ty) * 4u;
    const uint32_t cb = (uint32_t)(wn * 64 + tx);        // & 7 == tx
    o.xb_k = cb * 128u + ((cb & 7u) << 4);
    o.xb_mn = (uint32_t)(wn * 64 + 4 * tx) * 4u;
  }

  float2 acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.0f, 0.0f);
  {
    // the TMEM running sums start at zero
    float z[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) z[e] = 0.0f;
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_st16(taddr + 16u * c, z);
    tmem_wait_st();
  }

  // Fragments are double-buffered: group g+1 (or the next tile's group 0)
  // is loaded while group g's FMAs issue.
  float a0[4][8], b0[4][8], a1[4][8], b1[4][8];
  bool ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&full_bar[0]), 0u, p.timeout_ns));
  if (!ok) {
    if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
  } else {
    load_group<WM, WN, TA, TB>(smem, smem + T::A_BYTES, 0, o, a0, b0);
  }

  for (int t = 0; ok && t < nkt; ++t) {
    const int s = t % kStages;
    // Refill the stage consumed in the previous iteration with tile t-1+kStages.
    if (producer && t >= 1 && issued < nkt) {
      const int tp = t - 1;
      if (mbar_wait(smem_addr(&empty_bar[tp % kStages]), (uint32_t)(tp / kStages) & 1u, p.timeout_ns)) {
        issue(issued++);
      } else {
        atomicOr(p.fault, (unsigned)kFaultEmptyWait);
        ok = false;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;

    const uint8_t* a_tile = smem + s * T::STAGE_BYTES;
    const uint8_t* b_tile = a_tile + T::A_BYTES;
#pragma unroll
    for (int gp = 0; gp < 4; ++gp) {
      load_group<WM, WN, TA, TB>(a_tile, b_tile, 2 * gp + 1, o, a1, b1);
      fma_group(a0, b0, acc);
      if (gp < 3) {
        load_group<WM, WN, TA, TB>(a_tile, b_tile, 2 * gp + 2, o, a0, b0);
      } else if (t + 1 < nkt) {
        const int sn = (t + 1) % kStages;
        const bool w = __all_sync(0xffffffffu,
                                  mbar_wait(smem_addr(&full_bar[sn]), (uint32_t)((t + 1) / kStages) & 1u, p.timeout_ns));
        if (w) {
          const uint8_t* na = smem + sn * T::STAGE_BYTES;
          load_group<WM, WN, TA, TB>(na, na + T::A_BYTES, 0, o, a0, b0);
        } else {
          if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
          ok = false;
        }
      }
      fma_group(a1, b1, acc);
    }
    mbar_arrive(smem_addr(&empty_bar[s]));
    if (t % kFlushTiles == kFlushTiles - 1) fold_into_tmem(taddr, acc);
  }

  if (ok) {
    // fold the last partial sums: the block's results end up in fin[64]
    float m[4][16];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld16(taddr + 16u * c, m[c]);
    tmem_wait_ld();
    float fin[64];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tmem_ld_ready(m[c]);
#pragma unroll
      for (int e = 0; e < 16; ++e) fin[16 * c + e] = m[c][e];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        fin[8 * i + 2 * q] += acc[i][q].x;
        fin[8 * i + 2 * q + 1] += acc[i][q].y;
      }
    epilogue<WM, WN, TA, TB, SPLIT>(p, p.C + (int64_t)prod * p.stride_c,
                                    p.ws + ((int64_t)prod * gridDim.y + blockIdx.y) * p.M * p.ws_ld, m0, n0, wm,
                                    wn, ty, tx, fin);
  } else if (producer) {
    // A wait gave up.  Thread 0 must not leave while copies it issued into this
    // CTA's shared memory may still land: wait (bounded) for the last phase of
    // every stage that received a load.  C is not written.
    for (int t = issued > kStages ? issued - kStages : 0; t < issued; ++t)
      if (!mbar_wait(smem_addr(&full_bar[t % kStages]), (uint32_t)(t / kStages) & 1u, p.timeout_ns))
        atomicOr(p.fault, (unsigned)kFaultDrainWait);
  }

  // release the tensor memory once every warp is done with it
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem_slot, kTmemCols);
}

template <int WM, int WN, bool TA, bool TB>
cudaError_t launch(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p, int split,
                   cudaStream_t stream) {
  using T = Tile<WM, WN>;
  dim3 grid((unsigned)((int64_t)p.batch * p.tiles_m * p.tiles_n), (unsigned)split);
  if (split > 1)
    tma_gemm_kernel<WM, WN, TA, TB, true><<<grid, kThreads, T::SMEM_BYTES, stream>>>(mapA, mapB, p);
  else
    tma_gemm_kernel<WM, WN, TA, TB, false><<<grid, kThreads, T::SMEM_BYTES, stream>>>(mapA, mapB, p);
  return cudaGetLastError();
}

template <int WM, int WN, bool TA, bool TB>
cudaError_t set_attributes() {
  using T = Tile<WM, WN>;
  cudaError_t e = cudaFuncSetAttribute(tma_gemm_kernel<WM, WN, TA, TB, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(tma_gemm_kernel<WM, WN, TA, TB, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_BYTES);
}

}  // namespace tma
}  // namespace sgemm_impl
