// kernel_skinny.cu -- 3xTF32 SGEMM on the tcgen05 tensor cores for products
// with one short side: at most 64 rows of C (M <= 64) or at most 64 columns
// (N <= 64), for sm_103a.
//
// On the 128 x 128 tiles of the one-CTA kernel (kernel_tf32x3.cu) such a
// product leaves half or more of every tile empty, yet the tile costs its
// full split work and tensor-core time; and the operand with the short side
// is re-split by every CTA that reads it.  Here the kernel sees the product
// as (long side) x (short side): its own M is the long side (L, 128 TMEM
// lanes per tile), its own N the short side (S <= 64, one 64-column
// accumulator), so every tile is full along the long side and tcgen05.mma
// runs at N = 64.  When the short side is M, the kernel computes
// C^T = op(B)^T op(A)^T (the same sums; klklkl10086.github.io
// "Sgemm单精度矩阵乘法", 问题定义) and writes C transposed, a warp storing 32
// consecutive elements of a row of C per instruction.
//
// The short operand is split once per call (split_rows_kernel /
// split_transpose_kernel of kernel_presplit.cu) into K-contiguous hi and lo
// arrays in the workspace, which TMA copies into shared memory already in the
// layout the tensor core reads (the GEMM is a programmatic dependent launch of
// that pass: only the short operand's producer waits for it); only the long operand is split in the
// kernel, into tensor memory (A from TMEM, B from shared memory, as in the
// one-CTA kernel).  Per 32-k tile a CTA moves 16 KB of the long operand
// (read once from HBM for the whole call) and 16 KB of short hi/lo (L2).
//
// The split and the error bounds are those of the one-CTA kernel: hi = x
// rounded to TF32 (ties away), lo = x - hi, products lo*hi + hi*lo + hi*hi
// per k accumulated in FP32 in TMEM, a fresh accumulator per 32-k tile folded
// into FP32 registers with round-to-nearest adds, NaN sums computed again in
// FP32 (kernel_tc_common.cuh).
//
// Schedule: persistent CTAs over the tiles of 128 along the long side, whole
// tiles first, then stream-K over the K tiles of the rest (kernel_tc_common.cuh,
// cta_work / cta_segment); a tile whose K range several CTAs share is written
// as partial sums to the CTA's slots and skinny_fixup_kernel (a programmatic
// dependent launch) adds them in CTA order.  Slots are 64 x 128 floats,
// short index major, so both a folder warp's stores and the fixup's loads
// are 32 consecutive floats.
//
// CTA roles (20 warps):
//   warp 0     TMA producer of the long operand: per 32-k tile its FP32 tile
//              (128 x 32, as stored) into an 8-stage ring that the
//              splitters free.
//   warp 19    TMA producer of the short operand: per 32-k tile its hi and
//              lo tiles (64 x 32 each, K-major, 128-byte swizzle) into a
//              4-stage ring that the MMAs free.
//   warps 1,18 MMA issuers (one thread each; warp 1 takes even K tiles,
//              warp 18 odd ones): 4 k-steps x 3 tcgen05.mma (M=128, N=64,
//              K=8) per K tile.  Every ring has an even number of slots, so
//              each slot of each ring belongs to one issuer and its barrier
//              phases are consecutive for it.  Measured on GB300 at 64 x 4096
//              x 16384 (clock64 traces of one CTA; µs per call): a K tile
//              every ~1190 cycles, about the time one thread takes to issue
//              its 12 MMAs; one issuer 121 µs, two 80, three 85, four 82;
//              the tensor pipe is ~33% busy.  Ring sizes measured no faster:
//              6 + 6 long/short stages, 2 split stages with 6 accumulators,
//              6 split stages with 2 accumulators (one issuer), 10 long stages.
//   warps 2-9  splitters: the long tile -> hi/lo in TMEM (row in lane, k in
//              columns), 4 TMEM stages; warps 2-5 split k 0-15, warps 6-9
//              k 16-31, each half with its own full/empty barriers.
//   warps 10-17 folders: add accumulator t into FP32 registers (each thread:
//              32 columns of one row), then the alpha/beta epilogue.
// Every wait is bounded (mbarrier phases, p.timeout_ns); a wait that gives
// up sets a fault bit and the CTA winds down.
//
// TMEM columns: [64 b, +64) accumulator b (b < 4); [256 + 64 s, +32) long hi
// and [288 + 64 s, +32) long lo of split stage s (s < 4).
#include "kernel_tc_common.cuh"

namespace sgemm_impl {
namespace skinny {

using tc::CtaWork;
using tc::Segment;

constexpr int BM = 128, BN = 64, BK = 32;
// Two TMA rings: the long operand's FP32 tiles, freed as soon as the splitters have read them,
// and the short operand's hi/lo tiles, freed when the MMAs that read them complete.  Separate
// rings keep the HBM stream of the long operand kLongStages tiles ahead of the splitters.
constexpr int kLongStages = 8;
constexpr int kShortStages = 4;
constexpr int kLongBytes = BM * BK * 4;                     // 16 KB
constexpr int kShortBytes = BN * BK * 4;                    // 8 KB, one part
constexpr int kShortStageBytes = 2 * kShortBytes;           // hi + lo
constexpr int kSmemBytes = kLongStages * kLongBytes + kShortStages * kShortStageBytes + 1024;
constexpr int kSplitStages = 4;
constexpr int kHalves = 2;
constexpr int kSplitWarps = 8;
constexpr int kHalfWarps = kSplitWarps / kHalves;
constexpr int kFoldWarps = 8;
constexpr int kFirstFoldWarp = 2 + kSplitWarps;
constexpr int kSecondMmaWarp = kFirstFoldWarp + kFoldWarps;
constexpr int kShortProducerWarp = kSecondMmaWarp + 1;
constexpr int kThreads = 32 * (4 + kSplitWarps + kFoldWarps);
constexpr int kIssuers = 2;  // 1 or 2 (warps 1 and 18)
constexpr int kAccBufs = 4;
constexpr uint32_t kAccCols = BN;
constexpr uint32_t kACols = 64;  // long hi (32 k) + long lo (32 k) of one split stage
constexpr uint32_t kAColBase = kAccBufs * kAccCols;
constexpr uint32_t kTmemCols = 512;
constexpr int kCols = BN / 2;    // accumulator columns one folder thread holds
static_assert(kAColBase + kSplitStages * kACols <= kTmemCols, "accumulators and split stages must fit in TMEM");
static_assert(kShortStages % kIssuers == 0 && kSplitStages % kIssuers == 0 && kAccBufs % kIssuers == 0,
              "each slot of every ring must belong to one issuer");
static_assert(kSmemBytes + 1024 <= 232448, "shared memory per CTA");

// tcgen05 instruction descriptor, kind::tf32: FP32 accumulator, TF32 A and B, both K-major,
// N = 64, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Offset in C of element (i of the long side, j of the short side).
template <bool TRANSC>
__device__ __forceinline__ int64_t c_index(const GemmParams& p, int i, int j) {
  return TRANSC ? (int64_t)j * p.ldc + i : (int64_t)i * p.ldc + j;
}

__device__ __forceinline__ float epi(const GemmParams& p, float v, const float* c) {
  return p.beta == 0.0f ? p.alpha * v : fmaf(p.alpha, v, p.beta * *c);
}

// TL: the long operand is stored long-side contiguous ([K][L]); otherwise K-contiguous ([L][K],
// 128-byte swizzled tiles).  TRANSC: C holds the transpose of the kernel's L x S result.
template <bool TL, bool TRANSC>
__global__ void __launch_bounds__(kThreads, 1)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap mapL, const __grid_constant__ CUtensorMap mapSh,
                       const __grid_constant__ CUtensorMap mapSl, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t long_full[kLongStages], long_empty[kLongStages];
  __shared__ __align__(8) uint64_t short_full[kShortStages], short_empty[kShortStages];
  __shared__ __align__(8) uint64_t split_full[kSplitStages][kHalves], split_empty[kSplitStages][kHalves];
  __shared__ __align__(8) uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  __shared__ uint32_t tmem_slot;
  __shared__ CtaWork work_s;

  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  // [long stages][short stages], every tile 1024-byte aligned
  auto long_tile = [&](int r) { return sbase + (uint32_t)(r * kLongBytes); };
  auto short_tile = [&](int r, int part) {  // 0 hi, 1 lo
    return sbase + (uint32_t)(kLongStages * kLongBytes + r * kShortStageBytes + part * kShortBytes);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = (int)blockIdx.x;
  const int kt_total = (p.K + BK - 1) / BK;
  // the fixup kernel launched after this one may be scheduled now; it waits for this grid
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    work_s = tc::cta_work(p, cta, kt_total);
    for (int r = 0; r < kLongStages; ++r) {
      mbar_init(smem_addr(&long_full[r]), 1);
      mbar_init(smem_addr(&long_empty[r]), kSplitWarps);
    }
    for (int r = 0; r < kShortStages; ++r) {
      mbar_init(smem_addr(&short_full[r]), 1);
      mbar_init(smem_addr(&short_empty[r]), 1);
    }
    for (int s = 0; s < kSplitStages; ++s)
      for (int h = 0; h < kHalves; ++h) {
        mbar_init(smem_addr(&split_full[s][h]), kHalfWarps);
        mbar_init(smem_addr(&split_empty[s][h]), 1);
      }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(smem_addr(&acc_full[b]), 1);
      mbar_init(smem_addr(&acc_empty[b]), kFoldWarps);
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const int nkt = work_s.units;

  if (warp == 0 || warp == kShortProducerWarp) {
    // ------------------------------------------------ TMA producers (warp 0: long ring, warp 19: short ring)
    const bool is_long = warp == 0;
    const int nst = is_long ? kLongStages : kShortStages;
    uint64_t* fullb = is_long ? long_full : short_full;
    uint64_t* emptyb = is_long ? long_empty : short_empty;
    if (lane == 0) {
      if (is_long) {
        prefetch_tensormap(&mapL);
      } else {
        prefetch_tensormap(&mapSh);
        prefetch_tensormap(&mapSl);
        // launched as a programmatic dependent of the short operand's split pass: its arrays are
        // complete once that grid is (the long operand is read as stored, without waiting)
        asm volatile("griddepcontrol.wait;" ::: "memory");
      }
      int issued = 0;
      bool ok = true;
      const CtaWork work = work_s;
      for (int sgi = 0; ok && sgi < work.nseg; ++sgi) {
        const Segment g = tc::cta_segment(p, work, cta, sgi, kt_total);
        const int m0 = g.tile * BM;
        for (int kt = g.kb; kt < g.ke; ++kt) {
          const int t = issued;
          const int r = t % nst;
          if (t >= nst && !mbar_wait(smem_addr(&emptyb[r]), (uint32_t)((t / nst) - 1) & 1u, p.timeout_ns)) {
            atomicOr(p.fault, (unsigned)kFaultEmptyWait);
            ok = false;
            break;
          }
          const uint32_t fb = smem_addr(&fullb[r]);
          const int k0 = kt * BK;
          if (is_long) {
            mbar_arrive_expect_tx(fb, (uint32_t)kLongBytes);
            if (TL) tma_load_3d(long_tile(r), &mapL, fb, m0, k0, 0);
            else    tma_load_3d(long_tile(r), &mapL, fb, k0, m0, 0);
          } else {
            mbar_arrive_expect_tx(fb, (uint32_t)kShortStageBytes);
            tma_load_3d(short_tile(r, 0), &mapSh, fb, k0, 0, 0);
            tma_load_3d(short_tile(r, 1), &mapSl, fb, k0, 0, 0);
          }
          issued = t + 1;
        }
      }
      // leave only when every copy into shared memory has landed
      for (int t = issued > nst ? issued - nst : 0; t < issued; ++t)
        if (!mbar_wait(smem_addr(&fullb[t % nst]), (uint32_t)(t / nst) & 1u, p.timeout_ns))
          atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else if (warp == 1 || warp == kSecondMmaWarp) {
    // ------------------------------------------------ MMA issuers (K tiles t with t % kIssuers == issuer)
    const int issuer = warp == 1 ? 0 : 1;
    if (lane == 0 && issuer < kIssuers) {
      int done = -1;
      bool ok = true;
      for (int t = issuer; ok && t < nkt; t += kIssuers) {
        const int b = t % kAccBufs, r = t % kShortStages, s = t % kSplitStages;
        if (t >= kAccBufs && !mbar_wait(smem_addr(&acc_empty[b]), (uint32_t)((t / kAccBufs) - 1) & 1u, p.timeout_ns))
          ok = false;
        if (ok && !mbar_wait(smem_addr(&short_full[r]), (uint32_t)(t / kShortStages) & 1u, p.timeout_ns)) ok = false;
        if (!ok) break;
        const uint32_t acc = tmem + (uint32_t)b * kAccCols;
        const uint32_t ahi = tmem + kAColBase + (uint32_t)s * kACols, alo = ahi + 32u;
        const uint64_t bhi = tc::kmajor_sw128_desc(short_tile(r, 0)), blo = tc::kmajor_sw128_desc(short_tile(r, 1));
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          if (!mbar_wait(smem_addr(&split_full[s][h]), (uint32_t)(t / kSplitStages) & 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          tmem_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < BK / 8 / kHalves; ++kk) {
            const int ks = h * (BK / 8 / kHalves) + kk;
            const uint64_t step = (uint64_t)(ks * 32) >> 4;  // 8 TF32 = 32 bytes along K
            const uint32_t acol = (uint32_t)(8 * ks);
            mma_tf32_ts(acc, alo + acol, bhi + step, ks == 0 ? 0u : 1u);  // fresh accumulator per K tile
            mma_tf32_ts(acc, ahi + acol, blo + step, 1u);
            mma_tf32_ts(acc, ahi + acol, bhi + step, 1u);
          }
          mma_commit(smem_addr(&split_empty[s][h]));
        }
        if (!ok) break;
        mma_commit(smem_addr(&short_empty[r]));  // the short tiles of stage r have been read
        mma_commit(smem_addr(&acc_full[b]));  // accumulator b holds K tile t
        done = t;
      }
      if (!ok) atomicOr(p.fault, (unsigned)kFaultFullWait);
      if (done >= 0 &&
          !mbar_wait(smem_addr(&acc_full[done % kAccBufs]), (uint32_t)(done / kAccBufs) & 1u, p.timeout_ns))
        atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else if (warp < kFirstFoldWarp) {
    // ------------------------------------------------ splitters: long tile -> hi/lo in TMEM
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;        // which 16 k
    const int m = 32 * q + lane;             // row of the tile (TMEM lane)
    // Debug build: the largest shared- and tensor-memory offsets this thread uses lie in their tiles.
    const bool lay_ok = local_ok(p, kSiteSmem, TL ? (16 * half + 15) * BM + m : (m * 128 + 128) / 4 - 1, 1,
                                 kLongBytes / 4) &&
                        local_ok(p, kSiteTmem, kAColBase + (kSplitStages - 1) * kACols + 16 * half + 32, 16,
                                 kTmemCols);
    for (int t = 0; t < nkt; ++t) {
      const int r = t % kLongStages, s = t % kSplitStages;
      bool w = tc::warp_wait(smem_addr(&long_full[r]), (uint32_t)(t / kLongStages) & 1u, p.timeout_ns);
      if (w && t >= kSplitStages)
        w = tc::warp_wait(smem_addr(&split_empty[s][half]), (uint32_t)((t / kSplitStages) - 1) & 1u, p.timeout_ns);
      if (!w) {
        if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
        break;
      }
      tmem_fence_after_sync();
      if (lay_ok) {
        const uint8_t* ra = smem + (long_tile(r) - sbase);
        float hi[16], lo[16];
        if (!TL) {
          // K-contiguous rows, 128-byte swizzle: 16-byte chunk c of row m sits at c ^ (m & 7)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = 4 * half + j;
            const float4 x = *reinterpret_cast<const float4*>(ra + m * 128 + ((c ^ (m & 7)) << 4));
            float4 h, l;
            tc::split4(x, h, l);
            hi[4 * j + 0] = h.x; hi[4 * j + 1] = h.y; hi[4 * j + 2] = h.z; hi[4 * j + 3] = h.w;
            lo[4 * j + 0] = l.x; lo[4 * j + 1] = l.y; lo[4 * j + 2] = l.z; lo[4 * j + 3] = l.w;
          }
        } else {
          // [32 k][128 rows], rows contiguous: a warp reads 32 adjacent rows per k
          const float* fa = reinterpret_cast<const float*>(ra);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x = fa[(16 * half + j) * BM + m];
            hi[j] = tc::tf32_round(x);
            lo[j] = x - hi[j];
          }
        }
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kAColBase + (uint32_t)s * kACols + 16u * half;
        tmem_st16(ta, hi);
        tmem_st16(ta + 32u, lo);
      }
      tmem_wait_st();
      tmem_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&split_full[s][half]));
        mbar_arrive(smem_addr(&long_empty[r]));
      }
    }
  } else if (warp < kSecondMmaWarp) {
    // ------------------------------------------------ folders, then epilogue
    const int q = warp & 3;
    const int half = (warp - kFirstFoldWarp) >> 2;  // accumulator columns 32 * half .. +31
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kCols * half);
    float2 master2[kCols / 2];
#pragma unroll
    for (int e = 0; e < kCols / 2; ++e) master2[e] = make_float2(0.0f, 0.0f);
    bool ok = true;
    int u = 0;  // K tiles folded so far
    for (int sgi = 0; ok && sgi < work_s.nseg; ++sgi) {
      int len;
      {
        const Segment g = tc::cta_segment(p, work_s, cta, sgi, kt_total);
        len = g.ke - g.kb;
      }
      for (int i = 0; i < len; ++i, ++u) {
        const int b = u % kAccBufs;
        if (!tc::warp_wait(smem_addr(&acc_full[b]), (uint32_t)(u / kAccBufs) & 1u, p.timeout_ns)) {
          ok = false;
          if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
          break;
        }
        tmem_fence_after_sync();
        float v[kCols / 16][16];
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c) tmem_ld16(tq + (uint32_t)b * kAccCols + 16u * c, v[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kCols / 16; ++c) {
          tmem_ld_ready(v[c]);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            master2[8 * c + e] = __fadd2_rn(master2[8 * c + e], make_float2(v[c][2 * e], v[c][2 * e + 1]));
        }
        tmem_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&acc_empty[b]));
      }
      if (!ok) break;
      // epilogue: this thread holds row m0 + 32q + lane (long side), columns j0 .. j0 + 31 (short side)
      const Segment g = tc::cta_segment(p, work_s, cta, sgi, kt_total);
      const int row = 32 * q + lane;
      const int j0 = kCols * half;
      if (g.slot >= 0) {
        // partial sums -> this CTA's slot, [64 short][128 long]: 32 consecutive floats per warp store
        const int64_t base = (int64_t)g.slot * (BM * BN) + row;
#pragma unroll
        for (int e = 0; e < kCols / 2; ++e) {
          const int64_t o0 = base + (int64_t)(j0 + 2 * e) * BM, o1 = o0 + BM;
          if (ws_ok(p, o0, 1)) p.ws[o0] = master2[e].x;
          if (ws_ok(p, o1, 1)) p.ws[o1] = master2[e].y;
        }
      } else {
        const int i = g.tile * BM + row;
        if (i < p.M) {
          tc::repair_nans(p, 0, i, j0, master2);
          if (TRANSC || !p.c_vec) {
#pragma unroll
            for (int e = 0; e < kCols; ++e) {
              const int j = j0 + e;
              const float x = (e & 1) ? master2[e >> 1].y : master2[e >> 1].x;
              const int64_t ci = c_index<TRANSC>(p, i, j);
              if (j < p.N && c_ok(p, ci, 1)) p.C[ci] = epi(p, x, p.C + ci);
            }
          } else {
            float* crow = p.C + (int64_t)i * p.ldc;
#pragma unroll
            for (int e = 0; e < kCols / 4; ++e) {
              const int j = j0 + 4 * e;
              const float x[4] = {master2[2 * e].x, master2[2 * e].y, master2[2 * e + 1].x, master2[2 * e + 1].y};
              if (j >= p.N || !c_ok(p, (int64_t)i * p.ldc + j, min(4, p.N - j))) continue;
              if (j + 3 < p.N) {
                float4 o;
                if (p.beta == 0.0f) {
                  o = make_float4(p.alpha * x[0], p.alpha * x[1], p.alpha * x[2], p.alpha * x[3]);
                } else {
                  const float4 old = *reinterpret_cast<const float4*>(crow + j);
                  o = make_float4(fmaf(p.alpha, x[0], p.beta * old.x), fmaf(p.alpha, x[1], p.beta * old.y),
                                  fmaf(p.alpha, x[2], p.beta * old.z), fmaf(p.alpha, x[3], p.beta * old.w));
                }
                *reinterpret_cast<float4*>(crow + j) = o;
              } else {
                for (int k = 0; k < 4 && j + k < p.N; ++k) crow[j + k] = epi(p, x[k], crow + j + k);
              }
            }
          }
        }
      }
#pragma unroll
      for (int e = 0; e < kCols / 2; ++e) master2[e] = make_float2(0.0f, 0.0f);
    }
  }

  tmem_fence_before_sync();
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// CTA (j, y) of the fixup grid: floats [1024 y, 1024 y + 1024) of stream-K tile j (relative to
// the first) in the slots' short-major order, one float4 per thread: 4 consecutive long-side
// indices of one short-side index.  If several CTAs shared the tile, C = alpha * (sum of their
// slots, in CTA order) + beta * C over the in-range elements.  The order is fixed, so the result
// does not depend on scheduling.
constexpr int kFixupThreads = 256;
constexpr int kFixupFloats = 4 * kFixupThreads;
constexpr int kMaxSharers = 256;
template <bool TRANSC>
__global__ void __launch_bounds__(kFixupThreads) skinny_fixup_kernel(const GemmParams p) {
  __shared__ int s_n;
  __shared__ int s_slot[kMaxSharers];
  // The schedule and C's old values come first (as tc::fixup_prefetch_c: the GEMM never writes C
  // of a shared tile); the grid is a programmatic dependent of the GEMM kernel and waits for it
  // only before reading the partial sums.
  const int kt = (p.K + BK - 1) / BK;
  const int j = (int)blockIdx.x;
  if (threadIdx.x == 0) {
    const int64_t i0 = (int64_t)j * kt;
    const int c0 = tc::sk_owner(p, i0), c1 = tc::sk_owner(p, i0 + kt - 1);
    s_n = min(c1 - c0 + 1, kMaxSharers);
    s_slot[0] = c0;
  }
  __syncthreads();
  const int n = s_n;
  if (n == 1) return;
  const int c0 = s_slot[0];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kFixupThreads) s_slot[i] = tc::sk_slot(p, c0 + i, j, kt);
  __syncthreads();
  const int e = (int)blockIdx.y * kFixupFloats + 4 * (int)threadIdx.x;  // float of the slot
  const int c = e / BM, r = e % BM;                                     // short index, first long index
  const int m0 = (p.sk_tile0 + j) * BM;
  if (c >= p.N || m0 + r >= p.M) return;
  bool ok[4];
  float old[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = m0 + r + k;
    ok[k] = i < p.M && c_ok(p, c_index<TRANSC>(p, i, c), 1);
    old[k] = 0.0f;
    if (ok[k] && p.beta != 0.0f) old[k] = p.C[c_index<TRANSC>(p, i, c)];
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float4 v = tc::fixup_sum(p, s_slot, n, BM * BN, e);
  float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (!ok[k]) continue;
    const int i = m0 + r + k;
    if (!(fabsf(x[k]) <= 3.402823466e38f)) tc::repair_row(p, 0, i, c, &x[k], 1);
    p.C[c_index<TRANSC>(p, i, c)] = p.beta == 0.0f ? p.alpha * x[k] : fmaf(p.alpha, x[k], p.beta * old[k]);
  }
}

}  // namespace skinny

cudaError_t prepare_skinny() {
  using namespace skinny;
  cudaError_t e = cudaFuncSetAttribute(skinny_gemm_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(skinny_gemm_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(skinny_gemm_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(skinny_gemm_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  return e;
}

cudaError_t launch_skinny_gemm(bool long_contig, bool trans_c, const CUtensorMap& mapL, const CUtensorMap& mapSh,
                               const CUtensorMap& mapSl, const GemmParams& p, cudaStream_t stream) {
  using namespace skinny;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.sk_grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // after the split pass (see the producer)
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (long_contig && trans_c) return cudaLaunchKernelEx(&cfg, skinny_gemm_kernel<true, true>, mapL, mapSh, mapSl, p);
  if (long_contig) return cudaLaunchKernelEx(&cfg, skinny_gemm_kernel<true, false>, mapL, mapSh, mapSl, p);
  if (trans_c) return cudaLaunchKernelEx(&cfg, skinny_gemm_kernel<false, true>, mapL, mapSh, mapSl, p);
  return cudaLaunchKernelEx(&cfg, skinny_gemm_kernel<false, false>, mapL, mapSh, mapSl, p);
}

cudaError_t launch_skinny_fixup(bool trans_c, const GemmParams& p, int sk_tiles, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sk_tiles, skinny::BM * skinny::BN / skinny::kFixupFloats);
  cfg.blockDim = dim3(skinny::kFixupThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the GEMM kernel ends
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return trans_c ? cudaLaunchKernelEx(&cfg, skinny::skinny_fixup_kernel<true>, p)
                 : cudaLaunchKernelEx(&cfg, skinny::skinny_fixup_kernel<false>, p);
}

}  // namespace sgemm_impl
