// kernel_tf32x3.cu -- SGEMM on the 5th-generation tensor cores (tcgen05) with
// the 3xTF32 split, for sm_103a.
//
// Each float x is split into hi = x rounded to TF32 (round to nearest, ties
// away, done with integer ops on the bits) and lo = x - hi (exact in float).
// The tensor core reads TF32 operands as the top 19 bits of each 32-bit word,
// so it sees lo truncated: x = hi + lo' + e with |e| < 2^-21 |x|, and e has
// the sign of lo, which is random, so the split adds no bias.  A product is
// formed from three TF32 tensor-core products,
//     a*b ~= a_lo*b_hi + a_hi*b_lo + a_hi*b_hi      (a_lo*b_lo, < 2^-22 |ab|, dropped)
// accumulated in FP32 in tensor memory.  The pages name tensor cores as the
// missing piece of their SGEMM and TF32 as the tensor-core format for FP32
// inputs (itan.pw "CUDA NVIDIA 4090 高性能計算", §4; youngju.dev "CUDA
// architecture visualized", テンソルコア); the split keeps FP32 accuracy, and
// the result must pass the same error bounds as the SIMT kernel.
//
// The tensor core's FP32 accumulation is not round-to-nearest: measured on
// GB300, one accumulator over K = 4096 drifts to a relative Frobenius error of
// ~3e-5, growing linearly with the number of accumulated MMAs (~2e-8 each).
// So every chunk of kFoldTiles 32-k tiles gets a fresh accumulator, and the
// folder warps add it into FP32 registers with round-to-nearest adds; the
// error then no longer grows with K.
//
// TMA writes, split reads and writes and the tensor core's operand reads all
// use the shared-memory data path, so to keep that traffic down the A
// operand's hi/lo parts go to tensor memory (tcgen05.mma reads A from TMEM,
// B from shared memory).  What bounds the kernel is the latency of the feed
// chain (TMA, split, MMA issue, fold), not a bandwidth.
//
// Schedule (persistent CTAs, stream-K balancing without waits between CTAs):
// the grid has G CTAs (at most one per SM when the work allows).  CTA c first
// takes the whole 128x128 output tiles c, c+G, c+2G, ... below sk_tile0
// (data-parallel rounds), then an even share [B(c), B(c+1)) of the K
// iterations of the remaining tiles, B(c) = floor(c*I/G), I = (tiles -
// sk_tile0) * (K tiles per output tile).  A CTA writes a tile it covers
// whole straight to C; a tile whose K range is shared by several CTAs is
// written as partial sums to the CTA's slots (2c: its first stream-K tile,
// 2c+1: its last), and streamk_fixup_kernel (launched after it on the same
// stream as a programmatic dependent, so its launch overlaps this kernel)
// adds the slots of each shared tile in CTA order and applies alpha/beta.
// The output tiles of all products of a strided batch form one sequence.
//
// CTA roles (19 warps):
//   warp 0     TMA producer: FP32 tiles of op(A) and op(B) (as stored) into a
//              4-stage "raw" ring (32 KB per stage).
//   warps 1,18 MMA issuers (one thread each; warp 1 takes even K tiles,
//              warp 18 odd ones; tile t goes to accumulator t % 3): per
//              32-k tile, 4 k-steps x 3 tcgen05.mma (M=128, N=128, K=8);
//              tcgen05.commit releases the split stage and hands the
//              accumulator to the folders.  Issuing one tcgen05.mma takes a
//              thread ~100 cycles on GB300, more than the 64 cycles the tensor
//              core needs for it, so one issuer alone starves the tensor core.
//   warps 2-9  splitters: raw stage t -> A hi/lo in TMEM (row m in lane m, k
//              in columns) and B hi/lo tiles in the K-major, 128-byte swizzled
//              shared-memory layout the tensor core reads (transposed on the
//              way when B is N-contiguous in memory), 2 split stages.  Warps
//              2-5 split k 0-15 of every tile, warps 6-9 k 16-31; each half of
//              a split stage has its own full/empty barriers, so the issuer
//              starts a half's 6 MMAs as soon as it is split and releases it
//              right after them.
//   warps 10-17 folders: add accumulator t into FP32 registers (each thread:
//              64 columns of one row) as soon as its MMAs complete, then the
//              alpha/beta epilogue.
// Only lane 0 of a warp polls a barrier (the others then confirm the
// completed phase once) and arrives on it, which keeps barrier traffic off
// the shared-memory path.  Every wait is bounded (mbarrier phases).
//
// TMEM columns: [128 b, +128) accumulator b (b < 3); [384 + 64 s, +32) A hi
// and [416 + 64 s, +32) A lo of split stage s (s < 2).
#include "kernel_tc_common.cuh"

namespace sgemm_impl {
namespace tc {

constexpr int BM = 128, BN = 128, BK = 32;
constexpr int kRawStages = 4, kSplitStages = 2;
constexpr int kTileBytes = 128 * BK * 4;            // one 128 x 32 operand tile, 16 KB
constexpr int kRawBytes = 2 * kTileBytes;           // A + B as loaded
constexpr int kSplitBytes = 2 * kTileBytes;         // B_hi, B_lo (A's parts live in TMEM)
constexpr int kSmemBytes = kRawStages * kRawBytes + kSplitStages * kSplitBytes + 1024;
constexpr int kSplitWarps = 8;                      // warps 2-9
// The splitters work in two independent groups of 4 warps, one per 16-k half
// of a K tile (warps 2-5: k 0-15, warps 6-9: k 16-31).  Each half of a split
// stage has its own full/empty barriers, so the MMAs of a half start as soon
// as that half is split, and a half is refilled as soon as its 6 MMAs have
// read it.
constexpr int kHalves = 2;
constexpr int kHalfWarps = kSplitWarps / kHalves;
constexpr int kSplitters = 32 * kSplitWarps;
constexpr int kFoldWarps = 8;                       // warps 10-17
constexpr int kFirstFoldWarp = 2 + kSplitWarps;
constexpr int kSecondMmaWarp = kFirstFoldWarp + kFoldWarps;  // warp 18
constexpr int kThreads = 32 * (3 + kSplitWarps + kFoldWarps);
constexpr uint32_t kAccCols = 128;                  // one 128 x 128 FP32 accumulator
constexpr int kAccBufs = 3;                         // accumulators in flight (MMA ahead of the fold)
constexpr int kFoldTiles = 1;                       // 32-k tiles summed in one accumulator before a fold
// Two issuers may alternate only single-tile chunks: an issuer that skipped a
// phase of a stage barrier could not tell the phase it needs from the one
// two ahead (mbarrier waits are by phase parity).
constexpr int kIssuers = kFoldTiles == 1 ? 2 : 1;
static_assert(kFoldTiles == 1, "the folders walk the CTA's segments one accumulator per K tile");
constexpr uint32_t kACols = 64;                     // A hi (32 k) + A lo (32 k) of one split stage
constexpr uint32_t kAColBase = kAccBufs * kAccCols;
constexpr uint32_t kTmemCols = 512;                 // 3 accumulators + 2 A stages = 512
static_assert(kAColBase + kSplitStages * kACols <= kTmemCols, "accumulators and A stages must fit in TMEM");
static_assert(kSmemBytes + 1024 <= 232448, "shared memory per CTA");

// tcgen05 instruction descriptor, kind::tf32: FP32 accumulator, TF32 A and B,
// both K-major, N = 128, M = 128.
constexpr uint32_t kIdesc = (1u << 4)                 // D format: F32
                          | (2u << 7)                 // A format: TF32
                          | (2u << 10)                // B format: TF32
                          | ((uint32_t)(BN >> 3) << 17)
                          | ((uint32_t)(BM >> 4) << 24);

// D (TMEM) = or += A (TMEM, 128 lanes x 8 columns) * B (shared memory, descriptor)
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// Product and origin of output tile `tile` (numbered over all products).
__device__ __forceinline__ void tile_origin(const GemmParams& p, int tile, int& prod, int& m0, int& n0) {
  const int tiles = p.tiles_m * p.tiles_n;
  prod = tile / tiles;
  int tm, tn;
  tile_coords(tile - prod * tiles, p.tiles_m, p.tiles_n, tm, tn);
  m0 = tm * BM;
  n0 = tn * BN;
}

// Raw tile layouts (as the TMA engine copies them):
//   op(A) 'N': [128 rows of M][32 k], K contiguous, 128-byte swizzle;  'T': [32 k][128 m], M contiguous.
//   op(B) 'N': [32 k][128 n], N contiguous;  'T': [128 n][32 k], K contiguous, 128-byte swizzle.
//
// G > 1 (block-diagonal groups): products with M, N <= 128/G go G to a tile:
// rows and columns [g*128/G, (g+1)*128/G) of tile t hold product G*t + g (a
// missing product at the end of the batch reads zeros), so the accumulator's
// diagonal blocks are the G products and 1/G of the tensor-core work is
// useful, instead of 1/G^2 with one product per tile (pairs of 64x64: a half
// instead of a quarter; quads of 32x32: a quarter instead of a sixteenth).  Each operand tile is then G TMA boxes of 128/G rows or
// columns: K-contiguous ones stack into the same layout, while an
// M/N-contiguous one becomes G [32 k][128/G] blocks.  Only the diagonal blocks
// are folded and written to C: a folder warp's 32 rows lie in one block, and
// the two folder warps of a lane quarter take half of its columns each.  There
// is no stream-K in this mode.
template <bool TA, bool TB, int G>
__global__ void __launch_bounds__(kThreads, 1)
    tf32x3_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                       const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  __shared__ __align__(8) uint64_t split_full[kSplitStages][kHalves], split_empty[kSplitStages][kHalves];
  __shared__ __align__(8) uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  __shared__ uint32_t tmem_slot;
  __shared__ CtaWork work_s;  // this CTA's schedule, written once by thread 0 (kept out of registers)

  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  // [raw stages][split stages], every tile 1024-byte aligned
  auto raw_a = [&](int r) { return sbase + (uint32_t)(r * kRawBytes); };
  auto raw_b = [&](int r) { return sbase + (uint32_t)(r * kRawBytes + kTileBytes); };
  auto split_tile = [&](int s, int which) {  // 0 B_hi, 1 B_lo
    return sbase + (uint32_t)(kRawStages * kRawBytes + s * kSplitBytes + which * kTileBytes);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int cta = (int)blockIdx.x;
  const int kt_total = (p.K + BK - 1) / BK;
  // the fixup kernel launched after this one (programmatic dependent launch) may be
  // scheduled now; it waits for this grid to complete before it reads anything
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    work_s = cta_work(p, cta, kt_total);
    for (int r = 0; r < kRawStages; ++r) {
      mbar_init(smem_addr(&raw_full[r]), 1);
      mbar_init(smem_addr(&raw_empty[r]), kSplitWarps);
    }
    for (int s = 0; s < kSplitStages; ++s) {
      for (int h = 0; h < kHalves; ++h) {
        mbar_init(smem_addr(&split_full[s][h]), kHalfWarps);
        mbar_init(smem_addr(&split_empty[s][h]), 1);
      }
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
  const int nkt = work_s.units;  // K tiles this CTA processes, over all its segments (>= 1)

  if (warp == 0) {
    // ------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tensormap(&mapA);
      prefetch_tensormap(&mapB);
      int issued = 0;  // loads issued so far (= the next K tile's position in the ring sequence)
      bool ok = true;
      const CtaWork work = work_s;
      for (int sgi = 0; ok && sgi < work.nseg; ++sgi) {
        const Segment g = cta_segment(p, work, cta, sgi, kt_total);
        int prod, m0, n0;
        if (G > 1) {
          prod = G * g.tile;
          m0 = n0 = 0;
        } else {
          tile_origin(p, g.tile, prod, m0, n0);
        }
        const int za = prod * p.za, zb = prod * p.zb;
        for (int kt = g.kb; kt < g.ke; ++kt) {
          const int t = issued;
          const int r = t % kRawStages;
          if (t >= kRawStages &&
              !mbar_wait(smem_addr(&raw_empty[r]), (uint32_t)((t / kRawStages) - 1) & 1u, p.timeout_ns)) {
            atomicOr(p.fault, (unsigned)kFaultEmptyWait);
            ok = false;
            break;
          }
          const uint32_t fb = smem_addr(&raw_full[r]);
          mbar_arrive_expect_tx(fb, (uint32_t)kRawBytes);
          const int k0 = kt * BK;
          if (G > 1) {
            // G boxes of 128/G rows or columns per operand (16 KB / G each), product G*t + i at i * 16 KB / G
#pragma unroll
            for (int i = 0; i < G; ++i) {
              const uint32_t off = (uint32_t)(i * (kTileBytes / G));
              const int zai = (prod + i) * p.za, zbi = (prod + i) * p.zb;
              if (!TA) tma_load_3d(raw_a(r) + off, &mapA, fb, k0, 0, zai);
              else     tma_load_3d(raw_a(r) + off, &mapA, fb, 0, k0, zai);
              if (!TB) tma_load_3d(raw_b(r) + off, &mapB, fb, 0, k0, zbi);
              else     tma_load_3d(raw_b(r) + off, &mapB, fb, k0, 0, zbi);
            }
          } else {
            if (!TA) tma_load_3d(raw_a(r), &mapA, fb, k0, m0, za);
            else     tma_load_3d(raw_a(r), &mapA, fb, m0, k0, za);
            if (!TB) tma_load_3d(raw_b(r), &mapB, fb, n0, k0, zb);
            else     tma_load_3d(raw_b(r), &mapB, fb, k0, n0, zb);
          }
          issued = t + 1;
        }
      }
      // leave only when every copy into shared memory has landed
      for (int t = issued > kRawStages ? issued - kRawStages : 0; t < issued; ++t)
        if (!mbar_wait(smem_addr(&raw_full[t % kRawStages]), (uint32_t)(t / kRawStages) & 1u, p.timeout_ns))
          atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else if (warp == 1 || warp == kSecondMmaWarp) {
    // ------------------------------------------------ MMA issuers (fold chunks c with c % kIssuers == issuer)
    const int issuer = warp == 1 ? 0 : 1;
    if (lane == 0 && issuer < kIssuers) {
      const int nchunks = (nkt + kFoldTiles - 1) / kFoldTiles;
      int done = -1;  // last chunk whose MMAs this thread issued
      bool ok = true;
      for (int c = issuer; ok && c < nchunks; c += kIssuers) {
        const int b = c % kAccBufs;
        if (c >= kAccBufs &&
            !mbar_wait(smem_addr(&acc_empty[b]), (uint32_t)((c / kAccBufs) - 1) & 1u, p.timeout_ns)) {
          ok = false;
          break;
        }
        const uint32_t acc = tmem + (uint32_t)b * kAccCols;
        for (int t = c * kFoldTiles; t < min(nkt, (c + 1) * kFoldTiles); ++t) {
          const int s = t % kSplitStages;
          const uint32_t ahi = tmem + kAColBase + (uint32_t)s * kACols, alo = ahi + 32u;
          const uint64_t bhi = kmajor_sw128_desc(split_tile(s, 0)), blo = kmajor_sw128_desc(split_tile(s, 1));
          const bool first = t == c * kFoldTiles;
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
              const uint32_t acol = (uint32_t)(8 * ks);        // 8 TF32 = 8 TMEM columns
              mma_tf32_ts(acc, alo + acol, bhi + step, (first && ks == 0) ? 0u : 1u);  // fresh accumulator per chunk
              mma_tf32_ts(acc, ahi + acol, blo + step, 1u);
              mma_tf32_ts(acc, ahi + acol, bhi + step, 1u);
            }
            mma_commit(smem_addr(&split_empty[s][h]));  // this half reusable once these MMAs have read it
          }
          if (!ok) break;
        }
        mma_commit(smem_addr(&acc_full[b]));  // accumulator b holds chunk c
        done = c;
      }
      if (!ok) atomicOr(p.fault, (unsigned)kFaultFullWait);
      // leave only when none of this thread's MMAs is in flight
      if (done >= 0 &&
          !mbar_wait(smem_addr(&acc_full[done % kAccBufs]), (uint32_t)(done / kAccBufs) & 1u, p.timeout_ns))
        atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else if (warp < kFirstFoldWarp) {
    // ------------------------------------------------ splitters
    const int st = threadIdx.x - 64;                 // 0..255
    const int q = warp & 3;                          // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;                // which 16 k of A
    // Debug build: the largest shared- and tensor-memory offsets this thread uses (they do not
    // depend on the K tile) lie inside their tiles; otherwise its loads and stores are skipped.
    const bool lay_ok = [&] {
      const int m = 32 * q + lane, n = st & 127;
      constexpr int lda_s = BM / G, ldb_s = BN / G;
      const int a_max = TA ? (G > 1 ? (m / lda_s) * (BK * lda_s) : 0) + (16 * half + 15) * lda_s + (G > 1 ? m % lda_s : m)
                           : (m * 128 + 128) / 4 - 1;
      const int b_max = !TB ? (G > 1 ? (n / ldb_s) * (BK * ldb_s) : 0) + 31 * ldb_s + (G > 1 ? n % ldb_s : n)
                            : (n * 128 + 128) / 4 - 1;
      return local_ok(p, kSiteSmem, a_max, 1, kTileBytes / 4) && local_ok(p, kSiteSmem, b_max, 1, kTileBytes / 4) &&
             local_ok(p, kSiteSmem, n * 128, 128, kTileBytes) &&
             local_ok(p, kSiteTmem, kAColBase + (kSplitStages - 1) * kACols + 16 * half + 32, 16, kTmemCols);
    }();
    for (int t = 0; t < nkt; ++t) {
      const int r = t % kRawStages, s = t % kSplitStages;
      bool w = warp_wait(smem_addr(&raw_full[r]), (uint32_t)(t / kRawStages) & 1u, p.timeout_ns);
      if (w && t >= kSplitStages)
        w = warp_wait(smem_addr(&split_empty[s][half]), (uint32_t)((t / kSplitStages) - 1) & 1u, p.timeout_ns);
      if (!w) {
        if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
        break;
      }
      tmem_fence_after_sync();
      // A: this thread takes row m = 32q + lane (its TMEM lane) and k = 16*half .. +15.
      if (lay_ok) {
        const uint8_t* ra = smem + (raw_a(r) - sbase);
        const int m = 32 * q + lane;
        float hi[16], lo[16];
        if (!TA) {
          // K-contiguous rows, 128-byte swizzle: chunk c of row m sits at c ^ (m & 7)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c = 4 * half + j;
            const float4 x = *reinterpret_cast<const float4*>(ra + m * 128 + ((c ^ (m & 7)) << 4));
            float4 h, l;
            split4(x, h, l);
            hi[4 * j + 0] = h.x; hi[4 * j + 1] = h.y; hi[4 * j + 2] = h.z; hi[4 * j + 3] = h.w;
            lo[4 * j + 0] = l.x; lo[4 * j + 1] = l.y; lo[4 * j + 2] = l.z; lo[4 * j + 3] = l.w;
          }
        } else {
          // M-contiguous [32 k][128 m] (G > 1: G blocks [32 k][128/G m]): one float per k (a warp
          // reads 32 adjacent m, all in one block)
          constexpr int lda_s = BM / G;
          const float* fa = reinterpret_cast<const float*>(ra) + (G > 1 ? (m / lda_s) * (BK * lda_s) : 0);
          const int mm = G > 1 ? m % lda_s : m;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x = fa[(16 * half + j) * lda_s + mm];
            hi[j] = tf32_round(x);
            lo[j] = x - hi[j];
          }
        }
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kAColBase + (uint32_t)s * kACols + 16u * half;
        tmem_st16(ta, hi);
        tmem_st16(ta + 32u, lo);
      }
      // B -> K-major [128 n][32 k], 128-byte swizzle, the layout the descriptors describe;
      // this group writes the 16 k of its half (st / 128 == half).
      if (lay_ok) {
        uint8_t* bhi = smem + (split_tile(s, 0) - sbase);
        uint8_t* blo = smem + (split_tile(s, 1) - sbase);
        if (!TB) {
          // raw [32 k][128 n] (G > 1: G blocks [32 k][128/G n]): transpose; thread st owns column
          // n = st % 128, k chunks 4*(st/128) .. +3
          constexpr int ldb_s = BN / G;
          const int n = st & 127, kh = st >> 7;
          const float* rb =
              reinterpret_cast<const float*>(smem + (raw_b(r) - sbase)) + (G > 1 ? (n / ldb_s) * (BK * ldb_s) : 0);
          const int nn = G > 1 ? n % ldb_s : n;
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int kc = 4 * kh + kq;
            const float4 x = make_float4(rb[(4 * kc + 0) * ldb_s + nn], rb[(4 * kc + 1) * ldb_s + nn],
                                         rb[(4 * kc + 2) * ldb_s + nn], rb[(4 * kc + 3) * ldb_s + nn]);
            float4 hi, lo;
            split4(x, hi, lo);
            const uint32_t off = (uint32_t)n * 128u + ((uint32_t)(kc ^ (n & 7)) << 4);
            *reinterpret_cast<float4*>(bhi + off) = hi;
            *reinterpret_cast<float4*>(blo + off) = lo;
          }
        } else {
          // raw is already K-major and swizzled: split this half's 16-byte chunks in place
          // (thread st: row n = st % 128, logical k chunks 4*(st/128) .. +3)
          const uint8_t* rb = smem + (raw_b(r) - sbase);
          const int n = st & 127, kh = st >> 7;
#pragma unroll
          for (int kq = 0; kq < 4; ++kq) {
            const int kc = 4 * kh + kq;
            const uint32_t off = (uint32_t)n * 128u + ((uint32_t)(kc ^ (n & 7)) << 4);
            float4 hi, lo;
            split4(*reinterpret_cast<const float4*>(rb + off), hi, lo);
            *reinterpret_cast<float4*>(bhi + off) = hi;
            *reinterpret_cast<float4*>(blo + off) = lo;
          }
        }
      }
      tmem_wait_st();            // A parts have reached TMEM
      fence_proxy_async_smem();  // B parts (generic-proxy writes) -> visible to the tensor core
      tmem_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&split_full[s][half]));
        mbar_arrive(smem_addr(&raw_empty[r]));
      }
    }
  } else {
    // ------------------------------------------------ folders, then epilogue
    const int q = warp & 3;                          // TMEM lane quarter this warp may access
    const int half = (warp - kFirstFoldWarp) >> 2;   // which 64 accumulator columns
    // G > 1: only the diagonal block of this warp's 32 rows is a product; the two folder warps of
    // this lane quarter split its columns (the warp whose 64 columns hold the block takes the
    // first half, the other warp the second)
    constexpr int kBlock = BM / G;
    constexpr int kCols = G == 1 ? 64 : (kBlock < 64 ? kBlock : 64) / 2;  // accumulator columns a warp folds
    const int blk = G > 1 ? (32 * q) / kBlock : 0;
    const int col0 = G > 1 ? kBlock * blk + ((kBlock * blk) / 64 == half ? 0 : kCols) : 64 * half;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col0;
    float2 master2[kCols / 2];  // columns 2e, 2e+1 of the thread's kCols
#pragma unroll
    for (int e = 0; e < kCols / 2; ++e) master2[e] = make_float2(0.0f, 0.0f);
    bool ok = true;
    int u = 0;  // accumulator sequence number (one per K tile; kFoldTiles == 1)
    for (int sgi = 0; ok && sgi < work_s.nseg; ++sgi) {
      int len;  // K tiles of this segment (the segment itself is looked up again for its epilogue)
      {
        const Segment g = cta_segment(p, work_s, cta, sgi, kt_total);
        len = g.ke - g.kb;
      }
      for (int i = 0; i < len; ++i, ++u) {
        const int b = u % kAccBufs;
        if (!warp_wait(smem_addr(&acc_full[b]), (uint32_t)(u / kAccBufs) & 1u, p.timeout_ns)) {
          ok = false;
          if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
          break;
        }
        {
          tmem_fence_after_sync();
          float v[kCols / 16][16];
#pragma unroll
          for (int c = 0; c < kCols / 16; ++c) tmem_ld16(tq + (uint32_t)b * kAccCols + 16u * c, v[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < kCols / 16; ++c) {
            tmem_ld_ready(v[c]);
#pragma unroll
            for (int e = 0; e < 8; ++e)  // round-to-nearest FP32 adds, two per instruction
              master2[8 * c + e] = __fadd2_rn(master2[8 * c + e], make_float2(v[c][2 * e], v[c][2 * e + 1]));
          }
          tmem_fence_before_sync();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&acc_empty[b]));
      }
      if (!ok) break;
      // epilogue of this segment: this thread holds row 32q + lane, columns 64*half .. +63 of the tile
      const Segment g = cta_segment(p, work_s, cta, sgi, kt_total);
      if (g.slot >= 0) {
        // partial sums of a shared stream-K tile -> this CTA's slot (whole 128 x 128, no bounds)
        const int64_t woff = (int64_t)g.slot * (BM * BN) + (32 * q + lane) * BN + 64 * half;
        float* w = p.ws + woff;
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (ws_ok(p, woff + 4 * e, 4))
            *reinterpret_cast<float4*>(w + 4 * e) =
                make_float4(master2[2 * e].x, master2[2 * e].y, master2[2 * e + 1].x, master2[2 * e + 1].y);
      } else {
        int prod, m0, c0;  // product, origin row of the tile in it, first column of this thread's
        if (G > 1) {
          prod = G * g.tile + blk;  // rows and columns kBlock*blk .. +kBlock-1 of the tile
          m0 = -kBlock * blk;
          c0 = col0 - kBlock * blk;
        } else {
          int n0;
          tile_origin(p, g.tile, prod, m0, n0);
          c0 = n0 + 64 * half;
        }
        const int row = m0 + 32 * q + lane;
        if (row < p.M && (G == 1 || prod < p.batch)) {
          repair_nans(p, prod, row, c0, master2);
          const int64_t roff = (int64_t)prod * p.stride_c + (int64_t)row * p.ldc;
          float* crow = p.C + roff;
#pragma unroll
          for (int e = 0; e < kCols / 4; ++e) {
            const int col = c0 + 4 * e;
            const float x[4] = {master2[2 * e].x, master2[2 * e].y, master2[2 * e + 1].x, master2[2 * e + 1].y};
            if (col >= p.N || !c_ok(p, roff + col, min(4, p.N - col))) continue;
            if (p.c_vec && col + 3 < p.N) {
              float4 o;
              if (p.beta == 0.0f) {
                o = make_float4(p.alpha * x[0], p.alpha * x[1], p.alpha * x[2], p.alpha * x[3]);
              } else {
                const float4 old = *reinterpret_cast<const float4*>(crow + col);
                o = make_float4(fmaf(p.alpha, x[0], p.beta * old.x), fmaf(p.alpha, x[1], p.beta * old.y),
                                fmaf(p.alpha, x[2], p.beta * old.z), fmaf(p.alpha, x[3], p.beta * old.w));
              }
              *reinterpret_cast<float4*>(crow + col) = o;
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                if (col + k < p.N)
                  crow[col + k] = p.beta == 0.0f ? p.alpha * x[k] : fmaf(p.alpha, x[k], p.beta * crow[col + k]);
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

// CTA (j, y) of the fixup grid: rows 8y .. 8y+7 of stream-K tile j, one float4
// of 4 columns per thread.  If several CTAs shared tile j, C = alpha * (sum of
// their slots, in CTA order) + beta * C over the in-range elements.  The
// order is fixed, so the result does not depend on scheduling.
constexpr int kFixupRowsPerCta = 8;
constexpr int kFixupThreads = 256;
constexpr int kMaxSharers = 256;  // CTAs that may share one tile (the planner keeps to it)
template <bool CVEC>
__global__ void __launch_bounds__(kFixupThreads) streamk_fixup_kernel(const GemmParams p) {
  __shared__ int s_n;
  __shared__ int s_slot[kMaxSharers];
  // The schedule and C's old values come first (fixup_prefetch_c); the grid is a programmatic
  // dependent of the GEMM kernel and waits for it only before reading the partial sums.
  const int kt = (p.K + BK - 1) / BK;
  const int j = (int)blockIdx.x;
  // the tile's sharers and their slots, once per CTA (64-bit divisions stay off the threads' path)
  if (threadIdx.x == 0) {
    const int64_t i0 = (int64_t)j * kt;
    const int c0 = sk_owner(p, i0), c1 = sk_owner(p, i0 + kt - 1);
    s_n = min(c1 - c0 + 1, kMaxSharers);
    s_slot[0] = c0;
  }
  __syncthreads();
  const int n = s_n;
  if (n == 1) return;  // one CTA covered the whole tile and wrote C itself
  const int c0 = s_slot[0];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kFixupThreads) s_slot[i] = sk_slot(p, c0 + i, j, kt);
  __syncthreads();
  int prod, m0, n0;
  tile_origin(p, p.sk_tile0 + j, prod, m0, n0);
  const int r = (int)blockIdx.y * kFixupRowsPerCta + (int)(threadIdx.x >> 5);
  const int cc = (int)(threadIdx.x & 31) * 4;
  const int row = m0 + r, col = n0 + cc;
  if (row >= p.M || col >= p.N) return;
  const FixupOut f = fixup_prefetch_c<CVEC>(p, prod, row, col);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float4 v = fixup_sum(p, s_slot, n, BM * BN, (int64_t)r * BN + cc);
  repair_nans4(p, prod, row, col, v);
  fixup_store<CVEC>(p, f, v);
}

}  // namespace tc

namespace {

template <bool TA, bool TB, int G>
cudaError_t set_attrs() {
  return cudaFuncSetAttribute(tc::tf32x3_gemm_kernel<TA, TB, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              tc::kSmemBytes);
}

template <int G>
cudaError_t set_attrs_ops() {
  cudaError_t e = set_attrs<false, false, G>();
  if (e == cudaSuccess) e = set_attrs<false, true, G>();
  if (e == cudaSuccess) e = set_attrs<true, false, G>();
  if (e == cudaSuccess) e = set_attrs<true, true, G>();
  return e;
}

template <bool TA, bool TB, int G>
cudaError_t launch(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p, cudaStream_t stream) {
  tc::tf32x3_gemm_kernel<TA, TB, G><<<(unsigned)p.sk_grid, tc::kThreads, tc::kSmemBytes, stream>>>(mapA, mapB, p);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_ops(bool transA, bool transB, const CUtensorMap& mapA, const CUtensorMap& mapB,
                       const GemmParams& p, cudaStream_t stream) {
  if (!transA && !transB) return launch<false, false, G>(mapA, mapB, p, stream);
  if (!transA && transB) return launch<false, true, G>(mapA, mapB, p, stream);
  if (transA && !transB) return launch<true, false, G>(mapA, mapB, p, stream);
  return launch<true, true, G>(mapA, mapB, p, stream);
}

}  // namespace

cudaError_t prepare_tf32x3() {
  cudaError_t e = set_attrs_ops<1>();
  if (e == cudaSuccess) e = set_attrs_ops<2>();
  if (e == cudaSuccess) e = set_attrs_ops<4>();
  return e;
}

cudaError_t launch_tf32x3(bool transA, bool transB, int group, const CUtensorMap& mapA, const CUtensorMap& mapB,
                          const GemmParams& p, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_ops<1>(transA, transB, mapA, mapB, p, stream);
    case 2: return launch_ops<2>(transA, transB, mapA, mapB, p, stream);
    case 4: return launch_ops<4>(transA, transB, mapA, mapB, p, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_streamk_fixup(const GemmParams& p, int sk_tiles, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sk_tiles, tc::BM / tc::kFixupRowsPerCta);
  cfg.blockDim = dim3(tc::kFixupThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the GEMM kernel ends
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.c_vec ? cudaLaunchKernelEx(&cfg, tc::streamk_fixup_kernel<true>, p)
                 : cudaLaunchKernelEx(&cfg, tc::streamk_fixup_kernel<false>, p);
}

}  // namespace sgemm_impl
