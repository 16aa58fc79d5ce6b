// kernel_tc_pair.cu -- 3xTF32 SGEMM on CTA pairs (tcgen05 cta_group::2), for sm_103a.
//
// Same arithmetic as kernel_tf32x3.cu (each float split into a TF32 hi part
// and an FP32 lo part, three TF32 tensor-core products per k, a fresh TMEM
// accumulator per 32-k tile folded into FP32 registers with round-to-nearest
// adds), on output tiles of 256 x 128 computed by the two CTAs of a cluster
// (two SMs of one TPC).  One thread of the pair's even CTA issues every
// tcgen05.mma with M = 256: each CTA holds 128 rows of the tile's A (hi/lo
// parts in its own TMEM) and 64 of the tile's 128 columns of B (hi/lo parts
// in its own shared memory), and each CTA's TMEM receives its 128 rows of
// the accumulator.  The tensor core reads B from shared memory three times
// per k (hi, lo, hi), so per SM the pair halves that traffic, the largest
// share of the shared-memory data path in the one-CTA kernel, and halves the
// TMA and split traffic of B.  The pages name tensor cores as the missing
// piece of their SGEMM (itan.pw "CUDA NVIDIA 4090 高性能計算", §4).
//
// Schedule: the kernel in kernel_tf32x3.cu with the cluster as the unit: the
// grid holds G clusters; cluster c takes whole pair tiles c, c+G, ... below
// sk_tile0, then an even share of the K iterations of the rest (stream-K).
// CTA r of the pair covers rows [128 r, 128 r + 128) of each pair tile; a
// tile shared by several clusters leaves partial sums in slot 2 * s + r
// (s = 2c: the cluster's first stream-K tile, 2c + 1: its last), which
// pair_fixup_kernel adds in cluster order.
//
// Barriers.  Each CTA has its own raw TMA ring (raw_full / raw_empty, local).
// The even CTA's split_full (count: the splitter warps of both CTAs) and
// acc_empty (count: the folder warps of both CTAs) receive arrivals from both
// CTAs (remote mbarrier arrivals through the cluster shared-memory window).
// The issuer's tcgen05.commit multicasts split_empty and acc_full to both
// CTAs.  Before a CTA leaves, its splitters wait for the last split_empty
// phases (no commit may land in a CTA that has exited) and the two CTAs
// meet on a bounded handshake; only then is TMEM released.
//
// CTA roles (19 warps, as in the one-CTA kernel): warp 0 TMA producer;
// warps 1 and 18 MMA issuers (even CTA only; alternate K tiles); warps 2-9
// splitters (A: 128 rows x 32 k -> TMEM, B: 64 columns x 32 k -> K-major
// 128-byte-swizzled hi/lo tiles); warps 10-17 folders and epilogue.
//
// TMEM columns (both CTAs, allocated as a pair): [128 b, +128) accumulator b
// (b < 3); [384 + 64 s, +32) A hi and [416 + 64 s, +32) A lo of split stage s.
#include "kernel_tc_common.cuh"

namespace sgemm_impl {
namespace tcp {

using namespace tc;

constexpr int BM = 256;                  // rows of a pair tile
constexpr int BMC = 128;                 // rows one CTA covers
constexpr int BN = 128;                  // columns of a pair tile
constexpr int BNC = 64;                  // columns of B one CTA loads and splits
constexpr int BK = 32;
constexpr int kRawStages = 6, kSplitStages = 2;
constexpr int kATileBytes = BMC * BK * 4;           // 16 KB
constexpr int kBTileBytes = BNC * BK * 4;           // 8 KB
constexpr int kRawBytes = kATileBytes + kBTileBytes;
constexpr int kSplitBytes = 2 * kBTileBytes;        // B hi, B lo (A's parts live in TMEM)
constexpr int kSmemBytes = kRawStages * kRawBytes + kSplitStages * kSplitBytes + 1024;
constexpr int kSplitWarps = 8;                      // warps 2-9, two groups of 4 (one per 16-k half)
constexpr int kHalves = 2;
constexpr int kHalfWarps = kSplitWarps / kHalves;
constexpr int kFoldWarps = 8;                       // warps 10-17
constexpr int kFirstFoldWarp = 2 + kSplitWarps;
constexpr int kSecondMmaWarp = kFirstFoldWarp + kFoldWarps;  // warp 18
constexpr int kThreads = 32 * (3 + kSplitWarps + kFoldWarps);
constexpr uint32_t kAccCols = 128;
constexpr int kAccBufs = 3;
constexpr int kIssuers = 2;
constexpr uint32_t kACols = 64;
constexpr uint32_t kAColBase = kAccBufs * kAccCols;
constexpr uint32_t kTmemCols = 512;
static_assert(kAColBase + kSplitStages * kACols <= kTmemCols, "accumulators and A stages must fit in TMEM");
static_assert(kSmemBytes + 1024 <= 232448, "shared memory per CTA");

// tcgen05 instruction descriptor, kind::tf32: FP32 accumulator, TF32 A and B,
// both K-major, N = 128, M = 256 (the pair).
constexpr uint32_t kIdesc = (1u << 4)                 // D format: F32
                          | (2u << 7)                 // A format: TF32
                          | (2u << 10)                // B format: TF32
                          | ((uint32_t)(BN >> 3) << 17)
                          | ((uint32_t)(BM >> 4) << 24);

// D (both CTAs' TMEM) = or += A (both CTAs' TMEM, 128 lanes x 8 columns each) * B (64 rows of
// K-major shared memory in each CTA at the same address)
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

// Product and origin (first row, first column) of pair tile `tile`.
__device__ __forceinline__ void pair_tile_origin(const GemmParams& p, int tile, int& prod, int& m0, int& n0) {
  tile_origin_of(p, tile, BM, BN, prod, m0, n0);
}

// Raw tile layouts (as the TMA engine copies them), per CTA:
//   op(A) 'N': [128 rows of M][32 k], K contiguous, 128-byte swizzle;  'T': [32 k][128 m], M contiguous.
//   op(B) 'N': [32 k][64 n], N contiguous;  'T': [64 n][32 k], K contiguous, 128-byte swizzle.
template <bool TA, bool TB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    pair_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                     const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  __shared__ __align__(8) uint64_t split_full[kSplitStages][kHalves], split_empty[kSplitStages][kHalves];
  __shared__ __align__(8) uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  __shared__ __align__(8) uint64_t fin;
  __shared__ uint32_t tmem_slot;
  __shared__ CtaWork work_s;

  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;  // the same in both CTAs (same kernel)
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_addr + pad;
  // [raw stages: A 16 KB, B 8 KB][split stages: B hi 8 KB, B lo 8 KB], every tile 1024-byte aligned
  auto raw_a = [&](int r) { return sbase + (uint32_t)(r * kRawBytes); };
  auto raw_b = [&](int r) { return sbase + (uint32_t)(r * kRawBytes + kATileBytes); };
  auto split_tile = [&](int s, int which) {  // 0 B_hi, 1 B_lo
    return sbase + (uint32_t)(kRawStages * kRawBytes + s * kSplitBytes + which * kBTileBytes);
  };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: issues the pair's MMAs
  const int cl = (int)cluster_id_x();    // the scheduling unit
  const int kt_total = (p.K + BK - 1) / BK;
  // the fixup kernel launched after this one may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    work_s = cta_work(p, cl, kt_total);
    for (int r = 0; r < kRawStages; ++r) {
      mbar_init(smem_addr(&raw_full[r]), 1);
      mbar_init(smem_addr(&raw_empty[r]), kSplitWarps);
    }
    for (int s = 0; s < kSplitStages; ++s) {
      for (int h = 0; h < kHalves; ++h) {
        mbar_init(smem_addr(&split_full[s][h]), 2 * kHalfWarps);
        mbar_init(smem_addr(&split_empty[s][h]), 1);
      }
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(smem_addr(&acc_full[b]), 1);
      mbar_init(smem_addr(&acc_empty[b]), 2 * kFoldWarps);
    }
    mbar_init(smem_addr(&fin), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc_pair(smem_addr(&tmem_slot), kTmemCols);
  tmem_fence_before_sync();
  cluster_sync();  // both CTAs' barriers initialised and TMEM allocated before any cross-CTA traffic
  tmem_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const int nkt = work_s.units;  // K tiles of this cluster's work (the same in both CTAs)

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (each CTA: its rows of A, its columns of B)
    if (lane == 0) {
      prefetch_tensormap(&mapA);
      prefetch_tensormap(&mapB);
      int issued = 0;
      bool ok = true;
      const CtaWork work = work_s;
      for (int sgi = 0; ok && sgi < work.nseg; ++sgi) {
        const Segment g = cta_segment(p, work, cl, sgi, kt_total);
        int prod, m0, n0;
        pair_tile_origin(p, g.tile, prod, m0, n0);
        m0 += BMC * (int)rank;
        n0 += BNC * (int)rank;
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
          if (!TA) tma_load_3d(raw_a(r), &mapA, fb, k0, m0, za);
          else     tma_load_3d(raw_a(r), &mapA, fb, m0, k0, za);
          if (!TB) tma_load_3d(raw_b(r), &mapB, fb, n0, k0, zb);
          else     tma_load_3d(raw_b(r), &mapB, fb, k0, n0, zb);
          issued = t + 1;
        }
      }
      // leave only when every copy into shared memory has landed
      for (int t = issued > kRawStages ? issued - kRawStages : 0; t < issued; ++t)
        if (!mbar_wait(smem_addr(&raw_full[t % kRawStages]), (uint32_t)(t / kRawStages) & 1u, p.timeout_ns))
          atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else if (warp == 1 || warp == kSecondMmaWarp) {
    // ------------------------------------------------ MMA issuers (even CTA; tile t goes to issuer t % 2)
    const int issuer = warp == 1 ? 0 : 1;
    if (rank == 0 && lane == 0 && issuer < kIssuers) {
      int done = -1;
      bool ok = true;
      for (int t = issuer; ok && t < nkt; t += kIssuers) {
        const int b = t % kAccBufs;
        const uint32_t acc = tmem + (uint32_t)b * kAccCols;
        const int s = t % kSplitStages;
        const uint32_t ahi = tmem + kAColBase + (uint32_t)s * kACols, alo = ahi + 32u;
        const uint64_t bhi = kmajor_sw128_desc(split_tile(s, 0)), blo = kmajor_sw128_desc(split_tile(s, 1));
        // The accumulator is taken only once the tile's first operands are split: an accumulator
        // held while its issuer waits for split data lengthens the loop MMA -> fold -> MMA that
        // the three accumulators have to cover.
#pragma unroll
        for (int h = 0; h < kHalves; ++h) {
          if (!mbar_wait(smem_addr(&split_full[s][h]), (uint32_t)(t / kSplitStages) & 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          if (h == 0 && t >= kAccBufs &&
              !mbar_wait(smem_addr(&acc_empty[b]), (uint32_t)((t / kAccBufs) - 1) & 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          tmem_fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < BK / 8 / kHalves; ++kk) {
            const int ks = h * (BK / 8 / kHalves) + kk;
            const uint64_t step = (uint64_t)(ks * 32) >> 4;  // 8 TF32 = 32 bytes along K
            const uint32_t acol = (uint32_t)(8 * ks);        // 8 TF32 = 8 TMEM columns
            mma_pair(acc, alo + acol, bhi + step, ks == 0 ? 0u : 1u);  // fresh accumulator per K tile
            mma_pair(acc, ahi + acol, blo + step, 1u);
            mma_pair(acc, ahi + acol, bhi + step, 1u);
          }
          mma_commit_pair(smem_addr(&split_empty[s][h]));  // this half reusable in both CTAs
        }
        if (!ok) break;
        mma_commit_pair(smem_addr(&acc_full[b]));  // accumulator b (both CTAs) holds tile t
        done = t;
      }
      if (!ok) atomicOr(p.fault, (unsigned)kFaultFullWait);
      if (done >= 0 &&
          !mbar_wait(smem_addr(&acc_full[done % kAccBufs]), (uint32_t)(done / kAccBufs) & 1u, p.timeout_ns))
        atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else if (warp < kFirstFoldWarp) {
    // ------------------------------------------------ splitters (both CTAs)
    const int st = threadIdx.x - 64;                 // 0..255
    const int q = warp & 3;                          // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;                // which 16 k of the tile (st >> 7)
    // Debug build: the largest shared- and tensor-memory offsets this thread uses lie inside
    // their tiles; otherwise its loads and stores are skipped.
    const bool lay_ok = [&] {
      const int m = 32 * q + lane, n = st & 63;
      const int a_max = TA ? (16 * half + 15) * BMC + m : (m * 128 + 128) / 4 - 1;
      const int b_max = !TB ? 31 * BNC + n : (n * 128 + 128) / 4 - 1;
      return local_ok(p, kSiteSmem, a_max, 1, kATileBytes / 4) && local_ok(p, kSiteSmem, b_max, 1, kBTileBytes / 4) &&
             local_ok(p, kSiteSmem, n * 128, 128, kBTileBytes) &&
             local_ok(p, kSiteTmem, kAColBase + (kSplitStages - 1) * kACols + 16 * half + 32, 16, kTmemCols);
    }();
    int t = 0;
    for (; t < nkt; ++t) {
      const int r = t % kRawStages, s = t % kSplitStages;
      if (!warp_wait(smem_addr(&raw_full[r]), (uint32_t)(t / kRawStages) & 1u, p.timeout_ns)) {
        if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
        break;
      }
      // Load and split into registers first; only the stores wait for the split stage, so the
      // loads and the split arithmetic stay off the loop MMA completion -> split stage -> MMA.
      // A: this thread takes row m = 32q + lane (its TMEM lane) and k = 16*half .. +15.
      float hi[16], lo[16];
      if (lay_ok) {
        const uint8_t* ra = smem + (raw_a(r) - sbase);
        const int m = 32 * q + lane;
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
          // M-contiguous [32 k][128 m]: one float per k (a warp reads 32 adjacent m)
          const float* fa = reinterpret_cast<const float*>(ra);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float x = fa[(16 * half + j) * BMC + m];
            hi[j] = tf32_round(x);
            lo[j] = x - hi[j];
          }
        }
      }
      // B -> K-major [64 n][32 k], 128-byte swizzle, the layout the descriptors describe; thread st
      // takes column n = st % 64 and the two 4-k chunks 4*half + 2*((st / 64) % 2) + {0, 1}.
      const int n = st & 63, kp = (st >> 6) & 1;
      float4 bh[2], bl[2];
      if (!lay_ok) {
      } else if (!TB) {
        // raw [32 k][64 n]: transpose on the way (a warp reads 32 adjacent n of one k)
        const float* rb = reinterpret_cast<const float*>(smem + (raw_b(r) - sbase));
#pragma unroll
        for (int kq = 0; kq < 2; ++kq) {
          const int kc = 4 * half + 2 * kp + kq;
          const float4 x = make_float4(rb[(4 * kc + 0) * BNC + n], rb[(4 * kc + 1) * BNC + n],
                                       rb[(4 * kc + 2) * BNC + n], rb[(4 * kc + 3) * BNC + n]);
          split4(x, bh[kq], bl[kq]);
        }
      } else {
        // raw is already K-major and swizzled: the chunks keep their place
        const uint8_t* rb = smem + (raw_b(r) - sbase);
#pragma unroll
        for (int kq = 0; kq < 2; ++kq) {
          const int kc = 4 * half + 2 * kp + kq;
          const uint32_t off = (uint32_t)n * 128u + ((uint32_t)(kc ^ (n & 7)) << 4);
          split4(*reinterpret_cast<const float4*>(rb + off), bh[kq], bl[kq]);
        }
      }
      if (t >= kSplitStages &&
          !warp_wait(smem_addr(&split_empty[s][half]), (uint32_t)((t / kSplitStages) - 1) & 1u, p.timeout_ns)) {
        if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
        break;
      }
      tmem_fence_after_sync();
      if (lay_ok) {
        const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + kAColBase + (uint32_t)s * kACols + 16u * half;
        tmem_st16(ta, hi);
        tmem_st16(ta + 32u, lo);
        uint8_t* bhi = smem + (split_tile(s, 0) - sbase);
        uint8_t* blo = smem + (split_tile(s, 1) - sbase);
#pragma unroll
        for (int kq = 0; kq < 2; ++kq) {
          const int kc = 4 * half + 2 * kp + kq;
          const uint32_t off = (uint32_t)n * 128u + ((uint32_t)(kc ^ (n & 7)) << 4);
          *reinterpret_cast<float4*>(bhi + off) = bh[kq];
          *reinterpret_cast<float4*>(blo + off) = bl[kq];
        }
      }
      tmem_wait_st();            // A parts have reached TMEM
      fence_proxy_async_smem();  // B parts (generic-proxy writes) -> visible to the tensor core
      tmem_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_remote(smem_addr(&split_full[s][half]), 0);
        mbar_arrive(smem_addr(&raw_empty[r]));
      }
    }
    // the issuer's last commits on this half's split stages land in this CTA: wait for them
    if (t == nkt) {
      for (int u = nkt > kSplitStages ? nkt - kSplitStages : 0; u < nkt; ++u)
        if (!warp_wait(smem_addr(&split_empty[u % kSplitStages][half]), (uint32_t)(u / kSplitStages) & 1u,
                          p.timeout_ns)) {
          if (lane == 0) atomicOr(p.fault, (unsigned)kFaultDrainWait);
          break;
        }
    }
  } else {
    // ------------------------------------------------ folders, then epilogue (both CTAs)
    const int q = warp & 3;                          // TMEM lane quarter this warp may access
    const int half = (warp - kFirstFoldWarp) >> 2;   // which 64 accumulator columns
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * half);
    float2 master2[32];  // columns 2e, 2e+1 of the thread's 64
#pragma unroll
    for (int e = 0; e < 32; ++e) master2[e] = make_float2(0.0f, 0.0f);
    bool ok = true;
    int u = 0;  // accumulator sequence number (one per K tile)
    for (int sgi = 0; ok && sgi < work_s.nseg; ++sgi) {
      int len;
      {
        const Segment g = cta_segment(p, work_s, cl, sgi, kt_total);
        len = g.ke - g.kb;
      }
      for (int i = 0; i < len; ++i, ++u) {
        const int b = u % kAccBufs;
        if (!warp_wait(smem_addr(&acc_full[b]), (uint32_t)(u / kAccBufs) & 1u, p.timeout_ns)) {
          ok = false;
          if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
          break;
        }
        tmem_fence_after_sync();
        float v[4][16];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld16(tq + (uint32_t)b * kAccCols + 16u * c, v[c]);
        tmem_wait_ld();
        // the accumulator is in registers: hand it back to the issuer before adding
        tmem_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(smem_addr(&acc_empty[b]), 0);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tmem_ld_ready(v[c]);
#pragma unroll
          for (int e = 0; e < 8; ++e)  // round-to-nearest FP32 adds, two per instruction
            master2[8 * c + e] = __fadd2_rn(master2[8 * c + e], make_float2(v[c][2 * e], v[c][2 * e + 1]));
        }
      }
      if (!ok) break;
      // epilogue of this segment: this thread holds row 32q + lane of the CTA's 128 rows, columns
      // 64*half .. +63 of the tile
      const Segment g = cta_segment(p, work_s, cl, sgi, kt_total);
      if (g.slot >= 0) {
        // partial sums of a shared stream-K tile -> this CTA's slot (whole 128 x 128, no bounds)
        const int64_t woff = (int64_t)(2 * g.slot + (int)rank) * (BMC * BN) + (32 * q + lane) * BN + 64 * half;
        float* w = p.ws + woff;
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (ws_ok(p, woff + 4 * e, 4))
            *reinterpret_cast<float4*>(w + 4 * e) =
                make_float4(master2[2 * e].x, master2[2 * e].y, master2[2 * e + 1].x, master2[2 * e + 1].y);
      } else {
        int prod, m0, n0;
        pair_tile_origin(p, g.tile, prod, m0, n0);
        const int row = m0 + BMC * (int)rank + 32 * q + lane;
        const int c0 = n0 + 64 * half;
        if (row < p.M) {
          repair_nans(p, prod, row, c0, master2);
          const int64_t roff = (int64_t)prod * p.stride_c + (int64_t)row * p.ldc;
          float* crow = p.C + roff;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
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
      for (int e = 0; e < 32; ++e) master2[e] = make_float2(0.0f, 0.0f);
    }
  }

  tmem_fence_before_sync();
  __syncthreads();
  // Bounded handshake of the two CTAs: neither releases its TMEM or exits while the other may
  // still arrive on its barriers or have MMAs read its shared memory and TMEM.
  if (threadIdx.x == 0) {
    mbar_arrive_remote(smem_addr(&fin), rank ^ 1u);
    if (!mbar_wait(smem_addr(&fin), 0u, p.timeout_ns)) atomicOr(p.fault, (unsigned)kFaultDrainWait);
  }
  __syncthreads();
  tmem_fence_after_sync();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// CTA (x, y) of the fixup grid: x = 2 j + r covers rows 128 r .. 128 r + 127 of
// stream-K pair tile j, rows 8y .. 8y+7 of those, one float4 of 4 columns per
// thread.  If several clusters shared tile j, C = alpha * (sum of their slots,
// in cluster order) + beta * C over the in-range elements; the order is fixed,
// so the result does not depend on scheduling.
constexpr int kFixupRowsPerCta = 8;
constexpr int kFixupThreads = 256;
constexpr int kMaxSharers = 256;  // clusters that may share one tile (the planner keeps to it)
template <bool CVEC>
__global__ void __launch_bounds__(kFixupThreads) pair_fixup_kernel(const GemmParams p) {
  __shared__ int s_n;
  __shared__ int s_slot[kMaxSharers];
  // The schedule and C's old values come first (fixup_prefetch_c); the grid is a programmatic
  // dependent of the GEMM kernel and waits for it only before reading the partial sums.
  const int kt = (p.K + BK - 1) / BK;
  const int j = (int)blockIdx.x >> 1, r = (int)blockIdx.x & 1;
  if (threadIdx.x == 0) {
    const int64_t i0 = (int64_t)j * kt;
    const int c0 = sk_owner(p, i0), c1 = sk_owner(p, i0 + kt - 1);
    s_n = min(c1 - c0 + 1, kMaxSharers);
    s_slot[0] = c0;
  }
  __syncthreads();
  const int n = s_n;
  if (n == 1) return;  // one cluster covered the whole tile and wrote C itself
  const int c0 = s_slot[0];
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kFixupThreads) s_slot[i] = 2 * sk_slot(p, c0 + i, j, kt) + r;
  __syncthreads();
  int prod, m0, n0;
  pair_tile_origin(p, p.sk_tile0 + j, prod, m0, n0);
  const int rr = (int)blockIdx.y * kFixupRowsPerCta + (int)(threadIdx.x >> 5);
  const int cc = (int)(threadIdx.x & 31) * 4;
  const int row = m0 + BMC * r + rr, col = n0 + cc;
  if (row >= p.M || col >= p.N) return;
  const FixupOut f = fixup_prefetch_c<CVEC>(p, prod, row, col);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float4 v = fixup_sum(p, s_slot, n, BMC * BN, (int64_t)rr * BN + cc);
  repair_nans4(p, prod, row, col, v);
  fixup_store<CVEC>(p, f, v);
}

}  // namespace tcp

namespace {

template <bool TA, bool TB>
cudaError_t pair_attrs() {
  return cudaFuncSetAttribute(tcp::pair_gemm_kernel<TA, TB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              tcp::kSmemBytes);
}

template <bool TA, bool TB>
cudaError_t pair_launch(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p, cudaStream_t stream) {
  // grid: p.sk_grid clusters of 2 CTAs (the cluster shape is the kernel's compile-time attribute)
  tcp::pair_gemm_kernel<TA, TB><<<2u * (unsigned)p.sk_grid, tcp::kThreads, tcp::kSmemBytes, stream>>>(mapA, mapB, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t prepare_tc_pair() {
  cudaError_t e = pair_attrs<false, false>();
  if (e == cudaSuccess) e = pair_attrs<false, true>();
  if (e == cudaSuccess) e = pair_attrs<true, false>();
  if (e == cudaSuccess) e = pair_attrs<true, true>();
  return e;
}

cudaError_t tc_pair_max_clusters(int* clusters) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(tcp::kThreads);
  cfg.dynamicSmemBytes = tcp::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, tcp::pair_gemm_kernel<false, false>, &cfg);
}

cudaError_t launch_tc_pair(bool transA, bool transB, const CUtensorMap& mapA, const CUtensorMap& mapB,
                           const GemmParams& p, cudaStream_t stream) {
  if (!transA && !transB) return pair_launch<false, false>(mapA, mapB, p, stream);
  if (!transA && transB) return pair_launch<false, true>(mapA, mapB, p, stream);
  if (transA && !transB) return pair_launch<true, false>(mapA, mapB, p, stream);
  return pair_launch<true, true>(mapA, mapB, p, stream);
}

cudaError_t launch_pair_fixup(const GemmParams& p, int sk_tiles, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * (unsigned)sk_tiles, tcp::BMC / tcp::kFixupRowsPerCta);
  cfg.blockDim = dim3(tcp::kFixupThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the GEMM kernel ends
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.c_vec ? cudaLaunchKernelEx(&cfg, tcp::pair_fixup_kernel<true>, p)
                 : cudaLaunchKernelEx(&cfg, tcp::pair_fixup_kernel<false>, p);
}

}  // namespace sgemm_impl
