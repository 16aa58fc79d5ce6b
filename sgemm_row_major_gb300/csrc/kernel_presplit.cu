// kernel_presplit.cu -- 3xTF32 SGEMM with the operands split once per call, for sm_103a.
//
// The tensor-core kernels in kernel_tf32x3.cu and kernel_tc_pair.cu split
// every operand tile into its TF32 hi part and FP32 lo part inside the
// GEMM, once per output tile that reads it: an A panel is split by every
// tile of its row, a B panel by every tile of its column, and measured on
// GB300 that splitting bounds those kernels (with the split work removed
// the CTA-pair kernel ran 28% faster).  Here a split pass writes each
// operand once as K-contiguous hi and lo arrays (the same rounding: hi = x
// rounded to TF32 to nearest with ties away, lo = x - hi exactly), and the
// GEMM loads hi and lo tiles with TMA and hands them to the tensor cores
// straight from shared memory: no splitter warps, no split stages.
//
// GEMM: 256 x 256 x 32 tiles on the two CTAs of a cluster with
// tcgen05.mma.cta_group::2.kind::tf32, M = 256, N = 256, K = 8, A and B
// both from shared memory (each CTA holds 128 rows of A hi/lo and 128 of
// the tile's 256 columns of B hi/lo).  Per SM and K step the tensor core
// reads 4 KB of A and 4 KB of B (each CTA's B half is read once for both
// SMs) in 128 cycles, and the TMA ring writes 64 KB per K tile: about 106 of
// the shared-memory path's 128 bytes per cycle at the tensor core's rate.
// Each CTA's TMEM holds two 128 x 256 FP32 accumulators (512 columns); a
// fresh one per 32-k tile is folded into FP32 registers by 8 folder warps,
// as in the other tensor-core kernels.  The persistent data-parallel +
// stream-K schedule of kernel_tc_common.cuh runs with the cluster as the
// unit; presplit_fixup_kernel adds the partial sums of shared tiles in
// cluster order.
//
// Launch chain of a call: split pass of A, split pass of B, GEMM, fixup.
// Each launch after the first is a programmatic dependent of the one before:
// the B pass starts once every block of the A pass has started and waits for
// that pass at its end; the GEMM's prologue (barriers, TMEM, tensor maps)
// runs while the B pass finishes and its producer waits for that pass before
// the first load; the fixup waits for the GEMM.  (A dependent grid starts
// only when every block of the grid before it has started or finished, so
// the early blocks cannot hold the SMs that later blocks of that grid need.)
//
// The pages name tensor cores and TF32 as the missing piece of their SGEMM
// (itan.pw "CUDA NVIDIA 4090 高性能計算", §4; youngju.dev "CUDA architecture
// visualized", テンソルコア).
//
// CTA roles (10 warps): warp 0 TMA producer (each CTA loads its own halves);
// warp 1 of the even CTA issues the pair's MMAs (both CTAs' TMA loads complete on
// the even CTA's stage barriers), warp 1 of the odd CTA waits for the last
// commits before that CTA leaves; warps 2-9 folders (lane
// quarter warp % 4, columns 128 * ((warp - 2) / 4) .. +127) and epilogue.
#include <algorithm>

#include <cuda_bf16.h>

#include "kernel_tc_common.cuh"

namespace sgemm_impl {
namespace tps {

using namespace tc;

// ------------------------------------------------------------------ split pass
// Splits op(X) for `products` products into hi and lo, written as rows of K
// contiguous floats (row stride ldk, product stride rows * ldk): element (r,
// k) of product p is src[p * stride + r * ld + k] when the stored rows run
// along K, src[p * stride + k * ld + r] otherwise (then the pass transposes
// through shared memory, 64 x 64 tiles).  Both forms are HBM streams; each
// thread loads 16 (transposing) or kSplitUnroll x 4 (rows) elements before it
// splits and stores any, so an SM keeps about 128 KB of loads in flight (with
// one load per thread, 32 KB, the passes ran at 3.0-4.6 TB/s).
constexpr int kSplitTile = 64;
constexpr int kSplitUnroll = 4;
constexpr int kSplitSegChunks = 32 * kSplitUnroll;  // 4-float chunks one warp takes per row segment

__device__ __forceinline__ void split_one(float x, float& hi, float& lo) {
  hi = tf32_round(x);
  lo = __fmaf_rn(hi, -1.0f, x);  // exact: x - hi
}

// The hi part alone is the TF32 rounding of x, except for a NaN: the tensor core reads only the
// top 19 bits of a value, so a NaN whose payload lies in the 13 dropped fraction bits would reach
// it as +-Inf (with the add-and-mask, or as stored).  Every NaN becomes a quiet NaN with all
// payload bits set.  (With the lo part as well, lo = NaN carries it.)
__device__ __forceinline__ float keep_nan(float x, float hi) { return x != x ? __uint_as_float(0x7FFFFFFFu) : hi; }

// Stores of the hi part.  float: the TF32 hi of x (3xTF32, with lo) or its NaN-keeping form (hi
// only); __nv_bfloat16 (the BF16-input GEMM, hi only, lo == nullptr): x rounded to BF16, to
// nearest even (cvt.rn.bf16.f32: NaN stays NaN, a rounding past the largest BF16 value gives Inf).
__device__ __forceinline__ void store_hi(float* h, float x, float xh, bool with_lo) { *h = with_lo ? xh : keep_nan(x, xh); }
__device__ __forceinline__ void store_hi(__nv_bfloat16* h, float x, float, bool) { *h = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store_hi4(float* h, float4 x, float4 xh, bool with_lo) {
  if (!with_lo) xh = make_float4(keep_nan(x.x, xh.x), keep_nan(x.y, xh.y), keep_nan(x.z, xh.z), keep_nan(x.w, xh.w));
  *reinterpret_cast<float4*>(h) = xh;
}
__device__ __forceinline__ void store_hi4(__nv_bfloat16* h, float4 x, float4, bool) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&a);
  u.y = *reinterpret_cast<const uint32_t*>(&b);
  *reinterpret_cast<uint2*>(h) = u;  // 8-byte aligned: row strides are multiples of 8 elements
}

// Rows run along K: each thread takes 4 consecutive k (16-byte stores; 16-byte loads when
// VEC -- every source row 16-byte aligned -- else four 4-byte loads; K % 4 == 0 is not
// required: the tail is scalar).  lo == nullptr: only hi is written (the rounding pass of the
// TF32-input GEMM).
// (Chk: the bounds checks of the debug build on the source (extent src_elems) and on the split
// arrays (products * rows * ldk elements each).)
struct SplitChk {
  unsigned* fault;
  unsigned long long* word;
  int64_t src_elems, dst_elems;
  __device__ __forceinline__ bool src(int64_t off, int64_t n) const {
    return in_range(fault, word, kSiteA, off, n, src_elems);
  }
  __device__ __forceinline__ bool dst(int64_t off, int64_t n) const {
    return in_range(fault, word, kSiteSplit, off, n, dst_elems);
  }
};

// Launch order of a call's split passes and GEMM (programmatic dependent launches): the first
// split pass lets the next one start at once (`trigger`); a split pass launched as a dependent
// waits at its end for the pass before it, so its grid completes after that one; the GEMM,
// launched as a dependent of the last pass, waits for it before its first load of split data.
__device__ __forceinline__ void split_pass_begin(bool trigger) {
  if (trigger) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void split_pass_end() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Rows run along K.  Work unit: a segment of kSplitSegChunks 4-float chunks of one row, taken by
// one warp, lane l the chunks l, l + 32, l + 64, l + 96 of it (each load instruction of the warp
// reads 512 contiguous bytes); the last segment of a row also takes its tail of K % 4 elements.
// VEC: every source row 16-byte aligned (16-byte loads), else four 4-byte loads per chunk.
template <bool VEC, typename OutT>
__global__ void __launch_bounds__(256) split_rows_kernel(const float* __restrict__ src, int64_t ld, int64_t stride,
                                                         int rows, int K, int products, OutT* __restrict__ hi,
                                                         float* __restrict__ lo, int64_t ldk, const SplitChk chk,
                                                         bool trigger) {
  split_pass_begin(trigger);
  const int lane = (int)threadIdx.x & 31;
  const int kfull = K / 4;  // chunks of 4 whole k
  const int nseg = max(1, (kfull + kSplitSegChunks - 1) / kSplitSegChunks);
  const int64_t units = (int64_t)products * rows * nseg;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t u = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); u < units; u += warps) {
    const int64_t pr = u / nseg;  // product * rows + row
    const int sg = (int)(u - pr * nseg);
    const int64_t p = pr / rows, r = pr - p * rows;
    const int64_t so = p * stride + r * ld;
    const float* s = src + so;
    OutT* h = hi + pr * ldk;
    float* l = lo ? lo + pr * ldk : nullptr;
    float4 x[kSplitUnroll];
    bool ok[kSplitUnroll];
#pragma unroll
    for (int j = 0; j < kSplitUnroll; ++j) {
      const int c = sg * kSplitSegChunks + 32 * j + lane;
      ok[j] = c < kfull && chk.src(so + 4 * c, 4) && chk.dst(pr * ldk + 4 * c, 4);
      x[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (ok[j])
        x[j] = VEC ? *reinterpret_cast<const float4*>(s + 4 * c) : make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2],
                                                                              s[4 * c + 3]);
    }
#pragma unroll
    for (int j = 0; j < kSplitUnroll; ++j) {
      if (!ok[j]) continue;
      const int c = sg * kSplitSegChunks + 32 * j + lane;
      float4 xh, xl;
      split4(x[j], xh, xl);
      if (l) *reinterpret_cast<float4*>(l + 4 * c) = xl;
      store_hi4(h + 4 * c, x[j], xh, l != nullptr);
    }
    const int kt = 4 * kfull + lane;  // the tail: fewer than 4 elements
    if (sg == nseg - 1 && kt < K && chk.src(so + kt, 1) && chk.dst(pr * ldk + kt, 1)) {
      float xh, xl;
      split_one(s[kt], xh, xl);
      store_hi(h + kt, s[kt], xh, l != nullptr);
      if (l) l[kt] = xl;
    }
  }
  split_pass_end();
}

// Stored rows run along the other axis: a 64 x 64 block per CTA (32 x 8 threads, 16 elements
// each), read along the stored rows (any alignment), written along K; lo == nullptr: hi only.
template <typename OutT>
__global__ void __launch_bounds__(256) split_transpose_kernel(const float* __restrict__ src, int64_t ld,
                                                              int64_t stride, int rows, int K,
                                                              OutT* __restrict__ hi, float* __restrict__ lo,
                                                              int64_t ldk, const SplitChk chk, bool trigger) {
  split_pass_begin(trigger);
  __shared__ float tile[kSplitTile][kSplitTile + 1];
  const int p = (int)blockIdx.z;
  const int r0 = (int)blockIdx.x * kSplitTile, k0 = (int)blockIdx.y * kSplitTile;
  const int tx = (int)threadIdx.x, ty = (int)threadIdx.y;
  const float* s = src + (int64_t)p * stride;
  // read: stored row k = k0 + ty + j, element r = r0 + tx + c; all 16 loads before any store
  constexpr int kReads = (kSplitTile / 8) * (kSplitTile / 32);
  float v[kReads];
#pragma unroll
  for (int i = 0; i < kReads; ++i) {
    const int j = 8 * (i >> 1), c = 32 * (i & 1);
    const int k = k0 + ty + j, r = r0 + tx + c;
    const int64_t so = (int64_t)k * ld + r;
    v[i] = 0.0f;
    if (k < K && r < rows && chk.src((int64_t)p * stride + so, 1)) v[i] = s[so];
  }
#pragma unroll
  for (int i = 0; i < kReads; ++i) tile[ty + 8 * (i >> 1)][tx + 32 * (i & 1)] = v[i];
  __syncthreads();
  // write: row r = r0 + ty + j, k = k0 + tx + c
  OutT* h = hi + (int64_t)p * rows * ldk;
  float* l = lo ? lo + (int64_t)p * rows * ldk : nullptr;
#pragma unroll
  for (int j = 0; j < kSplitTile; j += 8)
#pragma unroll
    for (int c = 0; c < kSplitTile; c += 32) {
      const int r = r0 + ty + j, k = k0 + tx + c;
      if (r < rows && k < K && chk.dst(((int64_t)p * rows + r) * ldk + k, 1)) {
        const float x = tile[tx + c][ty + j];
        float xh, xl;
        split_one(x, xh, xl);
        store_hi(h + (int64_t)r * ldk + k, x, xh, lo != nullptr);
        if (lo) l[(int64_t)r * ldk + k] = xl;
      }
    }
  split_pass_end();
}

// ------------------------------------------------------------------ GEMM
constexpr int BM = 256;                   // rows of a pair tile
constexpr int BMC = 128;                  // rows one CTA covers
constexpr int BN = 256;                   // columns of a pair tile
constexpr int BNC = 128;                  // columns of B one CTA loads
constexpr int BK = 32;
constexpr int kPartBytes = 128 * BK * 4;  // 16 KB: 128 rows (or columns) x 32 k, K-major, 128-byte swizzle
// PARTS = 2: 3xTF32 (a stage holds A hi, A lo, B hi, B lo); PARTS = 1: TF32 inputs (A hi, B hi:
// one tensor-core product per k).  The stages fill shared memory (3xTF32 at 4096^3: three
// stages 267 TFLOPS; two stages 212; six 16-k stages with a 64-byte swizzle 247, their barrier,
// commit and relay traffic doubled).
template <int PARTS>
struct Cfg {
  static constexpr int kStages = PARTS == 2 ? 3 : 6;
  // K tiles summed in one TMEM accumulator before the folders add it into FP32 registers (the
  // tensor core's FP32 accumulation drifts with the number of products it adds; kernel_tf32x3.cu):
  // 3xTF32 12 products (4 k-steps x 3), the count the fold was sized for; one product per term
  // (TF32 or BF16 inputs) 24 (6 K tiles x 4 k-steps).  Measured at 4096^3 against the
  // rounded-input oracle, relative Frobenius error and TFLOPS for TF32 / BF16 inputs: 12 products
  // 2.8e-7, 479 / 1.7e-7, 708; 24 products 4.9e-7, 522 / 2.9e-7, 763; 48 products 9.2e-7, 555 /
  // 6.0e-7, 819 (too close to the 1e-6 gate for TF32).
  static constexpr int kFoldTiles = PARTS == 2 ? 1 : 6;
  static constexpr int kStageBytes = 2 * PARTS * kPartBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static_assert(kSmemBytes + 1024 <= 232448, "shared memory per CTA");
};
constexpr int kStages = Cfg<2>::kStages;
constexpr int kStageBytes = Cfg<2>::kStageBytes;
constexpr int kSmemBytes = Cfg<2>::kSmemBytes;
constexpr int kFoldWarps = 8;             // warps 2-9
constexpr int kThreads = 32 * (2 + kFoldWarps);
constexpr int kAccBufs = 2;
constexpr uint32_t kAccCols = 256;        // one 128 x 256 FP32 accumulator per CTA
constexpr uint32_t kTmemCols = 512;
constexpr int kFoldCols = 128;            // accumulator columns a folder thread owns
constexpr int kFoldChunk = 32;            // columns loaded per round trip (register budget; 64 measured slower)
static_assert(kAccBufs * kAccCols <= kTmemCols, "accumulators must fit in TMEM");

// tcgen05 instruction descriptor, kind::tf32: FP32 accumulator, TF32 A and B,
// both K-major, N = 256, M = 256 (the pair).
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

// ... and kind::f16 with BF16 A and B (the BF16-input GEMM): FP32 accumulator, both K-major,
// N = 256, M = 256; K = 16 per MMA, the same 32 bytes of a K-major row as 8 TF32 values.
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                ((uint32_t)(BM >> 4) << 24);

// D (both CTAs' TMEM) = or += A (128 rows in each CTA's shared memory) * B (128 columns in each
// CTA's shared memory); both operands K-major, described by the same descriptors in both CTAs.
__device__ __forceinline__ void mma_pair_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_pair_ss_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(kIdescBf16), "r"(accumulate)
      : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// the barrier `bar_cluster` (a shared::cluster address: this CTA's or its
// peer's barrier).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t inner, int32_t outer, int32_t product) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(inner), "r"(outer), "r"(product)
      : "memory");
}

// Product and origin of pair tile `tile`.
__device__ __forceinline__ void pair_tile_origin(const GemmParams& p, int tile, int& prod, int& m0, int& n0) {
  tile_origin_of(p, tile, BM, BN, prod, m0, n0);
}

// Tensor maps: the split operands as {K, rows, products} with boxes {32, 128, 1}, 128-byte
// swizzle; za / zb in GemmParams say whether the third coordinate is the product index.
template <bool CVEC>
__device__ __forceinline__ void store_row(const GemmParams& p, int64_t roff, int c0, const float2 (&m)[kFoldCols / 2]) {
  float* crow = p.C + roff;
#pragma unroll
  for (int e = 0; e < kFoldCols / 4; ++e) {
    const int col = c0 + 4 * e;
    const float x[4] = {m[2 * e].x, m[2 * e].y, m[2 * e + 1].x, m[2 * e + 1].y};
    if (col >= p.N || !c_ok(p, roff + col, min(4, p.N - col))) continue;
    if (CVEC && col + 3 < p.N) {
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

// BF16 (with PARTS == 1): the split arrays hold BF16 values, 64 per 128-byte row of a tile, so a
// K tile is 64 deep and its 4 k-steps are kind::f16 MMAs of K = 16.
template <int PARTS, bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    presplit_gemm_kernel(const __grid_constant__ CUtensorMap mapAh, const __grid_constant__ CUtensorMap mapAl,
                         const __grid_constant__ CUtensorMap mapBh, const __grid_constant__ CUtensorMap mapBl,
                         const GemmParams p) {
  constexpr int kStages = Cfg<PARTS>::kStages;
  constexpr int kStageBytes = Cfg<PARTS>::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ __align__(8) uint64_t acc_full[kAccBufs], acc_empty[kAccBufs];
  __shared__ __align__(8) uint64_t fin;
  __shared__ uint32_t tmem_slot;
  __shared__ CtaWork work_s;

  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;  // the same in both CTAs (same kernel)
  const uint32_t sbase = raw_addr + pad;
  // stage s: [A hi][A lo][B hi][B lo] (PARTS = 1: [A hi][B hi]), 16 KB each, 1024-byte aligned
  auto part = [&](int s, int which) { return sbase + (uint32_t)(s * kStageBytes + which * kPartBytes); };
  constexpr int kAhi = 0, kAlo = 1, kBhi = PARTS, kBlo = PARTS + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const int cl = (int)cluster_id_x();
  constexpr int kKTile = BF16 ? 2 * BK : BK;  // K elements per K tile (one 128-byte row of a tile)
  static_assert(!BF16 || PARTS == 1, "the BF16-input GEMM has one part per operand");
  const int kt_total = (p.K + kKTile - 1) / kKTile;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (threadIdx.x == 0) {
    work_s = cta_work(p, cl, kt_total);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&empty[s]), 1);
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
      prefetch_tensormap(&mapAh);
      prefetch_tensormap(&mapAl);
      prefetch_tensormap(&mapBh);
      prefetch_tensormap(&mapBl);
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the split passes' arrays are complete
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
          const int s = t % kStages;
          if (t >= kStages &&
              !mbar_wait(smem_addr(&empty[s]), (uint32_t)((t / kStages) - 1) & 1u, p.timeout_ns)) {
            atomicOr(p.fault, (unsigned)kFaultEmptyWait);
            ok = false;
            break;
          }
          const int k0 = kt * kKTile;
          // both CTAs' loads complete on the even CTA's barrier, which expects all their bytes
          // (measured: 270.1 TFLOPS at 4096^3, 268.3 with the odd CTA's completions relayed by a
          // thread's remote arrive)
          const uint32_t fb = map_to_rank(smem_addr(&full[s]), 0);
          if (rank == 0) mbar_arrive_expect_tx(smem_addr(&full[s]), 2u * (uint32_t)kStageBytes);
          tma_load_3d_pair(part(s, kAhi), &mapAh, fb, k0, m0, za);
          if (PARTS == 2) tma_load_3d_pair(part(s, kAlo), &mapAl, fb, k0, m0, za);
          tma_load_3d_pair(part(s, kBhi), &mapBh, fb, k0, n0, zb);
          if (PARTS == 2) tma_load_3d_pair(part(s, kBlo), &mapBl, fb, k0, n0, zb);
          issued = t + 1;
        }
      }
      // leave only when every copy into shared memory has landed (the odd CTA cannot see its
      // copies land: its warp 1 waits for the MMAs that read the last stages)
      if (rank == 0)
        for (int t = issued > kStages ? issued - kStages : 0; t < issued; ++t)
          if (!mbar_wait(smem_addr(&full[t % kStages]), (uint32_t)(t / kStages) & 1u, p.timeout_ns))
            atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank != 0) {
      // ---------------------------------------------- odd CTA: the issuer's last commits on the
      // stages land in this CTA (and imply its last copies have landed): wait for them
      bool ok = true;
      for (int u = nkt > kStages ? nkt - kStages : 0; ok && u < nkt; ++u)
        ok = mbar_wait(smem_addr(&empty[u % kStages]), (uint32_t)(u / kStages) & 1u, p.timeout_ns);
      if (!ok) atomicOr(p.fault, (unsigned)kFaultFullWait);
    } else if (lane == 0) {
      // ---------------------------------------------- MMA issuer (even CTA)
      // K tile t of the CTA's sequence uses stage t % kStages; chunk c (up to kFoldTiles K tiles of
      // one segment) accumulates in accumulator c % kAccBufs
      constexpr int kFold = Cfg<PARTS>::kFoldTiles;
      bool ok = true;
      int t = 0, c = 0, t_done = -1, c_done = -1;
      const CtaWork work = work_s;
      for (int sgi = 0; ok && sgi < work.nseg; ++sgi) {
        const Segment g = cta_segment(p, work, cl, sgi, kt_total);
        for (int i0 = g.kb; ok && i0 < g.ke; i0 += kFold, ++c) {
          const int n = min(kFold, g.ke - i0);
          const int b = c % kAccBufs;
          if (c >= kAccBufs &&
              !mbar_wait(smem_addr(&acc_empty[b]), (uint32_t)((c / kAccBufs) - 1) & 1u, p.timeout_ns)) {
            ok = false;
            break;
          }
          const uint32_t acc = tmem + (uint32_t)b * kAccCols;
          for (int j = 0; j < n; ++j, ++t) {
            const int s = t % kStages;
            if (!mbar_wait(smem_addr(&full[s]), (uint32_t)(t / kStages) & 1u, p.timeout_ns)) {
              ok = false;
              break;
            }
            tmem_fence_after_sync();
            const uint64_t ahi = kmajor_sw128_desc(part(s, kAhi)), bhi = kmajor_sw128_desc(part(s, kBhi));
#pragma unroll
            for (int ks = 0; ks < BK / 8; ++ks) {
              const uint64_t step = (uint64_t)(ks * 32) >> 4;  // 8 TF32 = 32 bytes along K
              const uint32_t fresh = (j == 0 && ks == 0) ? 0u : 1u;  // a fresh accumulator per chunk
              if (PARTS == 2) {
                const uint64_t alo = kmajor_sw128_desc(part(s, kAlo)), blo = kmajor_sw128_desc(part(s, kBlo));
                mma_pair_ss(acc, alo + step, bhi + step, fresh);
                mma_pair_ss(acc, ahi + step, blo + step, 1u);
                mma_pair_ss(acc, ahi + step, bhi + step, 1u);
              } else if (BF16) {
                mma_pair_ss_bf16(acc, ahi + step, bhi + step, fresh);
              } else {
                mma_pair_ss(acc, ahi + step, bhi + step, fresh);
              }
            }
            mma_commit_pair(smem_addr(&empty[s]));  // stage s reusable in both CTAs
            t_done = t;
          }
          if (!ok) break;
          mma_commit_pair(smem_addr(&acc_full[b]));  // accumulator b (both CTAs) holds chunk c
          c_done = c;
        }
      }
      if (!ok) atomicOr(p.fault, (unsigned)kFaultFullWait);
      // leave only when every MMA has completed and its commits have landed here
      for (int u = t_done + 1 > kStages ? t_done + 1 - kStages : 0; u <= t_done; ++u)
        if (!mbar_wait(smem_addr(&empty[u % kStages]), (uint32_t)(u / kStages) & 1u, p.timeout_ns))
          atomicOr(p.fault, (unsigned)kFaultDrainWait);
      if (c_done >= 0 &&
          !mbar_wait(smem_addr(&acc_full[c_done % kAccBufs]), (uint32_t)(c_done / kAccBufs) & 1u, p.timeout_ns))
        atomicOr(p.fault, (unsigned)kFaultDrainWait);
    }
  } else {
    // ------------------------------------------------ folders, then epilogue (both CTAs)
    const int q = warp & 3;                     // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;           // which 128 accumulator columns
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kFoldCols * half);
    float2 master2[kFoldCols / 2];
#pragma unroll
    for (int e = 0; e < kFoldCols / 2; ++e) master2[e] = make_float2(0.0f, 0.0f);
    bool ok = true;
    int u = 0;
    for (int sgi = 0; ok && sgi < work_s.nseg; ++sgi) {
      int len;
      {
        const Segment g = cta_segment(p, work_s, cl, sgi, kt_total);
        len = g.ke - g.kb;
      }
      for (int i = 0; i < len; i += Cfg<PARTS>::kFoldTiles, ++u) {  // chunk u: as the issuer's chunks
        const int b = u % kAccBufs;
        if (!warp_wait(smem_addr(&acc_full[b]), (uint32_t)(u / kAccBufs) & 1u, p.timeout_ns)) {
          ok = false;
          if (lane == 0) atomicOr(p.fault, (unsigned)kFaultFullWait);
          break;
        }
        tmem_fence_after_sync();
#pragma unroll
        for (int ch = 0; ch < kFoldCols / kFoldChunk; ++ch) {
          float v[kFoldChunk / 16][16];
#pragma unroll
          for (int c = 0; c < kFoldChunk / 16; ++c)
            tmem_ld16(tq + (uint32_t)b * kAccCols + (uint32_t)(kFoldChunk * ch + 16 * c), v[c]);
          tmem_wait_ld();
          if (ch == kFoldCols / kFoldChunk - 1) {
            // the whole accumulator is in registers or folded: hand it back to the issuer
            tmem_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(smem_addr(&acc_empty[b]), 0);
          }
#pragma unroll
          for (int c = 0; c < kFoldChunk / 16; ++c) {
            tmem_ld_ready(v[c]);
#pragma unroll
            for (int e = 0; e < 8; ++e) {  // round-to-nearest FP32 adds, two per instruction
              float2& m = master2[(kFoldChunk * ch + 16 * c) / 2 + e];
              m = __fadd2_rn(m, make_float2(v[c][2 * e], v[c][2 * e + 1]));
            }
          }
        }
      }
      if (!ok) break;
      // epilogue: this thread holds row 32q + lane of the CTA's 128 rows, columns 128*half .. +127
      const Segment g = cta_segment(p, work_s, cl, sgi, kt_total);
      if (g.slot >= 0) {
        const int64_t woff =
            (int64_t)(2 * g.slot + (int)rank) * (BMC * BN) + (32 * q + lane) * BN + kFoldCols * half;
        float* w = p.ws + woff;
#pragma unroll
        for (int e = 0; e < kFoldCols / 4; ++e)
          if (ws_ok(p, woff + 4 * e, 4))
            *reinterpret_cast<float4*>(w + 4 * e) =
                make_float4(master2[2 * e].x, master2[2 * e].y, master2[2 * e + 1].x, master2[2 * e + 1].y);
      } else {
        int prod, m0, n0;
        pair_tile_origin(p, g.tile, prod, m0, n0);
        const int row = m0 + BMC * (int)rank + 32 * q + lane;
        if (row < p.M) {
          if (PARTS == 2) repair_nans(p, prod, row, n0 + kFoldCols * half, master2);
          const int64_t roff = (int64_t)prod * p.stride_c + (int64_t)row * p.ldc;
          if (p.c_vec) store_row<true>(p, roff, n0 + kFoldCols * half, master2);
          else         store_row<false>(p, roff, n0 + kFoldCols * half, master2);
        }
      }
#pragma unroll
      for (int e = 0; e < kFoldCols / 2; ++e) master2[e] = make_float2(0.0f, 0.0f);
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
// stream-K pair tile j, rows 8y .. 8y+7 of those, two float4s of 4 columns
// per thread (columns 4 * lane and 128 + 4 * lane).  If several clusters
// shared tile j, C = alpha * (sum of their slots, in cluster order) + beta * C
// over the in-range elements.
constexpr int kFixupRowsPerCta = 8;
constexpr int kFixupThreads = 256;
constexpr int kMaxSharers = 256;
template <bool CVEC>
__global__ void __launch_bounds__(kFixupThreads) presplit_fixup_kernel(const GemmParams p, int k_tile) {
  __shared__ int s_n;
  __shared__ int s_slot[kMaxSharers];
  // The schedule and C's old values come first (fixup_prefetch_c); the grid is a programmatic
  // dependent of the GEMM kernel and waits for it only before reading the partial sums.
  const int kt = (p.K + k_tile - 1) / k_tile;  // the GEMM's K tiles (32, or 64 for BF16 inputs)
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
  const int row = m0 + BMC * r + rr;
  if (row >= p.M) return;
  FixupOut f[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int col = n0 + 128 * h + (int)(threadIdx.x & 31) * 4;
    f[h].cp = nullptr;
    if (col < p.N) f[h] = fixup_prefetch_c<CVEC>(p, prod, row, col);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int cc = 128 * h + (int)(threadIdx.x & 31) * 4;
    const int col = n0 + cc;
    if (col >= p.N) continue;
    float4 v = fixup_sum(p, s_slot, n, BMC * BN, (int64_t)rr * BN + cc);
    if (p.repair) repair_nans4(p, prod, row, col, v);
    fixup_store<CVEC>(p, f[h], v);
  }
}

}  // namespace tps

cudaError_t prepare_presplit() {
  cudaError_t e = cudaFuncSetAttribute(tps::presplit_gemm_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       tps::Cfg<2>::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tps::presplit_gemm_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tps::Cfg<1>::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(tps::presplit_gemm_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             tps::Cfg<1>::kSmemBytes);
  return e;
}

namespace {
template <typename OutT>
cudaError_t launch_split_pass(const float* src, int64_t ld, int64_t stride, bool k_contig, int rows, int K,
                              int products, OutT* hi, float* lo, int64_t ldk, int sm_count, cudaStream_t stream,
                              unsigned* fault, unsigned long long* bounds, int64_t src_elems, SplitOrder order) {
  if (rows <= 0 || K <= 0 || products <= 0) return cudaSuccess;
  const tps::SplitChk chk{fault, bounds, src_elems, (int64_t)products * rows * ldk};
  cudaLaunchConfig_t cfg = {};
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = order == SplitOrder::kDependent ? 1 : 0;
  const bool trigger = order == SplitOrder::kFirst;
  if (k_contig) {
    // one warp per row segment, at most 64 warps per SM (8 CTAs of 256 threads), row-segment loop
    const int64_t nseg = std::max<int64_t>(1, ((K / 4) + tps::kSplitSegChunks - 1) / tps::kSplitSegChunks);
    const int64_t warps = std::min<int64_t>((int64_t)products * rows * nseg, (int64_t)sm_count * 64);
    cfg.gridDim = dim3((unsigned)std::max<int64_t>((warps + 7) / 8, 1));
    cfg.blockDim = dim3(256);
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15u) == 0 && ld % 4 == 0 && (products == 1 || stride % 4 == 0);
    return vec ? cudaLaunchKernelEx(&cfg, tps::split_rows_kernel<true, OutT>, src, ld, stride, rows, K, products, hi,
                                    lo, ldk, chk, trigger)
               : cudaLaunchKernelEx(&cfg, tps::split_rows_kernel<false, OutT>, src, ld, stride, rows, K, products, hi,
                                    lo, ldk, chk, trigger);
  }
  cfg.gridDim = dim3((unsigned)((rows + tps::kSplitTile - 1) / tps::kSplitTile),
                     (unsigned)((K + tps::kSplitTile - 1) / tps::kSplitTile), (unsigned)products);
  cfg.blockDim = dim3(32, 8);  // 32 x 8 threads, 16 elements each
  return cudaLaunchKernelEx(&cfg, tps::split_transpose_kernel<OutT>, src, ld, stride, rows, K, hi, lo, ldk, chk,
                            trigger);
}
}  // namespace

cudaError_t launch_split_operand(const float* src, int64_t ld, int64_t stride, bool k_contig, int rows, int K,
                                 int products, float* hi, float* lo, int64_t ldk, int sm_count, cudaStream_t stream,
                                 unsigned* fault, unsigned long long* bounds, int64_t src_elems, SplitOrder order) {
  return launch_split_pass<float>(src, ld, stride, k_contig, rows, K, products, hi, lo, ldk, sm_count, stream, fault,
                                  bounds, src_elems, order);
}

cudaError_t launch_round_bf16(const float* src, int64_t ld, bool k_contig, int rows, int K, void* out, int64_t ldk,
                              int sm_count, cudaStream_t stream, unsigned* fault, unsigned long long* bounds,
                              int64_t src_elems, SplitOrder order) {
  return launch_split_pass<__nv_bfloat16>(src, ld, 0, k_contig, rows, K, 1, static_cast<__nv_bfloat16*>(out),
                                          nullptr, ldk, sm_count, stream, fault, bounds, src_elems, order);
}

namespace {
// The GEMM after the split passes: a programmatic dependent launch (its prologue overlaps the
// last pass; its producer waits for that pass before the first load).
template <int PARTS, bool BF16>
cudaError_t launch_gemm_after_split(const CUtensorMap& mapAh, const CUtensorMap& mapAl, const CUtensorMap& mapBh,
                                    const CUtensorMap& mapBl, const GemmParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * (unsigned)p.sk_grid);
  cfg.blockDim = dim3(tps::kThreads);
  cfg.dynamicSmemBytes = tps::Cfg<PARTS>::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tps::presplit_gemm_kernel<PARTS, BF16>, mapAh, mapAl, mapBh, mapBl, p);
}
}  // namespace

cudaError_t launch_presplit_gemm(const CUtensorMap& mapAh, const CUtensorMap& mapAl, const CUtensorMap& mapBh,
                                 const CUtensorMap& mapBl, const GemmParams& p, cudaStream_t stream) {
  return launch_gemm_after_split<2, false>(mapAh, mapAl, mapBh, mapBl, p, stream);
}

cudaError_t launch_tf32_gemm(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p,
                             cudaStream_t stream) {
  // (the lo maps are not read with one part)
  return launch_gemm_after_split<1, false>(mapA, mapA, mapB, mapB, p, stream);
}

cudaError_t launch_bf16_gemm(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p,
                             cudaStream_t stream) {
  return launch_gemm_after_split<1, true>(mapA, mapA, mapB, mapB, p, stream);
}

cudaError_t launch_presplit_fixup(const GemmParams& p, int sk_tiles, cudaStream_t stream, int k_tile) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * (unsigned)sk_tiles, tps::BMC / tps::kFixupRowsPerCta);
  cfg.blockDim = dim3(tps::kFixupThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the GEMM kernel ends
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return p.c_vec ? cudaLaunchKernelEx(&cfg, tps::presplit_fixup_kernel<true>, p, k_tile)
                 : cudaLaunchKernelEx(&cfg, tps::presplit_fixup_kernel<false>, p, k_tile);
}

}  // namespace sgemm_impl
