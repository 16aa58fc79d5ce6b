// api.cu -- the C ABI of libsgemm: argument checks, the variant planner,
// TMA descriptor encoding, workspace management and kernel launches.
//
// Argument conventions are those of BLAS/CBLAS row-major SGEMM (the pages
// give only the formula: itan.pw "CUDA NVIDIA 4090 高性能計算", 概要); error
// checking after each CUDA call follows youngju.dev "CUDA architecture
// visualized" (よくある落とし穴 6, cudaGetLastError).
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "kernel_small.h"
#include "kernel_tma.cuh"
#include "sgemm.h"
#include "sgemm_internal.h"

using namespace sgemm_impl;

namespace sgemm_impl {

int record_cuda_failure(cudaError_t e) {
  t_last_cuda_error_slot() = (int)e;
  return SGEMM_ERR_CUDA;
}

uint64_t wait_timeout_ns() {
  static const uint64_t ns = [] {
    const char* env = std::getenv("SGEMM_WAIT_TIMEOUT_MS");
    long long ms = env ? std::atoll(env) : 2000;
    if (ms < 1) ms = 1;
    return (uint64_t)ms * 1000000ull;
  }();
  return ns;
}

int& t_last_cuda_error_slot() {
  thread_local int slot = 0;
  return slot;
}

int pair_clusters_or_none() {
  int n = 0;
  if (tc_pair_max_clusters(&n) != cudaSuccess) {
    (void)cudaGetLastError();  // the failed query must not surface at a later launch check
    return 0;
  }
  return n > 0 ? n : 0;
}

}  // namespace sgemm_impl

namespace {

constexpr int kMaxDevices = 64;

std::atomic<int> g_override_variant{SGEMM_VARIANT_AUTO};
std::atomic<int> g_override_split{0};

struct DeviceState {
  std::mutex init_mutex;
  std::atomic<bool> ready{false};  // set once the set-up below has succeeded (a failed one is retried)
  int sm_count = 0;
  int pair_clusters = 0;  // co-resident clusters of the CTA-pair kernel; 0: pairs cannot run here
  unsigned* fault = nullptr;
  unsigned long long* bounds = nullptr;  // debug build: first bounds violation
  cudaMemPool_t pool = nullptr;
};
DeviceState g_devices[kMaxDevices];

int cuda_fail(cudaError_t e) { return record_cuda_failure(e); }

int op_code(char t) {
  if (t == 'N' || t == 'n') return 0;
  if (t == 'T' || t == 't' || t == 'C' || t == 'c') return 1;
  return -1;
}

// Per-device state: SM count, fault word address, kernel attributes, the
// co-resident CTA-pair clusters and the stream-ordered pool the workspace comes
// from.  Set up by the first call on the device that succeeds in it; a failed
// set-up (e.g. a first call made during a stream capture) is tried again by the
// next call.
int device_state(int* device_out, DeviceState** st_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
  DeviceState& st = g_devices[dev];
  if (!st.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(st.init_mutex);
    if (!st.ready.load(std::memory_order_relaxed)) {
      cudaError_t err = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
      if (err == cudaSuccess) err = fault_word(&st.fault);
      if (err == cudaSuccess) err = bounds_word(&st.bounds);
      if (err == cudaSuccess) err = prepare_tma_op_nn();
      if (err == cudaSuccess) err = prepare_tma_op_nt();
      if (err == cudaSuccess) err = prepare_tma_op_tn();
      if (err == cudaSuccess) err = prepare_tma_op_tt();
      if (err == cudaSuccess) err = prepare_tf32x3();
      if (err == cudaSuccess) err = prepare_small_gemm();
      if (err == cudaSuccess) err = prepare_tc_pair();
      if (err == cudaSuccess) err = prepare_presplit();
      if (err == cudaSuccess) err = prepare_skinny();
      if (err == cudaSuccess) st.pair_clusters = pair_clusters_or_none();
      if (err == cudaSuccess && !st.pool) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        err = cudaMemPoolCreate(&pool, &props);
        if (err == cudaSuccess) {
          uint64_t keep = UINT64_MAX;  // keep freed workspace for the next call (sgemm_release_workspace trims)
          err = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
          if (err == cudaSuccess) st.pool = pool;
          else (void)cudaMemPoolDestroy(pool);
        }
      }
      if (err != cudaSuccess) return cuda_fail(err);
      st.ready.store(true, std::memory_order_release);
    }
  }
  *device_out = dev;
  *st_out = &st;
  return SGEMM_OK;
}

struct Problem {
  int ta, tb;
  int64_t M, N, K;
  float alpha, beta;
  const float* A;
  const float* B;
  const float* C;
  int64_t lda, ldb, ldc;
  int64_t stride_a = 0, stride_b = 0, stride_c = 0;  // strided batch (elements)
  int64_t batch = 1;
};

int validate(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
             int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc, Problem* pr) {
  const int ta = op_code(transA), tb = op_code(transB);
  if (ta < 0) return -1;
  if (tb < 0) return -2;
  if (M < 0) return -3;
  if (N < 0) return -4;
  if (K < 0) return -5;
  const bool work = M > 0 && N > 0;
  const bool reads_ab = work && K > 0 && alpha != 0.0f;
  if (reads_ab && !A) return -7;
  if (lda < std::max<int64_t>(1, ta ? M : K)) return -8;
  if (reads_ab && !B) return -9;
  if (ldb < std::max<int64_t>(1, tb ? K : N)) return -10;
  if (work && !C) return -12;
  if (ldc < std::max<int64_t>(1, N)) return -13;
  *pr = Problem{ta, tb, M, N, K, alpha, beta, A, B, C, lda, ldb, ldc};
  return SGEMM_OK;
}

// Extra checks of a strided batch (argument indices of sgemm_strided_batched:
// 14 strideA, 15 strideB, 16 strideC, 17 batch_count).  Strides may be 0
// (one matrix shared by every product) or let A and B matrices overlap, but
// the C matrices of different products must not overlap.
int validate_batch(int64_t stride_a, int64_t stride_b, int64_t stride_c, int64_t batch, Problem* pr) {
  if (stride_a < 0) return -14;
  if (stride_b < 0) return -15;
  if (stride_c < 0) return -16;
  if (batch < 0) return -17;
  if (batch > 1 && pr->M > 0 && pr->N > 0) {
    const int64_t c_extent = (pr->M - 1) * pr->ldc + pr->N;  // elements one C matrix spans
    if (stride_c < c_extent) return -16;
    // every element offset of the last product must fit in int64
    const int64_t lim = INT64_MAX / 2;
    if (stride_a > lim / batch || stride_b > lim / batch || stride_c > lim / batch) return SGEMM_ERR_UNSUPPORTED;
  }
  pr->stride_a = stride_a;
  pr->stride_b = stride_b;
  pr->stride_c = stride_c;
  pr->batch = batch;
  return SGEMM_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Schedule of the persistent tensor-core kernel (see kernel_tf32x3.cu).
// Stream-K pays for every output tile it splits (partial sums written and
// read back by the fixup kernel), so it is used only when each CTA gets at
// least kMinStreamKIters K tiles of it:
//   tiles >= SMs: whole-tile rounds on one CTA per SM; the (tiles % SMs)
//     tiles of a ragged last round go to stream-K (measured at 4096^3: 266
//     against 226 TFLOPS for the split-operand kernel, whose operands fit in L2
//     only while the CTAs stay at the same K), or, when that share is short,
//     the last SMs + (tiles % SMs) tiles, or they stay whole if that is short too;
//   3/4 SMs <= tiles < SMs: one CTA (or cluster) per whole tile, the rest
//     of the SMs idle (measured at 2048^3 on the split-operand kernel, 64
//     tiles for 76 clusters: 169 against 161 TFLOPS for stream-K);
//   tiles < 3/4 SMs: stream-K over all tiles on one CTA per SM, or, if that
//     share is short, S = min(SMs / tiles, K tiles / 4) CTAs per tile;
//   forced split S (override): S CTAs per tile (S = 1: one CTA per tile,
//     scheduled by the hardware).
constexpr int64_t kMinStreamKIters = 32;

// Small-product kernel (kernel_small.cu, FP32 FFMA, selected by override):
// the output extents it covers.
constexpr int64_t kSmallMaxMN = 64;
// Block-diagonal groups on the tensor cores: products with M, N <= 64 two to a
// tile, with M, N <= 32 four to a tile, chosen by default for a batch of at
// least one product per SM (measured on GB300, TFLOPS, pairs / one product per
// tile / small-product kernel: 8192 x 64^3 51.0 / 24.8 / 40.9, 2048 x
// 64x64x1024 90.9 / 51.2 / 50.0; 76 pairs on 152 SMs, K = 1024: 41.1 / 40.6 /
// 22.1).
constexpr int64_t kGroupMaxMN = 64;
constexpr int64_t kSmallKChunk = 32;
constexpr int64_t kSmallCtasPerSm = 4;  // persistent grid: 4 x 32 KB of stages per SM

// min_iters: the stream-K share's minimum in K tiles; last_round: whether a short remainder may
// take the last whole round into stream-K with it.  The BF16-input GEMM (64-deep K tiles, a third
// of a 3xTF32 tile's tensor time) uses 16 and no last round: measured at 4096^3 694.6 against
// 670.2 TFLOPS (28 stream-K tiles instead of 104), 16384x1024x4096 678.4 / 656.6, 4097x3001x2053
// 432.3 / 409.5; with the last round, 8192x4096x1024 fell from 571.0 to 500.1 (132 tiles).
int plan_stream_k(int64_t tiles, int64_t kt, int sm_count, sgemm_plan_t* plan,
                  int64_t min_iters = kMinStreamKIters, bool last_round = true) {
  const int64_t sms = std::max(1, sm_count);
  int64_t grid, dp_tiles, sk_tiles;
  const int ov_split = g_override_split.load();
  if (ov_split > 0) {
    dp_tiles = 0;
    sk_tiles = tiles;
    grid = std::min<int64_t>({tiles * std::min(ov_split, 128), tiles * kt, int64_t{1} << 20});
  } else if (tiles >= sms) {
    // whole rounds, then the remainder's K iterations shared evenly (clusters or CTAs then work on
    // the same K range at the same time in the whole rounds, which keeps the operands in L2); when
    // that share is short, the last whole round goes to stream-K too
    grid = sms;
    const int64_t rem = tiles % sms;
    sk_tiles = 0;
    if (rem * kt / sms >= min_iters) sk_tiles = rem;
    else if (last_round && rem && (sms + rem) * kt / sms >= min_iters) sk_tiles = sms + rem;
    dp_tiles = tiles - sk_tiles;
  } else if (4 * tiles >= 3 * sms) {
    // at least 3/4 as many tiles as units: whole tiles, one per unit, the rest idle (at 2048^3 the
    // stream-K schedule's fixup read 52 MB of partial sums and took 19% of the call)
    grid = tiles;
    dp_tiles = tiles;
    sk_tiles = 0;
  } else {
    dp_tiles = 0;
    sk_tiles = tiles;
    // (at most 254 CTAs per tile: the fixup kernel handles up to 256 sharers of a tile)
    if (tiles * kt / sms >= min_iters) {
      grid = std::min<int64_t>(sms, tiles * 254);
    } else {
      const int64_t split = std::max<int64_t>(1, std::min<int64_t>({sms / tiles, kt / 4, 254}));
      grid = tiles * split;
    }
  }
  const int64_t sk_iters = sk_tiles * kt;
  // int64 headroom of the device's c * sk_iters and (i + 1) * grid products,
  // and an int count of K tiles per CTA
  if (sk_iters > (INT64_MAX / 4) / (grid + 1) || (dp_tiles / grid + 1) * kt + sk_iters / grid + 1 > INT_MAX)
    return SGEMM_ERR_UNSUPPORTED;
  // the most CTAs sharing one stream-K tile (owner(i) = ceil((i+1) G / I) - 1)
  int64_t most = 1;
  for (int64_t j = 0; j < sk_tiles; ++j) {
    const int64_t i0 = j * kt, i1 = i0 + kt - 1;
    const int64_t c0 = ((i0 + 1) * grid + sk_iters - 1) / sk_iters - 1;
    const int64_t c1 = ((i1 + 1) * grid + sk_iters - 1) / sk_iters - 1;
    most = std::max(most, c1 - c0 + 1);
  }
  if (most > 256) return SGEMM_ERR_UNSUPPORTED;  // the fixup kernel's limit (cannot happen: <= SMs/tiles + 2)
  plan->split_k = (int)most;
  plan->kernel_launches = most > 1 ? 2 : 1;
  plan->grid_x = grid;
  plan->grid_y = 1;
  plan->workspace_bytes = most > 1 ? 2 * grid * (int64_t)(128 * 128 * 4) : 0;
  plan->dp_tiles = dp_tiles;
  plan->sk_tiles = sk_tiles;
  plan->sk_iters = sk_iters;
  return SGEMM_OK;
}

// Shared memory per CTA of the CTA-pair kernel (kernel_tc_pair.cu: 6 raw
// stages of 24 KB, 2 split stages of 16 KB, alignment slack).
constexpr int64_t kPairSmemBytes = 6 * 24576 + 2 * 16384 + 1024;
// ... and of the split-operand kernel (kernel_presplit.cu: 3 stages of A hi/lo and B hi/lo, 64 KB each).
constexpr int64_t kPresplitSmemBytes = 3 * 65536 + 1024;
constexpr double kMinFlopPerSplitByte = 128.0;
// Calls with operands TMA cannot load go to the split-operand kernel from this size on (measured
// on GB300 with bases one float off alignment and ld % 4 != 0, split-operand / generic kernel:
// 512^3 27.3 / 22.7 us, 1000x1300x700 38.5 / 82.6 us, 2048^3 85.2 / 439 us, 4097x3001x2053
// 263 / 1311 us; below the crossover the split passes' latency dominates).
constexpr double kMinUnalignedSplitFlop = 2.0 * 640 * 640 * 640;
constexpr int64_t kMaxSplitBytes = int64_t{4} << 30;
// The short-side kernel (kernel_skinny.cu): the short side fits one 64-column accumulator.
constexpr int64_t kSkinnyMaxShort = 64;

// Whether the short-side kernel takes M as the short side (it then computes C^T = op(B)^T op(A)^T
// and writes C transposed); N otherwise.  The shorter of the two when both are short.
bool skinny_m_short(const Problem& pr) { return pr.M <= kSkinnyMaxShort && pr.M <= pr.N; }

// Which kernels can run a problem (alignment, extents, grid limits) and the
// derived quantities the planner's rules use.
struct Eligibility {
  bool tma = false;       // TMA can load A and B (tensor-core kernels, TMA-fed FFMA kernels)
  bool small = false;     // the small-product FP32 kernel can run it
  bool group = false;     // block-diagonal groups on the tensor cores
  bool presplit = false;  // the split-operand kernel (and its split pass) can run it
  bool pair = true;       // CTA pairs can be co-scheduled (the CTA-pair and split-operand kernels)
  bool skinny = false;    // the short-side kernel (and its split pass of the short operand) can run it
  int64_t group_size = 2;   // products per tile in a group (4 when M, N <= 32)
  int64_t small_grid = 0;   // persistent grid of the small-product kernel
  int64_t clusters = 1;     // co-resident CTA-pair clusters
};

Eligibility eligibility(const Problem& pr, int sm_count, int pair_clusters, bool allow_presplit) {
  Eligibility e;
  // TMA needs 16-byte aligned bases and row strides that are multiples of 16
  // bytes; in a batch, every product's base too (a stride that is a multiple
  // of 4 floats), and matrices that do not overlap (or one shared matrix).
  const auto batch_ok = [&](int64_t stride, int64_t rows, int64_t ld) {
    return pr.batch == 1 || stride == 0 || (stride % 4 == 0 && stride >= rows * ld);
  };
  e.tma = aligned16(pr.A) && aligned16(pr.B) && pr.lda % 4 == 0 && pr.ldb % 4 == 0 &&
          batch_ok(pr.stride_a, pr.ta ? pr.K : pr.M, pr.lda) && batch_ok(pr.stride_b, pr.tb ? pr.N : pr.K, pr.ldb);
  // The small-product kernel reads whole float4s along the contiguous axis
  // of each operand, so that extent must be a multiple of 4 as well.
  // Its persistent grid deals products round-robin; a CTA's (product, K
  // chunk) items are counted in an int.
  e.small_grid = std::min<int64_t>(pr.batch, kSmallCtasPerSm * std::max(1, sm_count));
  e.small = pr.M <= kSmallMaxMN && pr.N <= kSmallMaxMN && aligned16(pr.A) && aligned16(pr.B) &&
            pr.lda % 4 == 0 && pr.ldb % 4 == 0 && (pr.batch == 1 || (pr.stride_a % 4 == 0 && pr.stride_b % 4 == 0)) &&
            (pr.ta ? pr.M : pr.K) % 4 == 0 && (pr.tb ? pr.K : pr.N) % 4 == 0 &&
            ceil_div(pr.batch, e.small_grid) * ceil_div(pr.K, kSmallKChunk) < INT_MAX;
  e.group_size = pr.M <= kGroupMaxMN / 2 && pr.N <= kGroupMaxMN / 2 ? 4 : 2;
  e.group = e.tma && pr.M <= kGroupMaxMN && pr.N <= kGroupMaxMN;
  // pair_clusters: > 0 the device's co-resident CTA-pair clusters, 0 none (the CTA-pair kernels
  // cannot run), < 0 not known (a device of sm_count SMs: SMs / 2, one cluster per TPC)
  e.pair = pair_clusters != 0;
  e.clusters = std::max(1, pair_clusters > 0 ? pair_clusters : sm_count / 2);
  // The split pass reads the operands as stored, whatever their alignment, and writes aligned
  // K-contiguous arrays for the GEMM's TMA loads, so operands TMA cannot load qualify too (the
  // transposing pass's grid holds K / 32 and the products in dimensions y and z).
  e.presplit = e.pair && allow_presplit && ceil_div(pr.K, 32) <= 65535 && pr.batch <= 65535;
  // The short-side kernel: one product, a side of at most 64, TMA loads of the long operand as
  // stored (the short one goes through the split pass, any alignment), split arrays in the
  // workspace within kMaxSplitBytes.
  if (pr.batch == 1 && std::min(pr.M, pr.N) <= kSkinnyMaxShort && allow_presplit && ceil_div(pr.K, 32) <= 65535) {
    const bool m_short = skinny_m_short(pr);
    const float* lp = m_short ? pr.B : pr.A;
    const int64_t lld = m_short ? pr.ldb : pr.lda;
    e.skinny = aligned16(lp) && lld % 4 == 0 &&
               2 * std::min(pr.M, pr.N) * split_ldk(pr.K) * 4 <= kMaxSplitBytes;
  }
  return e;
}

// The planner's default kernel, then the process-wide override (a forced
// variant whose conditions the problem breaks falls back).
int choose_variant(const Problem& pr, const Eligibility& e, int sm_count) {
  // Default: a 3xTF32 tensor-core kernel whenever TMA can load the operands
  // (they beat the FP32 FFMA kernels on every measured shape): the
  // split-operand kernel, the CTA-pair kernel or one CTA per tile by the
  // rules below, several products to a tile (block-diagonal) for a batch of
  // at least one product per SM with M, N <= 64; the generic SIMT kernel
  // otherwise.  The FP32 FFMA kernels (TMA-fed, small-product) stay
  // selectable by override: IEEE FP32 operations throughout.
  int variant = e.tma ? SGEMM_VARIANT_TC_TF32X3 : SGEMM_VARIANT_GENERIC;
  // CTA pairs (256 x 128 tiles) when every cluster gets at least one whole
  // tile: measured on GB300 2-5% faster than one CTA per 128 x 128 tile on
  // 2048^3 .. 16384 x 1024 x 4096, slower on fewer tiles (1024^3: 70.5 against
  // 74.3 TFLOPS) and on M <= 128 (half of every pair tile idle).
  if (e.tma && e.pair && pr.M > 128 && ceil_div(pr.M, 256) * ceil_div(pr.N, 128) * pr.batch >= e.clusters)
    variant = SGEMM_VARIANT_TC_PAIR;
  // Operands split once per call (TC_PRESPLIT) when the GEMM reuses them enough to amortize the
  // split pass (read once, hi and lo written: 12 bytes per element of op(A) and op(B)) and there
  // are at least 4/5 as many 256 x 256 tiles as clusters; measured on GB300 (TFLOPS, split pass
  // included, against TC_PAIR): 4096^3 266.7 / 209.1, 8192x4096x1024 239.5 / 195.1,
  // 16384x1024x4096 244.6 / 218.8, 4097x3001x2053 200.2 / 166.1, 32 x 2048x1024x1024 with a
  // shared B 226.0 / 202.8, 64 tiles: 2048x2048x1024 166.7 / 139.1, 2048^3 163.8 / 159.5; slower
  // at 64 x 512x1024x1024 (60 FLOP per split byte: 142.4 / 195.1) and on fewer tiles (48 tiles:
  // 2048x1536x2048 154.8 / 160.5; 1024^3 49.7 / 71.7).  The split arrays are capped at
  // kMaxSplitBytes of workspace.
  const SplitLayout sl = split_layout(pr.M, pr.N, pr.K, pr.batch, pr.stride_a, pr.stride_b, 0);
  const bool split_fits = 2 * (sl.a_bytes + sl.b_bytes) <= kMaxSplitBytes;
  const double flops = 2.0 * (double)pr.M * (double)pr.N * (double)pr.K * (double)pr.batch;
  if (e.tma && e.presplit && split_fits && pr.M > 128 &&
      5 * ceil_div(pr.M, 256) * ceil_div(pr.N, 256) * pr.batch >= 4 * e.clusters &&
      flops >= kMinFlopPerSplitByte * 3.0 * (double)(sl.a_bytes + sl.b_bytes))
    variant = SGEMM_VARIANT_TC_PRESPLIT;
  // Operands TMA cannot load (a base not 16-byte aligned, lda or ldb not a multiple of 4, a batch
  // stride not a multiple of 4): the split pass rewrites them aligned, so the split-operand kernel
  // runs them on the tensor cores whenever the call is large enough to amortize the pass and its
  // 256 x 256 tiles are at least a quarter full; the generic FP32 kernel takes the rest (batches
  // of small products among them).
  if (!e.tma && e.presplit && split_fits && flops >= kMinUnalignedSplitFlop &&
      4.0 * (double)pr.M * (double)pr.N >= (double)(ceil_div(pr.M, 256) * 256) * (double)(ceil_div(pr.N, 256) * 256))
    variant = SGEMM_VARIANT_TC_PRESPLIT;
  if (e.group && pr.batch >= sm_count) variant = SGEMM_VARIANT_TC_GROUPED;
  // One short side (<= 64): the short-side kernel once the long side and K are large enough to
  // amortize its split pass; measured on GB300 (us, short-side / one-CTA kernel): 64x4096x16384
  // 81.0 / 98.6, 16384x64x16384 282 / 384, 8x16384x4096 91 / 111, 4096x64x4096 47.9 / 48.5;
  // slower with a long side of 1024 (1024x64x4096 38.8 / 33.0, 1024x64x16384 51.0 / 47.7) and
  // equal below L * K = 2^24 (64x4096x1024 31.4 / 31.1).
  // (Only the long operand must be TMA-aligned: the split pass reads the short one as stored.)
  if (e.skinny) {
    const int64_t L = std::max(pr.M, pr.N);
    if (L >= 2048 && (double)L * (double)pr.K >= 16777216.0) variant = SGEMM_VARIANT_TC_SKINNY;
  }

  switch (g_override_variant.load()) {
    case SGEMM_VARIANT_GENERIC: return SGEMM_VARIANT_GENERIC;
    case SGEMM_VARIANT_TMA_128x128: return e.tma ? SGEMM_VARIANT_TMA_128x128 : SGEMM_VARIANT_GENERIC;
    case SGEMM_VARIANT_TMA_64x256: return e.tma ? SGEMM_VARIANT_TMA_64x256 : SGEMM_VARIANT_GENERIC;
    case SGEMM_VARIANT_TC_TF32X3: return e.tma ? SGEMM_VARIANT_TC_TF32X3 : SGEMM_VARIANT_GENERIC;
    case SGEMM_VARIANT_SMALL: return e.small ? SGEMM_VARIANT_SMALL : SGEMM_VARIANT_GENERIC;
    case SGEMM_VARIANT_TC_GROUPED: return e.group ? SGEMM_VARIANT_TC_GROUPED : SGEMM_VARIANT_GENERIC;
    case SGEMM_VARIANT_TC_PAIR:
      return !e.tma ? SGEMM_VARIANT_GENERIC : e.pair ? SGEMM_VARIANT_TC_PAIR : SGEMM_VARIANT_TC_TF32X3;
    case SGEMM_VARIANT_TC_PRESPLIT:
      return e.presplit ? SGEMM_VARIANT_TC_PRESPLIT
             : !e.tma   ? SGEMM_VARIANT_GENERIC
             : e.pair   ? SGEMM_VARIANT_TC_PAIR
                        : SGEMM_VARIANT_TC_TF32X3;
    case SGEMM_VARIANT_TC_SKINNY:
      return e.skinny ? SGEMM_VARIANT_TC_SKINNY : e.tma ? SGEMM_VARIANT_TC_TF32X3 : SGEMM_VARIANT_GENERIC;
    default: return variant;
  }
}

// Block-diagonal groups: whole tiles (a group of products each) on one persistent CTA per SM,
// no stream-K.
int plan_grouped(const Problem& pr, const Eligibility& e, int sm_count, sgemm_plan_t* plan) {
  const int64_t tiles = ceil_div(pr.batch, e.group_size);
  const int64_t kt = ceil_div(pr.K, 32);
  const int64_t grid = std::min<int64_t>(tiles, std::max(1, sm_count));
  if ((tiles / grid + 1) * kt > INT_MAX) return SGEMM_ERR_UNSUPPORTED;
  plan->variant = SGEMM_VARIANT_TC_GROUPED;
  plan->tile_m = plan->tile_n = (int)(128 / e.group_size);
  plan->tile_k = 32;
  plan->stages = 4;
  plan->threads = 608;
  plan->smem_bytes = 4 * 32768 + 2 * 32768 + 1024;
  plan->kernel_launches = 1;
  plan->grid_x = grid;
  plan->grid_y = 1;
  plan->dp_tiles = tiles;
  return SGEMM_OK;
}

// The short-side kernel: tiles of 128 along the long side, the persistent stream-K schedule of the
// one-CTA kernel (slots of 128 x 64 floats), the split arrays of the short operand; launches: its
// split pass, the GEMM, the fixup when a tile is shared.
int plan_skinny(const Problem& pr, int sm_count, sgemm_plan_t* plan) {
  const bool m_short = skinny_m_short(pr);
  const int64_t L = m_short ? pr.N : pr.M, S = m_short ? pr.M : pr.N;
  const int s = plan_stream_k(ceil_div(L, 128), ceil_div(pr.K, 32), sm_count, plan);
  if (s != SGEMM_OK) return s;
  plan->variant = SGEMM_VARIANT_TC_SKINNY;
  plan->tile_m = 128;
  plan->tile_n = 64;
  plan->tile_k = 32;
  plan->stages = 8;                             // long-operand ring (the short one has 4 stages)
  plan->threads = 640;
  plan->smem_bytes = 8 * 16384 + 4 * 16384 + 1024;
  const int64_t slots = plan->split_k > 1 ? 2 * plan->grid_x * (int64_t)(128 * 64 * 4) : 0;
  plan->workspace_bytes = round256(slots) + 2 * round256(S * split_ldk(pr.K) * 4);
  plan->kernel_launches += 1;
  return SGEMM_OK;
}

int plan_small(const Eligibility& e, sgemm_plan_t* plan) {
  plan->variant = SGEMM_VARIANT_SMALL;
  plan->tile_m = plan->tile_n = (int)kSmallMaxMN;
  plan->tile_k = (int)kSmallKChunk;
  plan->stages = 2;
  plan->threads = 64;
  plan->smem_bytes = 2 * 2 * kSmallMaxMN * kSmallKChunk * 4;
  plan->kernel_launches = 1;
  plan->grid_x = e.small_grid;
  plan->grid_y = 1;
  return SGEMM_OK;
}

// Kernels over output tiles: the tensor-core kernels' persistent schedule, or grid.y K slices
// for the FFMA and generic kernels.
int plan_tiled(const Problem& pr, const Eligibility& e, int variant, int sm_count, sgemm_plan_t* plan) {
  int bm, bn, bk, threads, stages;
  int64_t smem = 0;
  if (variant == SGEMM_VARIANT_GENERIC) {
    const GenericTileShape g = generic_tile_shape();
    bm = g.bm; bn = g.bn; bk = g.bk; threads = g.threads; stages = 2;
  } else if (variant == SGEMM_VARIANT_TC_TF32X3) {
    bm = 128; bn = 128; bk = 32; threads = 608; stages = 4; smem = 4 * 32768 + 2 * 32768 + 1024;
  } else if (variant == SGEMM_VARIANT_TC_PAIR) {
    bm = 256; bn = 128; bk = 32; threads = 608; stages = 6; smem = kPairSmemBytes;
  } else if (variant == SGEMM_VARIANT_TC_PRESPLIT) {
    bm = 256; bn = 256; bk = 32; threads = 320; stages = 3; smem = kPresplitSmemBytes;
  } else if (variant == SGEMM_VARIANT_TMA_128x128) {
    using T = tma::Tile<4, 2>;
    bm = T::BM; bn = T::BN; bk = tma::kBK; threads = tma::kThreads; stages = tma::kStages; smem = T::SMEM_BYTES;
  } else {
    using T = tma::Tile<2, 4>;
    bm = T::BM; bn = T::BN; bk = tma::kBK; threads = tma::kThreads; stages = tma::kStages; smem = T::SMEM_BYTES;
  }
  // output tiles of all products (the grid's x extent)
  const int64_t tiles = ceil_div(pr.M, bm) * ceil_div(pr.N, bn) * pr.batch;
  const int64_t kt = ceil_div(pr.K, bk);
  if (tiles > INT_MAX) return SGEMM_ERR_UNSUPPORTED;

  plan->variant = variant;
  plan->tile_m = bm;
  plan->tile_n = bn;
  plan->tile_k = bk;
  plan->stages = stages;
  plan->threads = threads;
  plan->smem_bytes = smem;
  if (variant == SGEMM_VARIANT_TC_TF32X3) return plan_stream_k(tiles, kt, sm_count, plan);
  if (variant == SGEMM_VARIANT_TC_PAIR) {
    // the stream-K schedule with clusters as the unit; 2 CTAs, 2 partial-sum slots each, per cluster
    const int s = plan_stream_k(tiles, kt, (int)e.clusters, plan);
    plan->grid_x *= 2;
    plan->workspace_bytes *= 2;
    return s;
  }
  if (variant == SGEMM_VARIANT_TC_PRESPLIT) {
    // as TC_PAIR with 256 x 256 tiles (slots of 128 x 256 floats per CTA), plus the split arrays;
    // launches: the split pass of A and of B, the GEMM, the fixup when a tile is shared
    const int s = plan_stream_k(tiles, kt, (int)e.clusters, plan);
    if (s != SGEMM_OK) return s;
    plan->grid_x *= 2;
    plan->workspace_bytes *= 4;
    plan->workspace_bytes =
        split_layout(pr.M, pr.N, pr.K, pr.batch, pr.stride_a, pr.stride_b, plan->workspace_bytes).total();
    plan->kernel_launches += 2;
    return SGEMM_OK;
  }

  // Split K only when the output tiles cannot fill the SMs, keeping at least
  // 4 K tiles per slice.
  int64_t split = 1;
  if (tiles < sm_count) split = std::min<int64_t>(sm_count / tiles, kt / 4);
  const int ov_split = g_override_split.load();
  if (ov_split > 0) split = ov_split;
  split = std::max<int64_t>(1, std::min<int64_t>({split, kt, 256}));
  const int64_t per = ceil_div(kt, split);
  split = ceil_div(kt, per);  // no empty slice

  plan->split_k = (int)split;
  plan->kernel_launches = split > 1 ? 2 : 1;
  plan->grid_x = tiles;
  plan->grid_y = split;
  plan->workspace_bytes = split > 1 ? pr.batch * split * pr.M * (ceil_div(pr.N, 4) * 4) * 4 : 0;
  return SGEMM_OK;
}

// The planner: a pure function of the problem, the SM count, the number of
// co-resident CTA-pair clusters (< 0: not known, sm_count / 2; 0: none, no
// CTA-pair kernel) and the override.  allow_presplit = false (sgemm_noalloc:
// the split arrays need workspace) plans TC_PRESPLIT as TC_PAIR.
int make_plan(const Problem& pr, int sm_count, sgemm_plan_t* plan, int pair_clusters, bool allow_presplit = true) {
  *plan = sgemm_plan_t{};
  plan->split_k = 1;
  if (pr.M == 0 || pr.N == 0 || pr.batch == 0) {
    plan->variant = SGEMM_VARIANT_NONE;
    return SGEMM_OK;
  }
  if (pr.M > INT_MAX || pr.N > INT_MAX || pr.K > INT_MAX || pr.batch > INT_MAX) return SGEMM_ERR_UNSUPPORTED;
  if (pr.K == 0 || pr.alpha == 0.0f) {
    plan->variant = SGEMM_VARIANT_SCALE;
    plan->kernel_launches = 1;
    plan->threads = 256;
    return SGEMM_OK;
  }
  const Eligibility e = eligibility(pr, sm_count, pair_clusters, allow_presplit);
  const int variant = choose_variant(pr, e, sm_count);
  if (variant == SGEMM_VARIANT_TC_GROUPED) return plan_grouped(pr, e, sm_count, plan);
  if (variant == SGEMM_VARIANT_SMALL) return plan_small(e, plan);
  if (variant == SGEMM_VARIANT_TC_SKINNY) return plan_skinny(pr, sm_count, plan);
  return plan_tiled(pr, e, variant, sm_count, plan);
}

// The TF32-input GEMM (sgemm_tf32): op(A) and op(B) rounded to TF32 once into the workspace
// ([stream-K slots][A][B], 256-byte aligned parts, rows of round4(K) floats), then the CTA-pair
// kernel with one tensor-core product per k over 256 x 256 tiles (the split-operand kernel's
// schedule), then the fixup when a tile is shared.  Any alignment: the rounding pass reads the
// operands as stored.  Needs CTA pairs (pair_clusters != 0).
int make_tf32_plan(const Problem& pr, int sm_count, int pair_clusters, sgemm_plan_t* plan) {
  *plan = sgemm_plan_t{};
  plan->split_k = 1;
  if (pr.M == 0 || pr.N == 0) {
    plan->variant = SGEMM_VARIANT_NONE;
    return SGEMM_OK;
  }
  if (pr.M > INT_MAX || pr.N > INT_MAX || pr.K > INT_MAX) return SGEMM_ERR_UNSUPPORTED;
  if (pr.K == 0 || pr.alpha == 0.0f) {
    plan->variant = SGEMM_VARIANT_SCALE;
    plan->kernel_launches = 1;
    plan->threads = 256;
    return SGEMM_OK;
  }
  // the rounding pass's transposing grid holds K / 32 in dimension y
  if (pair_clusters == 0 || ceil_div(pr.K, 32) > 65535) return SGEMM_ERR_UNSUPPORTED;
  const int64_t clusters = std::max(1, pair_clusters > 0 ? pair_clusters : sm_count / 2);
  const int64_t tiles = ceil_div(pr.M, 256) * ceil_div(pr.N, 256);
  const int s = plan_stream_k(tiles, ceil_div(pr.K, 32), (int)clusters, plan);
  if (s != SGEMM_OK) return s;
  plan->variant = SGEMM_VARIANT_TC_TF32;
  plan->tile_m = plan->tile_n = 256;
  plan->tile_k = 32;
  plan->stages = 6;
  plan->threads = 320;
  plan->smem_bytes = 6 * 32768 + 1024;
  plan->grid_x *= 2;
  plan->workspace_bytes = split_layout(pr.M, pr.N, pr.K, 1, 0, 0, plan->workspace_bytes * 4, 1).total();
  plan->kernel_launches += 2;  // the rounding passes of A and B
  return SGEMM_OK;
}

// The BF16-input GEMM (sgemm_bf16): as the TF32-input GEMM, with op(A) and op(B) rounded to BF16
// (rows of round8(K) two-byte values) and K tiles of 64.
int64_t bf16_ldk(int64_t K) { return (K + 7) / 8 * 8; }

int make_bf16_plan(const Problem& pr, int sm_count, int pair_clusters, sgemm_plan_t* plan) {
  const int s = make_tf32_plan(pr, sm_count, pair_clusters, plan);  // shape checks, NONE / SCALE
  if (s != SGEMM_OK || plan->variant != SGEMM_VARIANT_TC_TF32) return s;
  const int64_t clusters = std::max(1, pair_clusters > 0 ? pair_clusters : sm_count / 2);
  const int64_t tiles = ceil_div(pr.M, 256) * ceil_div(pr.N, 256);
  *plan = sgemm_plan_t{};
  const int t = plan_stream_k(tiles, ceil_div(pr.K, 64), (int)clusters, plan, kMinStreamKIters / 2, false);
  if (t != SGEMM_OK) return t;
  plan->variant = SGEMM_VARIANT_TC_BF16;
  plan->tile_m = plan->tile_n = 256;
  plan->tile_k = 64;
  plan->stages = 6;
  plan->threads = 320;
  plan->smem_bytes = 6 * 32768 + 1024;
  plan->grid_x *= 2;
  const int64_t ldk = bf16_ldk(pr.K);
  plan->workspace_bytes = round256(plan->workspace_bytes * 4) + round256(pr.M * ldk * 2) + round256(pr.N * ldk * 2);
  plan->kernel_launches += 2;  // the rounding passes of A and B
  return SGEMM_OK;
}

cudaError_t launch_bf16(const Problem& pr, const sgemm_plan_t& plan, const DeviceState& st, uint8_t* ws,
                        GemmParams* p, cudaStream_t stream) {
  const int64_t slot_bytes = plan.split_k > 1 ? 2 * plan.grid_x * (int64_t)(128 * 256 * 4) : 0;
  const int64_t ldk = bf16_ldk(pr.K);
  uint8_t* ar = ws + round256(slot_bytes);
  uint8_t* br = ar + round256(pr.M * ldk * 2);
  p->ws = slot_bytes > 0 ? reinterpret_cast<float*>(ws) : nullptr;
  p->za = p->zb = 0;
  p->repair = 0;
  cudaError_t e = launch_round_bf16(pr.A, pr.lda, !pr.ta, (int)pr.M, (int)pr.K, ar, ldk, st.sm_count, stream,
                                    p->fault, p->bounds, p->a_elems, SplitOrder::kFirst);
  if (e == cudaSuccess)
    e = launch_round_bf16(pr.B, pr.ldb, pr.tb, (int)pr.N, (int)pr.K, br, ldk, st.sm_count, stream, p->fault,
                          p->bounds, p->b_elems, SplitOrder::kDependent);
  CUtensorMap ma, mb;
  if (e == cudaSuccess) e = encode_bf16_map(ar, pr.K, pr.M, ldk, &ma);
  if (e == cudaSuccess) e = encode_bf16_map(br, pr.K, pr.N, ldk, &mb);
  if (e == cudaSuccess) e = launch_bf16_gemm(ma, mb, *p, stream);
  if (e == cudaSuccess && slot_bytes > 0) e = launch_presplit_fixup(*p, (int)plan.sk_tiles, stream, 64);
  return e;
}

cudaError_t launch_tf32(const Problem& pr, const sgemm_plan_t& plan, const DeviceState& st, uint8_t* ws,
                        GemmParams* p, cudaStream_t stream) {
  const int64_t slot_bytes = plan.split_k > 1 ? 2 * plan.grid_x * (int64_t)(128 * 256 * 4) : 0;
  const SplitLayout l = split_layout(pr.M, pr.N, pr.K, 1, 0, 0, slot_bytes, 1);
  const int64_t ldk = split_ldk(pr.K);
  float* ar = reinterpret_cast<float*>(ws + round256(l.slots));
  float* br = reinterpret_cast<float*>(ws + round256(l.slots) + round256(l.a_bytes));
  p->ws = slot_bytes > 0 ? reinterpret_cast<float*>(ws) : nullptr;
  p->za = p->zb = 0;
  p->repair = 0;
  cudaError_t e = launch_split_operand(pr.A, pr.lda, 0, !pr.ta, (int)pr.M, (int)pr.K, 1, ar, nullptr, ldk,
                                       st.sm_count, stream, p->fault, p->bounds, p->a_elems, SplitOrder::kFirst);
  if (e == cudaSuccess)
    e = launch_split_operand(pr.B, pr.ldb, 0, pr.tb, (int)pr.N, (int)pr.K, 1, br, nullptr, ldk, st.sm_count, stream,
                             p->fault, p->bounds, p->b_elems, SplitOrder::kDependent);
  CUtensorMap ma, mb;
  if (e == cudaSuccess) e = encode_split_map(ar, pr.K, pr.M, ldk, 1, &ma);
  if (e == cudaSuccess) e = encode_split_map(br, pr.K, pr.N, ldk, 1, &mb);
  if (e == cudaSuccess) e = launch_tf32_gemm(ma, mb, *p, stream);
  if (e == cudaSuccess && slot_bytes > 0) e = launch_presplit_fixup(*p, (int)plan.sk_tiles, stream);
  return e;
}

// TC_PRESPLIT: the split pass of op(A) and op(B) into the workspace ([stream-K slots][A hi][A lo]
// [B hi][B lo], 256-byte aligned parts), then the GEMM over maps of the split arrays and the fixup.
cudaError_t launch_presplit(const Problem& pr, const sgemm_plan_t& plan, const DeviceState& st, uint8_t* ws,
                            GemmParams* p, cudaStream_t stream) {
  const int64_t slot_bytes = plan.kernel_launches > 3 ? 2 * plan.grid_x * (int64_t)(128 * 256 * 4) : 0;
  const SplitLayout l = split_layout(pr.M, pr.N, pr.K, pr.batch, pr.stride_a, pr.stride_b, slot_bytes);
  const int64_t ldk = split_ldk(pr.K);
  float* ahi = reinterpret_cast<float*>(ws + round256(l.slots));
  float* alo = reinterpret_cast<float*>(ws + round256(l.slots) + round256(l.a_bytes));
  float* bhi = reinterpret_cast<float*>(ws + round256(l.slots) + 2 * round256(l.a_bytes));
  float* blo = reinterpret_cast<float*>(ws + round256(l.slots) + 2 * round256(l.a_bytes) + round256(l.b_bytes));
  p->ws = slot_bytes > 0 ? reinterpret_cast<float*>(ws) : nullptr;
  // op(A) rows run along K when A is 'N'; op(B) rows (columns of op(B)) when B is 'T'
  cudaError_t e = launch_split_operand(pr.A, pr.lda, pr.stride_a, !pr.ta, (int)pr.M, (int)pr.K,
                                       (int)l.a_products, ahi, alo, ldk, st.sm_count, stream, p->fault, p->bounds,
                                       p->a_elems, SplitOrder::kFirst);
  if (e == cudaSuccess)
    e = launch_split_operand(pr.B, pr.ldb, pr.stride_b, pr.tb, (int)pr.N, (int)pr.K, (int)l.b_products, bhi, blo,
                             ldk, st.sm_count, stream, p->fault, p->bounds, p->b_elems, SplitOrder::kDependent);
  CUtensorMap mah, mal, mbh, mbl;
  if (e == cudaSuccess) e = encode_split_map(ahi, pr.K, pr.M, ldk, l.a_products, &mah);
  if (e == cudaSuccess) e = encode_split_map(alo, pr.K, pr.M, ldk, l.a_products, &mal);
  if (e == cudaSuccess) e = encode_split_map(bhi, pr.K, pr.N, ldk, l.b_products, &mbh);
  if (e == cudaSuccess) e = encode_split_map(blo, pr.K, pr.N, ldk, l.b_products, &mbl);
  p->za = l.a_products > 1 ? 1 : 0;
  p->zb = l.b_products > 1 ? 1 : 0;
  if (e == cudaSuccess) e = launch_presplit_gemm(mah, mal, mbh, mbl, *p, stream);
  if (e == cudaSuccess && slot_bytes > 0) e = launch_presplit_fixup(*p, (int)plan.sk_tiles, stream);
  return e;
}

// TC_SKINNY: the short operand split into the workspace ([stream-K slots][short hi][short lo],
// 256-byte aligned parts, rows of round4(K) floats), then the short-side GEMM on the product seen
// as (long side) x (short side) -- its op(A) the long operand, its op(B) the short one (the NaN
// repair reads both as stored), C written transposed when M is the short side -- then the fixup
// when a tile is shared.
cudaError_t launch_skinny(const Problem& pr, const sgemm_plan_t& plan, uint8_t* ws, const GemmParams& p,
                          int sm_count, cudaStream_t stream) {
  const bool m_short = skinny_m_short(pr);
  const int64_t L = m_short ? pr.N : pr.M, S = m_short ? pr.M : pr.N;
  const bool long_contig = m_short ? !pr.tb : pr.ta;    // long operand stored [K][L]
  const bool short_kcontig = m_short ? !pr.ta : pr.tb;  // short operand stored [S][K]
  const int64_t slot_bytes = plan.split_k > 1 ? 2 * plan.grid_x * (int64_t)(128 * 64 * 4) : 0;
  const int64_t ldk = split_ldk(pr.K);
  const int64_t part = round256(S * ldk * 4);
  float* shi = reinterpret_cast<float*>(ws + round256(slot_bytes));
  float* slo = reinterpret_cast<float*>(ws + round256(slot_bytes) + part);
  GemmParams q = p;
  q.M = (int)L;
  q.N = (int)S;
  q.A = m_short ? pr.B : pr.A;
  q.lda = m_short ? pr.ldb : pr.lda;
  q.ta = long_contig ? 1 : 0;
  q.B = m_short ? pr.A : pr.B;
  q.ldb = m_short ? pr.lda : pr.ldb;
  q.tb = short_kcontig ? 1 : 0;
  q.stride_a = q.stride_b = q.stride_c = 0;
  q.tiles_m = (int)ceil_div(L, 128);
  q.tiles_n = 1;
  q.ws = slot_bytes > 0 ? reinterpret_cast<float*>(ws) : nullptr;
  set_extents(&q, plan.workspace_bytes, p.bounds);
  if (m_short) q.c_elems = matrix_extent(S, L, pr.ldc, 1, 0);  // C is S x L
  cudaError_t e = launch_split_operand(q.B, q.ldb, 0, short_kcontig, (int)S, (int)pr.K, 1, shi, slo, ldk, sm_count,
                                       stream, p.fault, p.bounds, q.b_elems);
  CUtensorMap ml, msh, msl;
  if (e == cudaSuccess)
    e = long_contig ? encode_matrix_map(q.A, L, pr.K, q.lda, 128, 32, &ml)
                    : encode_matrix_map(q.A, pr.K, L, q.lda, 32, 128, &ml);
  if (e == cudaSuccess) e = encode_split_map(shi, pr.K, S, ldk, 1, &msh, 64);
  if (e == cudaSuccess) e = encode_split_map(slo, pr.K, S, ldk, 1, &msl, 64);
  if (e == cudaSuccess) e = launch_skinny_gemm(long_contig, m_short, ml, msh, msl, q, stream);
  if (e == cudaSuccess && slot_bytes > 0) e = launch_skinny_fixup(m_short, q, (int)plan.sk_tiles, stream);
  return e;
}

// ext_ws: the caller's workspace of at least plan.workspace_bytes (sgemm_ex), or nullptr to take
// the partial sums from the device's stream-ordered pool.
int launch_gemm(const Problem& pr, const sgemm_plan_t& plan, const DeviceState& st, float* C,
                cudaStream_t stream, void* ext_ws = nullptr) {
  GemmParams p{};
  p.M = (int)pr.M;
  p.N = (int)pr.N;
  p.K = (int)pr.K;
  p.alpha = pr.alpha;
  p.beta = pr.beta;
  p.A = pr.A;
  p.B = pr.B;
  p.C = C;
  p.lda = pr.lda;
  p.ldb = pr.ldb;
  p.ta = pr.ta;
  p.tb = pr.tb;
  p.ldc = pr.ldc;
  p.c_vec = aligned16(C) && pr.ldc % 4 == 0 && (pr.batch == 1 || pr.stride_c % 4 == 0);
  p.batch = (int)pr.batch;
  p.stride_a = pr.stride_a;
  p.stride_b = pr.stride_b;
  p.stride_c = pr.stride_c;
  p.timeout_ns = wait_timeout_ns();
  p.fault = st.fault;
  set_extents(&p, plan.workspace_bytes, st.bounds);

  if (plan.variant == SGEMM_VARIANT_SCALE) {
    cudaError_t e = launch_scale(p, stream);
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
  }

  const int split = plan.split_k;
  p.tiles_m = (int)ceil_div(pr.M, plan.tile_m);
  p.tiles_n = (int)ceil_div(pr.N, plan.tile_n);
  p.k_tiles_per_split = (int)ceil_div(ceil_div(pr.K, plan.tile_k), split);
  p.ws_ld = ceil_div(pr.N, 4) * 4;
  set_schedule(plan, &p);

  CUtensorMap mapA, mapB;
  if (plan.variant != SGEMM_VARIANT_GENERIC && plan.variant != SGEMM_VARIANT_SMALL &&
      plan.variant != SGEMM_VARIANT_TC_PRESPLIT && plan.variant != SGEMM_VARIANT_TC_TF32 &&
      plan.variant != SGEMM_VARIANT_TC_SKINNY && plan.variant != SGEMM_VARIANT_TC_BF16) {
    int box_m, box_n;
    operand_boxes(plan, &box_m, &box_n);
    cudaError_t e = encode_operand_maps(pr.ta, pr.tb, pr.M, pr.N, pr.K, pr.A, pr.lda, pr.stride_a, pr.B, pr.ldb,
                                        pr.stride_b, p.batch, box_m, box_n, plan.tile_k, &mapA, &mapB, &p.za,
                                        &p.zb);
    if (e != cudaSuccess) return cuda_fail(e);
  }

  void* ws = nullptr;
  if (plan.workspace_bytes > 0 && ext_ws) {
    p.ws = static_cast<float*>(ext_ws);
  } else if (plan.workspace_bytes > 0) {
    cudaError_t e = cudaMallocFromPoolAsync(&ws, (size_t)plan.workspace_bytes, st.pool, stream);
    if (e != cudaSuccess) {
      record_cuda_failure(e);
      return e == cudaErrorMemoryAllocation ? SGEMM_ERR_NOMEM : SGEMM_ERR_CUDA;
    }
    p.ws = static_cast<float*>(ws);
  }

  cudaError_t e;
  if (plan.variant == SGEMM_VARIANT_TC_PRESPLIT) {
    e = launch_presplit(pr, plan, st, static_cast<uint8_t*>(ws ? ws : ext_ws), &p, stream);
  } else if (plan.variant == SGEMM_VARIANT_TC_TF32) {
    e = launch_tf32(pr, plan, st, static_cast<uint8_t*>(ws ? ws : ext_ws), &p, stream);
  } else if (plan.variant == SGEMM_VARIANT_TC_BF16) {
    e = launch_bf16(pr, plan, st, static_cast<uint8_t*>(ws ? ws : ext_ws), &p, stream);
  } else if (plan.variant == SGEMM_VARIANT_TC_SKINNY) {
    e = launch_skinny(pr, plan, static_cast<uint8_t*>(ws ? ws : ext_ws), p, st.sm_count, stream);
  } else if (plan.variant == SGEMM_VARIANT_GENERIC) {
    e = launch_generic_gemm(pr.ta, pr.tb, p, split, stream);
  } else if (plan.variant == SGEMM_VARIANT_SMALL) {
    e = launch_small_gemm(pr.ta, pr.tb, p, (int)plan.grid_x, stream);
  } else if (plan.variant == SGEMM_VARIANT_TC_TF32X3 || plan.variant == SGEMM_VARIANT_TC_GROUPED) {
    e = launch_tf32x3(pr.ta, pr.tb, plan.variant == SGEMM_VARIANT_TC_GROUPED ? 128 / plan.tile_m : 1, mapA, mapB,
                      p, stream);
    if (e == cudaSuccess && plan.kernel_launches > 1) e = launch_streamk_fixup(p, (int)plan.sk_tiles, stream);
  } else if (plan.variant == SGEMM_VARIANT_TC_PAIR) {
    e = launch_tc_pair(pr.ta, pr.tb, mapA, mapB, p, stream);
    if (e == cudaSuccess && plan.kernel_launches > 1) e = launch_pair_fixup(p, (int)plan.sk_tiles, stream);
  } else {
    const TmaTile tile = plan.variant == SGEMM_VARIANT_TMA_128x128 ? TmaTile::k128x128 : TmaTile::k64x256;
    if (!pr.ta && !pr.tb) e = launch_tma_op_nn(tile, mapA, mapB, p, split, stream);
    else if (!pr.ta && pr.tb) e = launch_tma_op_nt(tile, mapA, mapB, p, split, stream);
    else if (pr.ta && !pr.tb) e = launch_tma_op_tn(tile, mapA, mapB, p, split, stream);
    else e = launch_tma_op_tt(tile, mapA, mapB, p, split, stream);
  }
  if (e == cudaSuccess && split > 1 && plan.variant != SGEMM_VARIANT_TC_TF32X3 &&
      plan.variant != SGEMM_VARIANT_TC_GROUPED && plan.variant != SGEMM_VARIANT_TC_PAIR &&
      plan.variant != SGEMM_VARIANT_TC_PRESPLIT && plan.variant != SGEMM_VARIANT_TC_TF32 &&
      plan.variant != SGEMM_VARIANT_TC_SKINNY && plan.variant != SGEMM_VARIANT_TC_BF16)
    e = launch_splitk_reduce(p, split, stream);
  if (ws) {
    cudaError_t ef = cudaFreeAsync(ws, stream);
    if (e == cudaSuccess) e = ef;
  }
  return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

}  // namespace

int sgemm_impl::plan_without_split_arrays(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                              int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc,
                              int sm_count, int pair_clusters, sgemm_plan_t* plan) {
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  return make_plan(pr, sm_count, plan, pair_clusters, false);
}

extern "C" {

int sgemm(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
          const float* B, int64_t ldb, float beta, float* C, int64_t ldc, struct CUstream_st* stream) {
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  if (M == 0 || N == 0) return SGEMM_OK;
  int dev;
  DeviceState* st;
  s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  sgemm_plan_t plan;
  s = make_plan(pr, st->sm_count, &plan, st->pair_clusters);
  if (s != SGEMM_OK) return s;
  return launch_gemm(pr, plan, *st, C, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_workspace_size(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                         int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc,
                         size_t* bytes) {
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  if (!bytes) return -14;
  *bytes = 0;
  if (M == 0 || N == 0) return SGEMM_OK;
  int dev;
  DeviceState* st;
  s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  sgemm_plan_t plan;
  s = make_plan(pr, st->sm_count, &plan, st->pair_clusters);
  if (s != SGEMM_OK) return s;
  *bytes = (size_t)plan.workspace_bytes;
  return SGEMM_OK;
}

int sgemm_ex(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
             const float* B, int64_t ldb, float beta, float* C, int64_t ldc, void* workspace, size_t workspace_bytes,
             struct CUstream_st* stream) {
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  if (workspace && !aligned16(workspace)) return -14;
  if (M == 0 || N == 0) return SGEMM_OK;
  int dev;
  DeviceState* st;
  s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  sgemm_plan_t plan;
  s = make_plan(pr, st->sm_count, &plan, st->pair_clusters);
  if (s != SGEMM_OK) return s;
  if (plan.workspace_bytes > 0) {
    if (!workspace) return -14;
    if ((uint64_t)workspace_bytes < (uint64_t)plan.workspace_bytes) return -15;
  }
  return launch_gemm(pr, plan, *st, C, reinterpret_cast<cudaStream_t>(stream), workspace);
}

int sgemm_plan(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
               int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc, int sm_count,
               sgemm_plan_t* plan) {
  if (!plan) return -15;
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  int pair_clusters = -1;
  if (sm_count <= 0) {
    int dev;
    DeviceState* st;
    s = device_state(&dev, &st);
    if (s != SGEMM_OK) return s;
    sm_count = st->sm_count;
    pair_clusters = st->pair_clusters;
  }
  return make_plan(pr, sm_count, plan, pair_clusters);
}

int sgemm_plan_for_device(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc,
                          int sm_count, int pair_clusters, sgemm_plan_t* plan) {
  if (!plan) return -16;
  if (sm_count <= 0) return -14;
  if (pair_clusters < 0) return -15;
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  return make_plan(pr, sm_count, plan, pair_clusters);
}

int sgemm_release_workspace(size_t keep_bytes) {
  int dev;
  DeviceState* st;
  int s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  cudaError_t e = cudaMemPoolTrimTo(st->pool, keep_bytes);
  if (e == cudaSuccess) e = trim_host_pool(dev, keep_bytes);
  return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

int sgemm_tf32(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
               const float* B, int64_t ldb, float beta, float* C, int64_t ldc, struct CUstream_st* stream) {
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  if (M == 0 || N == 0) return SGEMM_OK;
  int dev;
  DeviceState* st;
  s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  sgemm_plan_t plan;
  s = make_tf32_plan(pr, st->sm_count, st->pair_clusters, &plan);
  if (s != SGEMM_OK) return s;
  return launch_gemm(pr, plan, *st, C, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_tf32_plan(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                    int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc, int sm_count,
                    sgemm_plan_t* plan) {
  if (!plan) return -15;
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  int pair_clusters = -1;
  if (sm_count <= 0) {
    int dev;
    DeviceState* st;
    s = device_state(&dev, &st);
    if (s != SGEMM_OK) return s;
    sm_count = st->sm_count;
    pair_clusters = st->pair_clusters;
  }
  return make_tf32_plan(pr, sm_count, pair_clusters, plan);
}

int sgemm_bf16(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
               const float* B, int64_t ldb, float beta, float* C, int64_t ldc, struct CUstream_st* stream) {
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  if (M == 0 || N == 0) return SGEMM_OK;
  int dev;
  DeviceState* st;
  s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  sgemm_plan_t plan;
  s = make_bf16_plan(pr, st->sm_count, st->pair_clusters, &plan);
  if (s != SGEMM_OK) return s;
  return launch_gemm(pr, plan, *st, C, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_bf16_plan(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                    int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc, int sm_count,
                    sgemm_plan_t* plan) {
  if (!plan) return -15;
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  int pair_clusters = -1;
  if (sm_count <= 0) {
    int dev;
    DeviceState* st;
    s = device_state(&dev, &st);
    if (s != SGEMM_OK) return s;
    sm_count = st->sm_count;
    pair_clusters = st->pair_clusters;
  }
  return make_bf16_plan(pr, sm_count, pair_clusters, plan);
}

int sgemm_strided_batched(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                          int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                          int64_t strideA, int64_t strideB, int64_t strideC, int64_t batch_count,
                          struct CUstream_st* stream) {
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  s = validate_batch(strideA, strideB, strideC, batch_count, &pr);
  if (s != SGEMM_OK) return s;
  if (M == 0 || N == 0 || batch_count == 0) return SGEMM_OK;
  int dev;
  DeviceState* st;
  s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  sgemm_plan_t plan;
  s = make_plan(pr, st->sm_count, &plan, st->pair_clusters);
  if (s != SGEMM_OK) return s;
  return launch_gemm(pr, plan, *st, C, reinterpret_cast<cudaStream_t>(stream));
}

int sgemm_plan_strided_batched(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                               const float* A, int64_t lda, const float* B, int64_t ldb, float beta, const float* C,
                               int64_t ldc, int64_t strideA, int64_t strideB, int64_t strideC, int64_t batch_count,
                               int sm_count, sgemm_plan_t* plan) {
  if (!plan) return -19;
  Problem pr;
  int s = validate(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, &pr);
  if (s != SGEMM_OK) return s;
  s = validate_batch(strideA, strideB, strideC, batch_count, &pr);
  if (s != SGEMM_OK) return s;
  int pair_clusters = -1;
  if (sm_count <= 0) {
    int dev;
    DeviceState* st;
    s = device_state(&dev, &st);
    if (s != SGEMM_OK) return s;
    sm_count = st->sm_count;
    pair_clusters = st->pair_clusters;
  }
  return make_plan(pr, sm_count, plan, pair_clusters);
}

int sgemm_set_variant_override(int variant, int split_k) {
  if (variant != SGEMM_VARIANT_AUTO && variant != SGEMM_VARIANT_GENERIC && variant != SGEMM_VARIANT_TMA_128x128 &&
      variant != SGEMM_VARIANT_TMA_64x256 && variant != SGEMM_VARIANT_TC_TF32X3 && variant != SGEMM_VARIANT_SMALL &&
      variant != SGEMM_VARIANT_TC_GROUPED && variant != SGEMM_VARIANT_TC_PAIR &&
      variant != SGEMM_VARIANT_TC_PRESPLIT && variant != SGEMM_VARIANT_TC_SKINNY)
    return -1;
  g_override_variant.store(variant);
  g_override_split.store(split_k < 0 ? 0 : split_k);
  return SGEMM_OK;
}

const char* sgemm_status_string(int status) {
  switch (status) {
    case SGEMM_OK: return "SGEMM_OK";
    case SGEMM_ERR_CUDA: return "SGEMM_ERR_CUDA: a CUDA runtime call failed";
    case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a bounded in-kernel wait gave up";
    case SGEMM_ERR_NOMEM: return "SGEMM_ERR_NOMEM: workspace allocation failed";
    case SGEMM_ERR_UNSUPPORTED: return "SGEMM_ERR_UNSUPPORTED: dimension too large or no usable device";
    case SGEMM_ERR_SCRATCH_LIMIT:
      return "SGEMM_ERR_SCRATCH_LIMIT: split-K partial sums exceed sgemm_noalloc's static scratch array";
    case SGEMM_ERR_BOUNDS:
      return "SGEMM_ERR_BOUNDS: (debug build) a kernel index fell outside its buffer; the access was skipped";
    case -1: return "invalid argument 1 (transA)";
    case -2: return "invalid argument 2 (transB)";
    case -3: return "invalid argument 3 (M < 0)";
    case -4: return "invalid argument 4 (N < 0)";
    case -5: return "invalid argument 5 (K < 0)";
    case -7: return "invalid argument 7 (A is NULL)";
    case -8: return "invalid argument 8 (lda too small)";
    case -9: return "invalid argument 9 (B is NULL)";
    case -10: return "invalid argument 10 (ldb too small)";
    case -12: return "invalid argument 12 (C is NULL)";
    case -13: return "invalid argument 13 (ldc too small)";
    case -14:
      return "invalid argument 14 (strideA < 0; sgemm_ex: workspace NULL although needed, or not 16-byte aligned; "
             "sgemm_workspace_size: bytes is NULL; sgemm_plan_for_device: sm_count <= 0)";
    case -15:
      return "invalid argument 15 (plan is NULL; strideB < 0 in the batched calls; sgemm_ex: workspace_bytes "
             "smaller than sgemm_workspace_size(); sgemm_plan_for_device: pair_clusters < 0)";
    case -16:
      return "invalid argument 16 (strideC < 0, or C matrices of a batch overlap; sgemm_plan_for_device: plan is "
             "NULL)";
    case -17: return "invalid argument 17 (batch_count < 0)";
    case -19: return "invalid argument 19 (plan is NULL)";
    default: return status < 0 ? "invalid argument" : "unknown status";
  }
}

int sgemm_last_cuda_error(void) { return t_last_cuda_error_slot(); }

int sgemm_sync_status(struct CUstream_st* stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned bits = 0;
  e = take_faults(&bits);
  if (e != cudaSuccess) return cuda_fail(e);
  if (bits & kFaultBounds) return SGEMM_ERR_BOUNDS;
  return bits ? SGEMM_ERR_TIMEOUT : SGEMM_OK;
}

int sgemm_bounds_report(unsigned* site, long long* offset) {
  if (!site) return -1;
  if (!offset) return -2;
  unsigned long long w = 0;
  cudaError_t e = take_bounds(&w);
  if (e != cudaSuccess) return cuda_fail(e);
  *site = (unsigned)(w >> 48);
  *offset = (long long)(w & ((1ull << 48) - 1));
  return SGEMM_OK;
}

int sgemm_debug_bounds_enabled(void) {
#ifdef SGEMM_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

int sgemm_selftest_bounds(struct CUstream_st* stream) {
  int dev;
  DeviceState* st;
  int s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned bits = 0;
  unsigned long long w = 0;
  cudaError_t e = cudaStreamSynchronize(cs);
  if (e == cudaSuccess) e = take_faults(&bits);
  if (e == cudaSuccess) e = take_bounds(&w);
  if (e == cudaSuccess) e = launch_bounds_selftest(st->fault, st->bounds, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) return cuda_fail(e);
  return SGEMM_OK;
}

int sgemm_clock_snapshot(unsigned long long* out, int slots, struct CUstream_st* stream) {
  if (!out) return -1;
  if (slots < 1) return -2;
  int dev;
  DeviceState* st;
  int s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  cudaError_t e = launch_clock_snapshot(out, slots, st->sm_count, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SGEMM_OK : cuda_fail(e);
}

int sgemm_selftest_wait_timeout(unsigned timeout_us, struct CUstream_st* stream) {
  if (timeout_us < 1 || timeout_us > 10000000u) return -1;
  int dev;
  DeviceState* st;
  int s = device_state(&dev, &st);
  if (s != SGEMM_OK) return s;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  unsigned bits = 0;
  cudaError_t e = cudaStreamSynchronize(cs);
  if (e == cudaSuccess) e = take_faults(&bits);  // start from a clear fault word
  if (e == cudaSuccess) e = launch_wait_selftest((uint64_t)timeout_us * 1000ull, st->fault, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e == cudaSuccess) e = take_faults(&bits);
  if (e != cudaSuccess) return cuda_fail(e);
  return (bits & kFaultSelftest) ? SGEMM_ERR_TIMEOUT : SGEMM_OK;
}

}  // extern "C"
