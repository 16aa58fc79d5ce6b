// noalloc.cu -- sgemm_noalloc(): the same SGEMM as sgemm(), for callers that
// cannot allocate device memory while the call runs.
//
// Who needs it: sgemm() takes its split-K partial sums from a stream-ordered
// memory pool, which may grow (allocate) on a call.  Some callers cannot allow
// that: an application that has already handed nearly all device memory to
// its own allocator (so a new allocation can fail at an arbitrary call), or
// latency-critical code that cannot absorb the cost of a pool growing in the
// middle of its work.  sgemm_noalloc() gives them the same kernels with the
// partial sums in a fixed array that is part of the library image itself.
//
// The scratch array: a file-scope __device__ array of
// SGEMM_NOALLOC_SCRATCH_BYTES.  Every GPU that loads the library holds one
// copy of it until the process exits.  Host code cannot use the array's name
// as a device address (on the host it names a stand-in object), so the
// device address is looked up with cudaGetSymbolAddress once per device, with
// that device current, on the first sgemm_noalloc() call there; that first
// call should therefore come before any stream capture (a set-up that fails,
// for instance inside a capture, returns SGEMM_ERR_CUDA and is tried again
// by the next call).  Nothing in the array
// needs to start at zero: the GEMM kernel writes every partial sum the
// reduction reads in the same call.  All calls on a device share the array,
// so two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it.
#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>

#include "kernel_small.h"
#include "kernel_tma.cuh"
#include "sgemm.h"
#include "sgemm_internal.h"

using namespace sgemm_impl;

namespace {

static __device__ __align__(256) float g_noalloc_scratch[SGEMM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

constexpr int kMaxDevices = 64;

struct NoallocDevice {
  std::mutex init_mutex;
  std::atomic<bool> ready{false};  // set once the set-up has succeeded (a failed one is retried)
  int sm_count = 0;
  int pair_clusters = 0;     // co-resident CTA-pair clusters (0: the CTA-pair kernel cannot run here)
  unsigned* fault = nullptr;
  unsigned long long* bounds = nullptr;  // debug build: first bounds violation
  float* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};
NoallocDevice g_nd[kMaxDevices];

// Per-device set-up with the device current: SM count, co-resident CTA-pair
// clusters (the same query sgemm() plans with), fault word, scratch address
// and kernel attributes.  No allocation happens here.  Done by the first call
// on the device that succeeds in it; a failed set-up is tried again next call.
cudaError_t setup(int dev, NoallocDevice** out) {
  NoallocDevice& d = g_nd[dev];
  *out = &d;
  if (d.ready.load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(d.init_mutex);
  if (d.ready.load(std::memory_order_relaxed)) return cudaSuccess;
  cudaError_t e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = fault_word(&d.fault);
  if (e == cudaSuccess) e = bounds_word(&d.bounds);
  if (e == cudaSuccess) e = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.scratch), g_noalloc_scratch);
  if (e == cudaSuccess) e = prepare_tma_op_nn();
  if (e == cudaSuccess) e = prepare_tma_op_nt();
  if (e == cudaSuccess) e = prepare_tma_op_tn();
  if (e == cudaSuccess) e = prepare_tma_op_tt();
  if (e == cudaSuccess) e = prepare_tf32x3();
  if (e == cudaSuccess) e = prepare_small_gemm();
  if (e == cudaSuccess) e = prepare_tc_pair();
  if (e == cudaSuccess) d.pair_clusters = pair_clusters_or_none();
  if (e == cudaSuccess) d.ready.store(true, std::memory_order_release);
  return e;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" int sgemm_noalloc(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                             const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                             int64_t ldc, struct CUstream_st* stream) {
  // Same argument checks and the same planner as sgemm() (pure host logic);
  // a first pass with a nominal SM count rejects bad arguments before any
  // CUDA call, the second uses the device's SM count.
  sgemm_plan_t plan;
  int st = sgemm_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, 152, &plan);
  if (st != SGEMM_OK) return st;
  if (plan.variant == SGEMM_VARIANT_NONE) return SGEMM_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda_failure(e);
  if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
  NoallocDevice* nd = nullptr;
  e = setup(dev, &nd);
  if (e != cudaSuccess) return record_cuda_failure(e);
  st = plan_without_split_arrays(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nd->sm_count,
                                 nd->pair_clusters, &plan);
  if (st != SGEMM_OK) return st;
  if ((uint64_t)plan.workspace_bytes > (uint64_t)SGEMM_NOALLOC_SCRATCH_BYTES) return SGEMM_ERR_SCRATCH_LIMIT;

  const bool ta = transA == 'T' || transA == 't' || transA == 'C' || transA == 'c';
  const bool tb = transB == 'T' || transB == 't' || transB == 'C' || transB == 'c';
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  GemmParams p{};
  p.M = (int)M;
  p.N = (int)N;
  p.K = (int)K;
  p.alpha = alpha;
  p.beta = beta;
  p.A = A;
  p.B = B;
  p.C = C;
  p.lda = lda;
  p.ldb = ldb;
  p.ta = ta ? 1 : 0;
  p.tb = tb ? 1 : 0;
  p.ldc = ldc;
  p.c_vec = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0;
  p.timeout_ns = wait_timeout_ns();
  p.fault = nd->fault;
  set_extents(&p, plan.workspace_bytes, nd->bounds);

  if (plan.variant == SGEMM_VARIANT_SCALE) {
    e = launch_scale(p, cs);
    return e == cudaSuccess ? SGEMM_OK : record_cuda_failure(e);
  }
  const int split = plan.split_k;
  p.tiles_m = (int)ceil_div(M, plan.tile_m);
  p.tiles_n = (int)ceil_div(N, plan.tile_n);
  p.k_tiles_per_split = (int)ceil_div(ceil_div(K, plan.tile_k), split);
  p.ws_ld = ceil_div(N, 4) * 4;
  p.ws = plan.workspace_bytes > 0 ? nd->scratch : nullptr;
  set_schedule(plan, &p);

  if (plan.variant == SGEMM_VARIANT_GENERIC) {
    e = launch_generic_gemm(ta, tb, p, split, cs);
  } else if (plan.variant == SGEMM_VARIANT_SMALL) {
    e = launch_small_gemm(ta, tb, p, (int)plan.grid_x, cs);
  } else {
    CUtensorMap mapA, mapB;
    int box_m, box_n;
    operand_boxes(plan, &box_m, &box_n);
    e = encode_operand_maps(ta, tb, M, N, K, A, lda, 0, B, ldb, 0, 1, box_m, box_n, plan.tile_k, &mapA, &mapB, &p.za,
                            &p.zb);
    if (e != cudaSuccess) return record_cuda_failure(e);
    const TmaTile tile = plan.variant == SGEMM_VARIANT_TMA_128x128 ? TmaTile::k128x128 : TmaTile::k64x256;
    if (plan.variant == SGEMM_VARIANT_TC_TF32X3 || plan.variant == SGEMM_VARIANT_TC_GROUPED) {
      e = launch_tf32x3(ta, tb, plan.variant == SGEMM_VARIANT_TC_GROUPED ? 128 / plan.tile_m : 1, mapA, mapB, p,
                        cs);
      if (e == cudaSuccess && plan.kernel_launches > 1) e = launch_streamk_fixup(p, (int)plan.sk_tiles, cs);
    } else if (plan.variant == SGEMM_VARIANT_TC_PAIR) {
      e = launch_tc_pair(ta, tb, mapA, mapB, p, cs);
      if (e == cudaSuccess && plan.kernel_launches > 1) e = launch_pair_fixup(p, (int)plan.sk_tiles, cs);
    } else if (!ta && !tb) e = launch_tma_op_nn(tile, mapA, mapB, p, split, cs);
    else if (!ta && tb) e = launch_tma_op_nt(tile, mapA, mapB, p, split, cs);
    else if (ta && !tb) e = launch_tma_op_tn(tile, mapA, mapB, p, split, cs);
    else e = launch_tma_op_tt(tile, mapA, mapB, p, split, cs);
  }
  if (e == cudaSuccess && split > 1 && plan.variant != SGEMM_VARIANT_TC_TF32X3 &&
      plan.variant != SGEMM_VARIANT_TC_PAIR)
    e = launch_splitk_reduce(p, split, cs);
  return e == cudaSuccess ? SGEMM_OK : record_cuda_failure(e);
}
