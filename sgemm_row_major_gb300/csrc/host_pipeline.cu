// host_pipeline.cu -- sgemm_host(): SGEMM on operands that live in host memory.
//
// Three library-owned streams per device:
//   h2d   copies B once, then op(A) and C of each row block of C, in order;
//   comp  runs the GEMM of each row block as soon as its inputs are in;
//   d2h   copies each finished row block of C back to the host.
// The host link is the slowest part (B alone is a quarter to a half of the
// bytes that cross it), so copies are issued strictly in the order the GEMMs
// need them: the first GEMM starts after B and the first block, and from
// then on the GEMMs, the remaining host-to-device copies and the
// device-to-host copies of finished blocks overlap.  Row blocks rotate
// through kSets device buffer sets; a set is refilled only after its GEMM has
// read it and its C has left.  Device copies get leading dimensions rounded
// up to 4 floats and 256-byte aligned bases from the stream-ordered pool, so
// every block can take the TMA-fed kernels whatever the host layout.  The
// whole sequence is ordered after the work already on the caller's stream,
// and the caller's stream waits for all of it, so the call is asynchronous
// exactly like sgemm().
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSets = 3;  // device buffer sets for row blocks in flight

struct HostPipeDevice {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr, ev_done = nullptr, ev_h2d_end = nullptr, ev_comp_end = nullptr;
  cudaEvent_t ev_in[kSets] = {}, ev_gemm[kSets] = {}, ev_out[kSets] = {};
  cudaMemPool_t pool = nullptr;
  std::mutex mu;  // one enqueue sequence at a time per device (the events are shared)
};
HostPipeDevice g_hp[kMaxDevices];

int64_t round4(int64_t x) { return (x + 3) / 4 * 4; }

cudaError_t setup(int dev, HostPipeDevice** out) {
  HostPipeDevice& d = g_hp[dev];
  std::call_once(d.once, [&] {
    cudaError_t e = cudaStreamCreateWithFlags(&d.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d.comp, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d.d2h, cudaStreamNonBlocking);
    cudaEvent_t* evs[] = {&d.ev_start, &d.ev_done, &d.ev_h2d_end, &d.ev_comp_end};
    for (cudaEvent_t* ev : evs)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int i = 0; i < kSets && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&d.ev_in[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_gemm[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_out[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) {
      cudaMemPoolProps props = {};
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      e = cudaMemPoolCreate(&d.pool, &props);
      if (e == cudaSuccess) {
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep);
      }
    }
    d.err = e;
  });
  *out = &d;
  return d.err;
}

int status_of(cudaError_t e) {
  if (e == cudaSuccess) return SGEMM_OK;
  return e == cudaErrorMemoryAllocation ? SGEMM_ERR_NOMEM : SGEMM_ERR_CUDA;
}

}  // namespace

extern "C" int sgemm_host(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha,
                          const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C,
                          int64_t ldc, struct CUstream_st* stream) {
  // Argument checks of sgemm() (pure host logic; pointers are not dereferenced).
  sgemm_plan_t plan;
  int st = sgemm_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, 152, &plan);
  if (st != SGEMM_OK) return st;
  if (plan.variant == SGEMM_VARIANT_NONE) return SGEMM_OK;
  const bool ta = transA == 'T' || transA == 't' || transA == 'C' || transA == 'c';
  const bool tb = transB == 'T' || transB == 't' || transB == 'C' || transB == 'c';
  const bool reads_ab = K > 0 && alpha != 0.0f;
  const bool reads_c = beta != 0.0f;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return SGEMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
  HostPipeDevice* d = nullptr;
  if (setup(dev, &d) != cudaSuccess) return SGEMM_ERR_CUDA;
  std::lock_guard<std::mutex> lock(d->mu);
  cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);

  // Row blocks of C: about 4 to 8 blocks of a multiple of 128 rows.
  const int64_t nblocks = std::max<int64_t>(1, std::min<int64_t>(8, M / 512));
  int64_t mb = ((M + nblocks - 1) / nblocks + 127) / 128 * 128;
  if (mb > M) mb = M;
  const int nsets = (int)std::min<int64_t>(kSets, (M + mb - 1) / mb);
  // Device leading dimensions (multiples of 4 floats).
  const int64_t b_rows = tb ? N : K, b_cols = tb ? K : N;  // stored B
  const int64_t ldb_d = round4(std::max<int64_t>(b_cols, 1));
  const int64_t a_rows = ta ? K : mb, a_cols = ta ? mb : K;  // stored A block
  const int64_t lda_d = round4(std::max<int64_t>(a_cols, 1));
  const int64_t ldc_d = round4(N);

  float* dB = nullptr;
  float* dA[kSets] = {};
  float* dC[kSets] = {};
  int status = SGEMM_OK;
  auto fail = [&](cudaError_t err) {
    if (status == SGEMM_OK) status = status_of(err);
  };

  e = cudaEventRecord(d->ev_start, user);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d->h2d, d->ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d->comp, d->ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d->d2h, d->ev_start, 0);
  if (e != cudaSuccess) return SGEMM_ERR_CUDA;

  // Buffers (ordered on h2d; the other streams use them only after its events), then B.
  if (reads_ab) {
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dB), (size_t)(b_rows * ldb_d * 4), d->pool, d->h2d);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(dB, (size_t)ldb_d * 4, B, (size_t)ldb * 4, (size_t)b_cols * 4, (size_t)b_rows,
                            cudaMemcpyHostToDevice, d->h2d);
    if (e != cudaSuccess) fail(e);
  }
  for (int i = 0; i < nsets && status == SGEMM_OK; ++i) {
    if (reads_ab) {
      e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dA[i]), (size_t)(a_rows * lda_d * 4), d->pool, d->h2d);
      if (e != cudaSuccess) fail(e);
    }
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dC[i]), (size_t)(mb * ldc_d * 4), d->pool, d->h2d);
    if (e != cudaSuccess) fail(e);
  }

  for (int64_t r0 = 0, blk = 0; r0 < M && status == SGEMM_OK; r0 += mb, ++blk) {
    const int i = (int)(blk % nsets);
    const int64_t rows = std::min<int64_t>(mb, M - r0);
    // h2d: refill set i once its previous GEMM has read it and its C has left
    if (blk >= nsets) {
      e = cudaStreamWaitEvent(d->h2d, d->ev_gemm[i], 0);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(d->h2d, d->ev_out[i], 0);
      if (e != cudaSuccess) { fail(e); break; }
    }
    if (reads_ab) {
      // op(A) rows r0 .. r0+rows: stored rows for 'N', stored columns for 'T'
      if (!ta)
        e = cudaMemcpy2DAsync(dA[i], (size_t)lda_d * 4, A + r0 * lda, (size_t)lda * 4, (size_t)K * 4, (size_t)rows,
                              cudaMemcpyHostToDevice, d->h2d);
      else
        e = cudaMemcpy2DAsync(dA[i], (size_t)lda_d * 4, A + r0, (size_t)lda * 4, (size_t)rows * 4, (size_t)K,
                              cudaMemcpyHostToDevice, d->h2d);
      if (e != cudaSuccess) { fail(e); break; }
    }
    if (reads_c) {
      e = cudaMemcpy2DAsync(dC[i], (size_t)ldc_d * 4, C + r0 * ldc, (size_t)ldc * 4, (size_t)N * 4, (size_t)rows,
                            cudaMemcpyHostToDevice, d->h2d);
      if (e != cudaSuccess) { fail(e); break; }
    }
    e = cudaEventRecord(d->ev_in[i], d->h2d);
    // comp: the block's GEMM (the GEMMs run one after another, each on the whole GPU)
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->comp, d->ev_in[i], 0);
    if (e != cudaSuccess) { fail(e); break; }
    st = sgemm(transA, transB, rows, N, K, alpha, dA[i], lda_d, dB, ldb_d, beta, dC[i], ldc_d,
               reinterpret_cast<struct CUstream_st*>(d->comp));
    if (st != SGEMM_OK) { status = st; break; }
    e = cudaEventRecord(d->ev_gemm[i], d->comp);
    // d2h: the block's C back to the host
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->d2h, d->ev_gemm[i], 0);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(C + r0 * ldc, (size_t)ldc * 4, dC[i], (size_t)ldc_d * 4, (size_t)N * 4, (size_t)rows,
                            cudaMemcpyDeviceToHost, d->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(d->ev_out[i], d->d2h);
    if (e != cudaSuccess) { fail(e); break; }
  }

  // Free in stream order once all three streams are done with the buffers,
  // then make the caller's stream wait for all of it.
  e = cudaEventRecord(d->ev_h2d_end, d->h2d);
  if (e == cudaSuccess) e = cudaEventRecord(d->ev_comp_end, d->comp);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d->d2h, d->ev_h2d_end, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d->d2h, d->ev_comp_end, 0);
  if (e != cudaSuccess) fail(e);
  for (int i = 0; i < kSets; ++i) {
    if (dA[i]) cudaFreeAsync(dA[i], d->d2h);
    if (dC[i]) cudaFreeAsync(dC[i], d->d2h);
  }
  if (dB) cudaFreeAsync(dB, d->d2h);
  e = cudaEventRecord(d->ev_done, d->d2h);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(user, d->ev_done, 0);
  if (e != cudaSuccess) fail(e);
  return status;
}
