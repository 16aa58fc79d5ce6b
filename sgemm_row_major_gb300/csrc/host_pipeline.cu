// host_pipeline.cu -- sgemm_host(): SGEMM on operands that live in host memory.
//
// B is copied to the device once; op(A) and C then move in row blocks of C
// on two library-owned streams, so the host-to-device copies of block i and
// the device-to-host copy of block i-1 overlap the GEMM of the other block.
// Device copies get leading dimensions rounded up to 4 floats and 256-byte
// aligned bases from the stream-ordered pool, so every block can take the
// TMA-fed kernels whatever the host layout.  The whole sequence is ordered
// after the work already on the caller's stream, and the caller's stream waits
// for all of it, so the call is asynchronous exactly like sgemm().
#include <algorithm>
#include <cstdint>
#include <mutex>

#include "sgemm.h"
#include "sgemm_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct HostPipeDevice {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  cudaStream_t s[2] = {nullptr, nullptr};
  cudaEvent_t ev_start = nullptr, ev_b = nullptr, ev_done[2] = {nullptr, nullptr};
  cudaMemPool_t pool = nullptr;
  std::mutex mu;  // one enqueue sequence at a time per device (the events are shared)
};
HostPipeDevice g_hp[kMaxDevices];

int64_t round4(int64_t x) { return (x + 3) / 4 * 4; }

cudaError_t setup(int dev, HostPipeDevice** out) {
  HostPipeDevice& d = g_hp[dev];
  std::call_once(d.once, [&] {
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&d.s[i], cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_b, cudaEventDisableTiming);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&d.ev_done[i], cudaEventDisableTiming);
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
  // Device leading dimensions (multiples of 4 floats).
  const int64_t b_rows = tb ? N : K, b_cols = tb ? K : N;  // stored B
  const int64_t ldb_d = round4(std::max<int64_t>(b_cols, 1));
  const int64_t a_rows = ta ? K : mb, a_cols = ta ? mb : K;  // stored A block
  const int64_t lda_d = round4(std::max<int64_t>(a_cols, 1));
  const int64_t ldc_d = round4(N);

  float* dB = nullptr;
  float* dA[2] = {nullptr, nullptr};
  float* dC[2] = {nullptr, nullptr};
  int status = SGEMM_OK;
  auto fail = [&](cudaError_t err) {
    if (status == SGEMM_OK) status = status_of(err);
  };

  e = cudaEventRecord(d->ev_start, user);
  for (int i = 0; i < 2 && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(d->s[i], d->ev_start, 0);
  if (e != cudaSuccess) return SGEMM_ERR_CUDA;

  // B once, on stream 0.
  if (reads_ab) {
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dB), (size_t)(b_rows * ldb_d * 4), d->pool, d->s[0]);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(dB, (size_t)ldb_d * 4, B, (size_t)ldb * 4, (size_t)b_cols * 4, (size_t)b_rows,
                            cudaMemcpyHostToDevice, d->s[0]);
    if (e == cudaSuccess) e = cudaEventRecord(d->ev_b, d->s[0]);
    if (e != cudaSuccess) fail(e);
  }
  for (int i = 0; i < 2 && status == SGEMM_OK; ++i) {
    if (reads_ab) {
      e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dA[i]), (size_t)(a_rows * lda_d * 4), d->pool, d->s[i]);
      if (e != cudaSuccess) fail(e);
    }
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dC[i]), (size_t)(mb * ldc_d * 4), d->pool, d->s[i]);
    if (e != cudaSuccess) fail(e);
  }

  for (int64_t r0 = 0, blk = 0; r0 < M && status == SGEMM_OK; r0 += mb, ++blk) {
    const int i = (int)(blk & 1);
    cudaStream_t s = d->s[i];
    const int64_t rows = std::min<int64_t>(mb, M - r0);
    if (reads_ab) {
      // op(A) rows r0 .. r0+rows: stored rows for 'N', stored columns for 'T'
      if (!ta)
        e = cudaMemcpy2DAsync(dA[i], (size_t)lda_d * 4, A + r0 * lda, (size_t)lda * 4, (size_t)K * 4, (size_t)rows,
                              cudaMemcpyHostToDevice, s);
      else
        e = cudaMemcpy2DAsync(dA[i], (size_t)lda_d * 4, A + r0, (size_t)lda * 4, (size_t)rows * 4, (size_t)K,
                              cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) { fail(e); break; }
    }
    if (reads_c) {
      e = cudaMemcpy2DAsync(dC[i], (size_t)ldc_d * 4, C + r0 * ldc, (size_t)ldc * 4, (size_t)N * 4, (size_t)rows,
                            cudaMemcpyHostToDevice, s);
      if (e != cudaSuccess) { fail(e); break; }
    }
    // only the GEMM needs B; stream 1's first copies already ran beside B's
    if (reads_ab && i == 1 && blk == 1) {
      e = cudaStreamWaitEvent(s, d->ev_b, 0);
      if (e != cudaSuccess) { fail(e); break; }
    }
    st = sgemm(transA, transB, rows, N, K, alpha, dA[i], lda_d, dB, ldb_d, beta, dC[i], ldc_d,
               reinterpret_cast<struct CUstream_st*>(s));
    if (st != SGEMM_OK) { status = st; break; }
    e = cudaMemcpy2DAsync(C + r0 * ldc, (size_t)ldc * 4, dC[i], (size_t)ldc_d * 4, (size_t)N * 4, (size_t)rows,
                          cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) { fail(e); break; }
  }

  // Free in stream order and make the caller's stream wait for both streams.
  for (int i = 0; i < 2; ++i) {
    if (dA[i]) cudaFreeAsync(dA[i], d->s[i]);
    if (dC[i]) cudaFreeAsync(dC[i], d->s[i]);
  }
  if (dB) {
    // stream 1 may still read B: free it after both streams are done
    cudaEventRecord(d->ev_done[1], d->s[1]);
    cudaStreamWaitEvent(d->s[0], d->ev_done[1], 0);
    cudaFreeAsync(dB, d->s[0]);
  }
  for (int i = 0; i < 2; ++i) {
    e = cudaEventRecord(d->ev_done[i], d->s[i]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(user, d->ev_done[i], 0);
    if (e != cudaSuccess) fail(e);
  }
  return status;
}
