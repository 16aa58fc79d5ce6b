// host_pipeline.cu -- sgemm_host(): SGEMM on operands that live in host memory.
//
// Three library-owned streams per device:
//   h2d   copies op(A) and C of each row block of C, and B once, in order;
//   comp  runs the GEMM of each row block as soon as its inputs are in;
//   d2h   copies each finished row block of C back to the host.
// The host link is the slowest part (B alone is a quarter to a half of the
// bytes that cross it), so copies are issued strictly in the order the GEMMs
// need them: the first block's op(A) and C, then B in kBChunks K-chunks --
// the GEMM of the first block (of the first kChunkedBlocks blocks) runs one
// per chunk (beta on the first, 1 after), each as soon as its chunk of B is
// in -- then the other blocks; from then on the GEMMs, the remaining
// host-to-device copies and the device-to-host copies of finished blocks
// overlap.  Row blocks rotate
// through kSets device buffer sets; a set is refilled only after its GEMM has
// read it and its C has left.  Device copies get leading dimensions rounded
// up to 4 floats and 256-byte aligned bases from the stream-ordered pool, so
// every block can take the TMA-fed kernels whatever the host layout.  The
// whole sequence is ordered after the work already on the caller's stream,
// and the caller's stream waits for all of it, so the call is asynchronous
// exactly like sgemm().
#include <algorithm>
#include <cstdint>
#include <atomic>
#include <mutex>
#include <vector>

#include "sgemm.h"
#include "sgemm_internal.h"

using sgemm_impl::record_cuda_failure;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSets = 3;     // device buffer sets for row blocks in flight
constexpr int kBChunks = 4;        // K-chunks of B when K is large enough
constexpr int kChunkedBlocks = 1;  // first row blocks whose GEMMs run chunk by chunk as B arrives
                                   // (2 measured no faster: the later blocks' GEMMs then bound the call)

struct HostPipeDevice {
  std::mutex init_mutex;
  std::atomic<bool> ready{false};  // set once the set-up has succeeded (a failed one is retried)
  cudaStream_t h2d = nullptr, comp = nullptr, d2h = nullptr;
  cudaEvent_t ev_start = nullptr, ev_done = nullptr, ev_h2d_end = nullptr, ev_comp_end = nullptr;
  cudaEvent_t ev_in[kSets] = {}, ev_gemm[kSets] = {}, ev_out[kSets] = {};
  cudaEvent_t ev_b[kBChunks] = {};
  cudaMemPool_t pool = nullptr;
  std::mutex mu;  // one enqueue sequence at a time per device (the events are shared)
};
HostPipeDevice g_hp[kMaxDevices];

int64_t round4(int64_t x) { return (x + 3) / 4 * 4; }

// Streams, events and the buffer pool of a device, made by the first call
// there that succeeds; what a failed attempt made is kept and the rest is
// made by the next call.
cudaError_t setup(int dev, HostPipeDevice** out) {
  HostPipeDevice& d = g_hp[dev];
  *out = &d;
  if (d.ready.load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(d.init_mutex);
  if (d.ready.load(std::memory_order_relaxed)) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  for (cudaStream_t* s : {&d.h2d, &d.comp, &d.d2h})
    if (e == cudaSuccess && !*s) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  std::vector<cudaEvent_t*> evs = {&d.ev_start, &d.ev_done, &d.ev_h2d_end, &d.ev_comp_end};
  for (int i = 0; i < kBChunks; ++i) evs.push_back(&d.ev_b[i]);
  for (int i = 0; i < kSets; ++i) {
    evs.push_back(&d.ev_in[i]);
    evs.push_back(&d.ev_gemm[i]);
    evs.push_back(&d.ev_out[i]);
  }
  for (cudaEvent_t* ev : evs)
    if (e == cudaSuccess && !*ev) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e == cudaSuccess && !d.pool) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    e = cudaMemPoolCreate(&pool, &props);
    if (e == cudaSuccess) {
      uint64_t keep = UINT64_MAX;  // keep freed buffers for the next call (sgemm_release_workspace trims)
      e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      if (e == cudaSuccess) d.pool = pool;
      else (void)cudaMemPoolDestroy(pool);
    }
  }
  if (e == cudaSuccess) d.ready.store(true, std::memory_order_release);
  return e;
}

int status_of(cudaError_t e) {
  if (e == cudaSuccess) return SGEMM_OK;
  record_cuda_failure(e);
  return e == cudaErrorMemoryAllocation ? SGEMM_ERR_NOMEM : SGEMM_ERR_CUDA;
}

}  // namespace

cudaError_t sgemm_impl::trim_host_pool(int dev, size_t keep_bytes) {
  if (dev < 0 || dev >= kMaxDevices) return cudaSuccess;
  HostPipeDevice& d = g_hp[dev];
  std::lock_guard<std::mutex> lock(d.mu);
  return d.pool ? cudaMemPoolTrimTo(d.pool, keep_bytes) : cudaSuccess;
}

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
  if (e != cudaSuccess) return record_cuda_failure(e);
  if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED;
  HostPipeDevice* d = nullptr;
  e = setup(dev, &d);
  if (e != cudaSuccess) return record_cuda_failure(e);
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
  // K-chunks of B: multiples of 32 floats, so every chunk of A and B starts 128-byte aligned
  const int nq = (reads_ab && K >= kBChunks * 256) ? kBChunks : 1;
  const int64_t kc = ((K + nq - 1) / nq + 31) / 32 * 32;

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
  if (e != cudaSuccess) return record_cuda_failure(e);

  // Buffers (ordered on h2d; the other streams use them only after its events).
  if (reads_ab) {
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dB), (size_t)(b_rows * ldb_d * 4), d->pool, d->h2d);
    if (e != cudaSuccess) fail(e);
  }
  // B's K-chunk q: stored rows q*kc.. for 'N', stored columns q*kc.. for 'T'
  auto copy_b_chunk = [&](int q) {
    const int64_t k0 = q * kc, kq = std::min<int64_t>(kc, K - k0);
    if (!tb)
      return cudaMemcpy2DAsync(dB + k0 * ldb_d, (size_t)ldb_d * 4, B + k0 * ldb, (size_t)ldb * 4, (size_t)N * 4,
                               (size_t)kq, cudaMemcpyHostToDevice, d->h2d);
    return cudaMemcpy2DAsync(dB + k0, (size_t)ldb_d * 4, B + k0, (size_t)ldb * 4, (size_t)kq * 4, (size_t)N,
                             cudaMemcpyHostToDevice, d->h2d);
  };
  for (int i = 0; i < nsets && status == SGEMM_OK; ++i) {
    if (reads_ab) {
      e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dA[i]), (size_t)(a_rows * lda_d * 4), d->pool, d->h2d);
      if (e != cudaSuccess) fail(e);
    }
    e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&dC[i]), (size_t)(mb * ldc_d * 4), d->pool, d->h2d);
    if (e != cudaSuccess) fail(e);
  }

  const int64_t nblk = (M + mb - 1) / mb;
  // the first blocks' GEMMs run chunk by chunk while B arrives
  const int64_t nchunked = (reads_ab && nq > 1) ? std::min<int64_t>(kChunkedBlocks, nblk) : 0;

  // h2d: op(A) rows of block blk (stored rows for 'N', stored columns for 'T') and its C, into set
  // blk % nsets once that set's previous GEMM has read it and its C has left
  auto copy_in = [&](int64_t blk) -> cudaError_t {
    const int i = (int)(blk % nsets);
    const int64_t r0 = blk * mb, rows = std::min<int64_t>(mb, M - r0);
    cudaError_t err = cudaSuccess;
    if (blk >= nsets) {
      err = cudaStreamWaitEvent(d->h2d, d->ev_gemm[i], 0);
      if (err == cudaSuccess) err = cudaStreamWaitEvent(d->h2d, d->ev_out[i], 0);
    }
    if (err == cudaSuccess && reads_ab)
      err = !ta ? cudaMemcpy2DAsync(dA[i], (size_t)lda_d * 4, A + r0 * lda, (size_t)lda * 4, (size_t)K * 4,
                                    (size_t)rows, cudaMemcpyHostToDevice, d->h2d)
                : cudaMemcpy2DAsync(dA[i], (size_t)lda_d * 4, A + r0, (size_t)lda * 4, (size_t)rows * 4, (size_t)K,
                                    cudaMemcpyHostToDevice, d->h2d);
    if (err == cudaSuccess && reads_c)
      err = cudaMemcpy2DAsync(dC[i], (size_t)ldc_d * 4, C + r0 * ldc, (size_t)ldc * 4, (size_t)N * 4, (size_t)rows,
                              cudaMemcpyHostToDevice, d->h2d);
    if (err == cudaSuccess) err = cudaEventRecord(d->ev_in[i], d->h2d);
    return err;
  };
  // comp: the GEMM of block blk over K-chunk q (q < 0: all of K):
  // C = alpha*op(A)[:, chunk]*op(B)[chunk, :] + (first chunk ? beta : 1)*C
  auto gemm = [&](int64_t blk, int q) -> int {
    const int i = (int)(blk % nsets);
    const int64_t rows = std::min<int64_t>(mb, M - blk * mb);
    const int64_t k0 = q < 0 ? 0 : q * kc, kq = q < 0 ? K : std::min<int64_t>(kc, K - k0);
    const float* a_q = dA[i] ? (ta ? dA[i] + k0 * lda_d : dA[i] + k0) : nullptr;
    const float* b_q = dB ? (tb ? dB + k0 : dB + k0 * ldb_d) : nullptr;
    return sgemm(transA, transB, rows, N, kq, alpha, a_q, lda_d, b_q, ldb_d, q > 0 ? 1.0f : beta, dC[i], ldc_d,
                 reinterpret_cast<struct CUstream_st*>(d->comp));
  };
  // comp -> d2h: block blk's C back to the host once its GEMM is done
  auto copy_out = [&](int64_t blk) -> cudaError_t {
    const int i = (int)(blk % nsets);
    const int64_t r0 = blk * mb, rows = std::min<int64_t>(mb, M - r0);
    cudaError_t err = cudaEventRecord(d->ev_gemm[i], d->comp);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(d->d2h, d->ev_gemm[i], 0);
    if (err == cudaSuccess)
      err = cudaMemcpy2DAsync(C + r0 * ldc, (size_t)ldc * 4, dC[i], (size_t)ldc_d * 4, (size_t)N * 4, (size_t)rows,
                              cudaMemcpyDeviceToHost, d->d2h);
    if (err == cudaSuccess) err = cudaEventRecord(d->ev_out[i], d->d2h);
    return err;
  };

  if (status == SGEMM_OK && nchunked > 0) {
    // h2d order: block 0, B chunk 0, the other chunked blocks, the rest of B
    e = copy_in(0);
    if (e == cudaSuccess) e = copy_b_chunk(0);
    if (e == cudaSuccess) e = cudaEventRecord(d->ev_b[0], d->h2d);
    for (int64_t blk = 1; blk < nchunked && e == cudaSuccess; ++blk) e = copy_in(blk);
    for (int q = 1; q < nq && e == cudaSuccess; ++q) {
      e = copy_b_chunk(q);
      if (e == cudaSuccess) e = cudaEventRecord(d->ev_b[q], d->h2d);
    }
    // comp: chunk q of every chunked block as soon as chunk q of B is in
    for (int q = 0; q < nq && e == cudaSuccess && status == SGEMM_OK; ++q) {
      e = cudaStreamWaitEvent(d->comp, d->ev_b[q], 0);
      for (int64_t blk = 0; blk < nchunked && e == cudaSuccess; ++blk) {
        if (q == 0) e = cudaStreamWaitEvent(d->comp, d->ev_in[blk % nsets], 0);
        if (e != cudaSuccess) break;
        st = gemm(blk, q);
        if (st != SGEMM_OK) { status = st; break; }
        if (q == nq - 1) e = copy_out(blk);
      }
    }
    if (e != cudaSuccess) fail(e);
  } else if (status == SGEMM_OK && reads_ab) {
    e = copy_b_chunk(0);  // nq == 1: all of B, before any block
    if (e != cudaSuccess) fail(e);
  }
  for (int64_t blk = nchunked; blk < nblk && status == SGEMM_OK; ++blk) {
    e = copy_in(blk);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(d->comp, d->ev_in[blk % nsets], 0);
    if (e != cudaSuccess) { fail(e); break; }
    st = gemm(blk, -1);
    if (st != SGEMM_OK) { status = st; break; }
    e = copy_out(blk);
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
