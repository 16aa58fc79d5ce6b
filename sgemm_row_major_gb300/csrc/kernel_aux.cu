// kernel_aux.cu -- the small kernels around the GEMM kernels: the split-K
// reduction with the fused alpha/beta epilogue, C = beta*C for alpha == 0 or
// K == 0, the bounded-wait self-test, the per-SM clock snapshot, and the
// device fault word.
#include "bounds.cuh"
#include "device_utils.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {

// One fault word per device (each device that loads the library has its own
// copy of a __device__ variable).  Kernels receive its address in GemmParams.
__device__ unsigned g_fault_word;
// Debug build: the first bounds violation of the device (site << 48 | offset), 0 when none.
__device__ unsigned long long g_bounds_word;

namespace {

__device__ __forceinline__ float epilogue(float alpha, float beta, float v, const float* c) {
  return beta == 0.0f ? alpha * v : fmaf(alpha, v, beta * *c);
}

// Sums the split partial tiles in slice order 0, 1, ..., split-1 (a fixed
// order, so the result does not depend on scheduling), then applies
// C = alpha * sum + beta * C.  One thread per 4 consecutive columns of one
// row of one product; the workspace is [product][slice][M][ws_ld].
template <bool CVEC>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const GemmParams p, int split) {
  const int64_t groups = (p.N + 3) / 4;
  const int64_t per_product = (int64_t)p.M * groups;
  const int64_t total = per_product * p.batch;
  const int64_t slice = (int64_t)p.M * p.ws_ld;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t prod = g / per_product;
    const int64_t r = g - prod * per_product;
    const int row = (int)(r / groups);
    const int col = (int)(r % groups) * 4;
    const int64_t wi = prod * split * slice + (int64_t)row * p.ws_ld + col;
    const float* w = p.ws + wi;
    float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int z = 0; z < split; ++z) {
      if (!ws_ok(p, wi + z * slice, 4)) continue;
      const float4 u = *reinterpret_cast<const float4*>(w + z * slice);
      if (z == 0) v = u;
      else { v.x += u.x; v.y += u.y; v.z += u.z; v.w += u.w; }
    }
    const int64_t ci = prod * p.stride_c + (int64_t)row * p.ldc + col;
    if (!c_ok(p, ci, min(4, p.N - col))) continue;
    float* c = p.C + ci;
    if (CVEC && col + 3 < p.N) {
      float4 o;
      if (p.beta == 0.0f) {
        o = make_float4(p.alpha * v.x, p.alpha * v.y, p.alpha * v.z, p.alpha * v.w);
      } else {
        const float4 old = *reinterpret_cast<const float4*>(c);
        o = make_float4(fmaf(p.alpha, v.x, p.beta * old.x), fmaf(p.alpha, v.y, p.beta * old.y),
                        fmaf(p.alpha, v.z, p.beta * old.z), fmaf(p.alpha, v.w, p.beta * old.w));
      }
      *reinterpret_cast<float4*>(c) = o;
    } else {
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (col + q < p.N) c[q] = epilogue(p.alpha, p.beta, vv[q], c + q);
    }
  }
}

// C = beta * C (every product); with beta == 0, C = 0 without reading C.
__global__ void __launch_bounds__(256) scale_kernel(const GemmParams p) {
  const int64_t per_product = (int64_t)p.M * p.N;
  const int64_t total = per_product * p.batch;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t prod = e / per_product;
    const int64_t r = e - prod * per_product;
    const int64_t ci = prod * p.stride_c + (r / p.N) * p.ldc + (r % p.N);
    if (!c_ok(p, ci, 1)) continue;
    float* c = p.C + ci;
    *c = p.beta == 0.0f ? 0.0f : p.beta * *c;
  }
}

// Waits on a shared-memory mbarrier that nothing arrives on.  The wait must
// give up after `timeout_ns` and record kFaultSelftest; no copy is in flight.
__global__ void wait_selftest_kernel(uint64_t timeout_ns, unsigned* fault) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(b, 0, timeout_ns)) atomicOr(fault, (unsigned)kFaultSelftest);
}

// Thread 0 of every CTA writes its SM's cycle counter and the global nanosecond
// timer to out[2 * smid], out[2 * smid + 1] (a later CTA on the same SM
// overwrites an earlier one).  Two snapshots around a stretch of work give each
// SM's average clock over it: cycles / nanoseconds.
__global__ void clock_snapshot_kernel(unsigned long long* out, int slots) {
  if (threadIdx.x != 0) return;
  unsigned smid;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
  if ((int)smid >= slots) return;
  const unsigned long long t = global_timer_ns();
  out[2 * smid] = (unsigned long long)clock64();
  out[2 * smid + 1] = t;
}

// Checks an index one past its limit: in the debug build the check records it and declines the
// access (nothing is dereferenced); in the normal build there is no check and nothing happens.
__global__ void bounds_selftest_kernel(unsigned* fault, unsigned long long* word) {
  (void)in_range(fault, word, kSiteSelftest, 64, 1, 64);
}

unsigned grid_for(int64_t work, int per_block) {
  int64_t blocks = (work + per_block - 1) / per_block;
  if (blocks < 1) blocks = 1;
  if (blocks > 152 * 32) blocks = 152 * 32;  // grid-stride beyond ~32 blocks per SM
  return (unsigned)blocks;
}

}  // namespace

cudaError_t launch_splitk_reduce(const GemmParams& p, int split, cudaStream_t stream) {
  const int64_t work = (int64_t)p.batch * p.M * ((p.N + 3) / 4);
  if (p.c_vec)
    splitk_reduce_kernel<true><<<grid_for(work, 256), 256, 0, stream>>>(p, split);
  else
    splitk_reduce_kernel<false><<<grid_for(work, 256), 256, 0, stream>>>(p, split);
  return cudaGetLastError();
}

cudaError_t launch_scale(const GemmParams& p, cudaStream_t stream) {
  scale_kernel<<<grid_for((int64_t)p.batch * p.M * p.N, 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, unsigned* fault, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns, fault);
  return cudaGetLastError();
}

cudaError_t launch_clock_snapshot(unsigned long long* out, int slots, int sm_count, cudaStream_t stream) {
  clock_snapshot_kernel<<<(unsigned)(4 * sm_count), 32, 0, stream>>>(out, slots);
  return cudaGetLastError();
}

cudaError_t launch_bounds_selftest(unsigned* fault, unsigned long long* word, cudaStream_t stream) {
  bounds_selftest_kernel<<<1, 1, 0, stream>>>(fault, word);
  return cudaGetLastError();
}

cudaError_t fault_word(unsigned** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_fault_word);
}

cudaError_t bounds_word(unsigned long long** ptr) {
  return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_bounds_word);
}

cudaError_t take_bounds(unsigned long long* word) {
  cudaError_t e = cudaMemcpyFromSymbol(word, g_bounds_word, sizeof(unsigned long long));
  if (e != cudaSuccess) return e;
  const unsigned long long zero = 0;
  return cudaMemcpyToSymbol(g_bounds_word, &zero, sizeof(unsigned long long));
}

cudaError_t take_faults(unsigned* bits) {
  cudaError_t e = cudaMemcpyFromSymbol(bits, g_fault_word, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned));
}

}  // namespace sgemm_impl
