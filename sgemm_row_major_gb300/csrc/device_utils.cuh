// device_utils.cuh -- PTX wrappers for sm_103a: mbarriers, TMA tile loads,
// and bounded waits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace sgemm_impl {

// Bits a kernel ORs into the device fault word when a bounded wait gives up.
enum FaultBits : unsigned {
  kFaultFullWait = 1u,     // consumer gave up waiting for a TMA tile
  kFaultEmptyWait = 2u,    // producer gave up waiting for a free stage
  kFaultDrainWait = 4u,    // producer gave up waiting for its copies to land
  kFaultSelftest = 8u,     // the self-test wait gave up (expected)
  kFaultBounds = 16u,      // debug build: an index fell outside its buffer (the access was skipped)
};

// ---- Bounds checks of the debug build (compiled with -DSGEMM_DEBUG_BOUNDS)
//
// The kernels pass every global-memory access (and the computed shared- and
// tensor-memory offsets of the SIMT splitters) through in_range(): elements
// [first, first + count) must lie in [0, limit) of their buffer.  In a debug
// build a violation sets kFaultBounds in the fault word, keeps the first
// violation's site and offset in the bounds word (site << 48 | offset), and the
// caller skips the access -- nothing traps, nothing is read or written out of
// bounds.  In the normal build in_range() is the constant true.
enum BoundsSite : unsigned {
  kSiteC = 1,        // C (epilogues, fixups, split-K reduction, scaling)
  kSiteWs = 2,       // partial-sum workspace (stream-K slots, split-K slices)
  kSiteA = 3,        // A (generic and small-product kernels, split pass, NaN repair)
  kSiteB = 4,        // B
  kSiteSplit = 5,    // split arrays written by the split pass
  kSiteSmem = 6,     // shared-memory offsets of the splitters
  kSiteTmem = 7,     // tensor-memory columns of the splitters
  kSiteSelftest = 8  // the self-test's deliberate out-of-range index (never dereferenced)
};

#ifdef SGEMM_DEBUG_BOUNDS
static __device__ __noinline__ bool bounds_violation(unsigned* fault, unsigned long long* word, unsigned site,
                                              int64_t first) {
  if (fault) atomicOr(fault, (unsigned)kFaultBounds);
  if (word) {
    const unsigned long long off = (unsigned long long)first & ((1ull << 48) - 1);
    atomicCAS(word, 0ull, ((unsigned long long)site << 48) | off);
  }
  return false;
}
__device__ __forceinline__ bool in_range(unsigned* fault, unsigned long long* word, unsigned site, int64_t first,
                                         int64_t count, int64_t limit) {
  return (first >= 0 && count >= 0 && first <= limit - count) ? true : bounds_violation(fault, word, site, first);
}
#else
__device__ __forceinline__ bool in_range(unsigned*, unsigned long long*, unsigned, int64_t, int64_t, int64_t) {
  return true;
}
#endif

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// As mbar_try_wait, but a thread whose phase is not complete yet is suspended
// (issuing nothing) until the phase completes or about `hint_ns` pass.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Slow path of a bounded wait: sleeps on the barrier (suspended threads take
// no issue slots from the warps doing work) until the phase with `parity`
// completes or `timeout_ns` of wall time (the global nanosecond timer) has passed.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// Waits for the mbarrier phase with `parity`; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, timeout_ns);
}

// TMA tile load from a 3-D map {inner, outer, product} into shared memory;
// completion is signalled on `bar` as transaction bytes.  Coordinates are
// element indices; the tensor map zero-fills any part of the box outside the
// tensor.  `inner` times 4 bytes must be a multiple of 16 (tile origins are).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t inner, int32_t outer, int32_t product) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(inner), "r"(outer), "r"(product)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- Tensor memory (TMEM): 512 columns x 128 lanes x 32 bit per SM.
// Warp-collective (.sync.aligned): every lane of the warp must execute these.

// Allocates `ncols` columns (a power of two >= 32) and writes the TMEM base
// address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tmem_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane (shape 32x32b:
// lane = TMEM lane base of the warp + lane id).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Values returned by tmem_ld16 may only be used after tmem_wait_ld().  Passing
// them through an empty volatile asm placed after the wait makes every later
// use depend on an instruction that the compiler keeps behind the wait.
template <int NV>
__device__ __forceinline__ void tmem_ld_ready(float (&v)[NV]) {
#pragma unroll
  for (int i = 0; i < NV; ++i) asm volatile("" : "+f"(v[i]));
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace sgemm_impl
