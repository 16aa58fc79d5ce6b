// bounds.cuh -- the bounds checks of the debug build (-DSGEMM_DEBUG_BOUNDS) applied to a call's
// buffers: offsets are elements from the buffer's first element, extents come from GemmParams
// (set_extents).  In the normal build every check is the constant true (device_utils.cuh).
#pragma once

#include "device_utils.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {

__device__ __forceinline__ bool c_ok(const GemmParams& p, int64_t off, int64_t n) {
  return in_range(p.fault, p.bounds, kSiteC, off, n, p.c_elems);
}
__device__ __forceinline__ bool ws_ok(const GemmParams& p, int64_t off, int64_t n) {
  return in_range(p.fault, p.bounds, kSiteWs, off, n, p.ws_elems);
}
__device__ __forceinline__ bool a_ok(const GemmParams& p, int64_t off, int64_t n) {
  return in_range(p.fault, p.bounds, kSiteA, off, n, p.a_elems);
}
__device__ __forceinline__ bool b_ok(const GemmParams& p, int64_t off, int64_t n) {
  return in_range(p.fault, p.bounds, kSiteB, off, n, p.b_elems);
}
// Shared- or tensor-memory offset check of the splitters (bytes or columns).
__device__ __forceinline__ bool local_ok(const GemmParams& p, unsigned site, int64_t off, int64_t n, int64_t limit) {
  return in_range(p.fault, p.bounds, site, off, n, limit);
}

}  // namespace sgemm_impl
