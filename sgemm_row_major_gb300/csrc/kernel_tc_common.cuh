// kernel_tc_common.cuh -- device helpers shared by the tensor-core SGEMM
// kernels (kernel_tf32x3.cu: one CTA per tile; kernel_tc_pair.cu: CTA pairs;
// kernel_presplit.cu: CTA pairs on split operands): the 3xTF32 operand split,
// the shared-memory matrix descriptor of the K-major tiles, warp-level
// bounded waits, the tile raster, the persistent data-parallel + stream-K
// schedule, and the cluster, pair-TMEM and cross-CTA barrier operations of
// the CTA-pair kernels.
#pragma once

#include "bounds.cuh"
#include "device_utils.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace tc {

// Shared-memory matrix descriptor of a K-major tile with the 128-byte swizzle:
// rows of 128 bytes (32 TF32 values of K), 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= (uint64_t)((smem_byte_addr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)(16u >> 4) << 16;                    // leading byte offset (unused: K fits one atom)
  d |= (uint64_t)(1024u >> 4) << 32;                  // stride byte offset: next 8 rows
  d |= (uint64_t)1 << 46;                             // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                             // 128-byte swizzle
  return d;
}

// Warp-level bounded wait: lane 0 polls, then every lane confirms the phase
// (an immediate success) so each thread has its own acquire.  Warp-uniform.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const int lane = threadIdx.x & 31;
  bool ok = true;
  if (lane == 0) ok = mbar_wait(bar, parity, timeout_ns);
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  if (ok) ok = mbar_wait(bar, parity, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

// x rounded to TF32 (10 explicit mantissa bits), to nearest with ties away
// from zero: add half of the dropped range to the magnitude bits, then clear
// them (a carry into the exponent is the correct rounding).
__device__ __forceinline__ float tf32_round(float x) {
  return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

__device__ __forceinline__ void split4(const float4 x, float4& hi, float4& lo) {
  hi = make_float4(tf32_round(x.x), tf32_round(x.y), tf32_round(x.z), tf32_round(x.w));
  // lo = x - hi (exact), two at a time: fma(hi, -1, x) rounds an exact value
  const float2 m1 = make_float2(-1.0f, -1.0f);
  const float2 l01 = __ffma2_rn(make_float2(hi.x, hi.y), m1, make_float2(x.x, x.y));
  const float2 l23 = __ffma2_rn(make_float2(hi.z, hi.w), m1, make_float2(x.z, x.w));
  lo = make_float4(l01.x, l01.y, l23.x, l23.y);
}

// ---- Results the split cannot carry
//
// The split fails for two kinds of input: a finite x at or above (2 - 2^-11) *
// 2^127 in magnitude, whose hi part rounds to Inf (lo = x - hi is then -Inf),
// and x = +-Inf (hi = Inf, lo = Inf - Inf = NaN).  Every tensor-core product
// such an element takes part in is then Inf - Inf, Inf * 0 or NaN, so the
// folded sum is NaN, although the definition C_ij = sum_k op(A)_ik op(B)_kj
// (klklkl10086.github.io "Sgemm单精度矩阵乘法", 问题定义) gives a finite sum
// for the first kind and +-Inf (or NaN) for the second.  Nothing else makes
// the folded sum NaN except a NaN operand (or Inf - Inf between products),
// where the definition gives NaN too.  So the epilogues test the folded sums
// of a thread once per tile (a chain of packed adds and one compare) and
// compute each NaN sum again with FP32 FMAs over op(A)'s row and op(B)'s
// column, k ascending, 32-k partial sums added into a running sum as the
// fold does: IEEE FP32 semantics for Inf and NaN, the per-element error of a
// plain FP32 dot product for finite results.  The hot loop gains nothing;
// calls whose results are mostly NaN or +-Inf run this slow path for them.

// sum_k a[k * as] * b[k * bs] with FP32 FMAs in k order.  A NaN running sum
// is final, so the loop stops at it.
__device__ __forceinline__ float fp32_dot(const float* __restrict__ a, int64_t as, const float* __restrict__ b,
                                          int64_t bs, int K) {
  float sum = 0.0f;
#pragma unroll 1
  for (int k0 = 0; k0 < K; k0 += 32) {
    const int k1 = min(K, k0 + 32);
    float part = 0.0f;
#pragma unroll 1
    for (int k = k0; k < k1; ++k) part = __fmaf_rn(a[(int64_t)k * as], b[(int64_t)k * bs], part);
    sum = __fadd_rn(sum, part);
    if (sum != sum) break;
  }
  return sum;
}

// True when some value of m is NaN or +-Inf (or the packed sum of the values
// overflows, which only sends the caller to its per-element NaN test).
template <int N2>
__device__ __forceinline__ bool any_nonfinite(const float2 (&m)[N2]) {
  float2 s0 = m[0], s1 = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int e = 1; e < N2; ++e) {
    if (e & 1) s1 = __fadd2_rn(s1, m[e]);
    else       s0 = __fadd2_rn(s0, m[e]);
  }
  s0 = __fadd2_rn(s0, s1);
  return !(fabsf(s0.x + s0.y) <= 3.402823466e38f);
}

// Replaces each NaN sum v[i] (row `row`, column col0 + i < N of product
// `prod`, i < n) by the FP32 dot product of op(A)'s row and op(B)'s column.
// v is a local array: only this cold path indexes it at run time.
__device__ __forceinline__ void repair_row(const GemmParams& p, int prod, int row, int col0, float* v, int n) {
  const int64_t aoff = (int64_t)prod * p.stride_a + (p.ta ? (int64_t)row : (int64_t)row * p.lda);
  const int64_t as = p.ta ? p.lda : 1, bs = p.tb ? 1 : p.ldb;
  if (!a_ok(p, aoff, 1) || !a_ok(p, aoff + (int64_t)(p.K - 1) * as, 1)) return;
  const float* a = p.A + aoff;
#pragma unroll 1
  for (int i = 0; i < n; ++i) {
    const int col = col0 + i;
    if (v[i] != v[i] && col < p.N) {
      const int64_t boff = (int64_t)prod * p.stride_b + (p.tb ? (int64_t)col * p.ldb : (int64_t)col);
      if (b_ok(p, boff, 1) && b_ok(p, boff + (int64_t)(p.K - 1) * bs, 1)) v[i] = fp32_dot(a, as, p.B + boff, bs, p.K);
    }
  }
}

// The check and repair of a folder thread's sums m (row `row`, columns col0 ..
// col0 + 2 * N2 - 1 of product `prod`); the caller has checked the row.
template <int N2>
__device__ __forceinline__ void repair_nans(const GemmParams& p, int prod, int row, int col0, float2 (&m)[N2]) {
  if (!any_nonfinite(m)) return;
  float v[2 * N2];
#pragma unroll
  for (int e = 0; e < N2; ++e) {
    v[2 * e] = m[e].x;
    v[2 * e + 1] = m[e].y;
  }
  repair_row(p, prod, row, col0, v, 2 * N2);
#pragma unroll
  for (int e = 0; e < N2; ++e) m[e] = make_float2(v[2 * e], v[2 * e + 1]);
}

// The same for the four sums of a fixup thread (columns col .. col + 3).
__device__ __forceinline__ void repair_nans4(const GemmParams& p, int prod, int row, int col, float4& s) {
  if (fabsf(s.x + s.y + s.z + s.w) <= 3.402823466e38f) return;
  float v[4] = {s.x, s.y, s.z, s.w};
  repair_row(p, prod, row, col, v, 4);
  s = make_float4(v[0], v[1], v[2], v[3]);
}

// ---- fixup of tiles that several CTAs (or clusters) shared under stream-K
// A fixup thread owns 4 consecutive columns of one row of C.  It reads C's old values before it
// waits for its GEMM grid (it is launched as that grid's programmatic dependent): the GEMM never
// writes C of a shared tile, and every kernel of the stream before that GEMM has completed once
// this grid runs, so the read is off the path that starts when the GEMM ends.
struct FixupOut {
  float* cp;     // C element of the first column (nullptr: nothing to write)
  int cnt;       // columns in range, 1..4
  float old[4];  // C's old values (read when beta != 0)
};

template <bool CVEC>
__device__ __forceinline__ FixupOut fixup_prefetch_c(const GemmParams& p, int prod, int row, int col) {
  FixupOut f;
  f.cp = nullptr;
  f.cnt = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) f.old[k] = 0.0f;
  const int64_t coff = (int64_t)prod * p.stride_c + (int64_t)row * p.ldc + col;
  const int cnt = min(4, p.N - col);
  if (!c_ok(p, coff, cnt)) return f;
  f.cp = p.C + coff;
  f.cnt = cnt;
  if (p.beta != 0.0f) {
    if (CVEC && cnt == 4) {
      const float4 o = *reinterpret_cast<const float4*>(f.cp);
      f.old[0] = o.x;
      f.old[1] = o.y;
      f.old[2] = o.z;
      f.old[3] = o.w;
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (k < cnt) f.old[k] = f.cp[k];
    }
  }
  return f;
}

// Sum of one float4 of n slots in sharer order (slot[i] * slot_elems + off in the workspace); the
// loads of four slots are issued before their adds.
__device__ __forceinline__ float4 fixup_sum(const GemmParams& p, const int* slot, int n, int64_t slot_elems,
                                            int64_t off) {
  float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int i0 = 0; i0 < n; i0 += 4) {
    float4 u[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      u[t] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      if (i0 + t < n) {
        const int64_t o = (int64_t)slot[i0 + t] * slot_elems + off;
        if (ws_ok(p, o, 4)) u[t] = *reinterpret_cast<const float4*>(p.ws + o);
      }
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      if (i0 + t >= n) break;
      if (i0 + t == 0) {
        v = u[t];
      } else {
        v.x += u[t].x;
        v.y += u[t].y;
        v.z += u[t].z;
        v.w += u[t].w;
      }
    }
  }
  return v;
}

// C = alpha * v + beta * old over the thread's in-range columns.
template <bool CVEC>
__device__ __forceinline__ void fixup_store(const GemmParams& p, const FixupOut& f, float4 v) {
  if (f.cp == nullptr) return;
  const float x[4] = {v.x, v.y, v.z, v.w};
  float o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = p.beta == 0.0f ? p.alpha * x[k] : fmaf(p.alpha, x[k], p.beta * f.old[k]);
  if (CVEC && f.cnt == 4) {
    *reinterpret_cast<float4*>(f.cp) = make_float4(o[0], o[1], o[2], o[3]);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < f.cnt) f.cp[k] = o[k];
  }
}

__device__ __forceinline__ void tile_coords(int bid, int tiles_m, int tiles_n, int& tm, int& tn) {
  constexpr int kGroupM = 8;
  const int span = kGroupM * tiles_n;
  const int group = bid / span;
  const int first = group * kGroupM;
  const int rows = min(tiles_m - first, kGroupM);
  const int local = bid - group * span;
  tm = first + local % rows;
  tn = local / rows;
}

// First stream-K iteration of CTA c: floor(c * I / G).
__device__ __forceinline__ int64_t sk_bound(const GemmParams& p, int c) {
  return (int64_t)c * p.sk_iters / p.sk_grid;
}

// The CTA whose stream-K range holds iteration i: the largest c with B(c) <= i.
__device__ __forceinline__ int sk_owner(const GemmParams& p, int64_t i) {
  return (int)(((i + 1) * p.sk_grid + p.sk_iters - 1) / p.sk_iters - 1);
}

// Partial-sum slot of CTA c for stream-K tile j (relative to the first stream-K tile).
__device__ __forceinline__ int sk_slot(const GemmParams& p, int c, int j, int kt) {
  return (int)(sk_bound(p, c) / kt) == j ? 2 * c : 2 * c + 1;
}

// A CTA's work: `dp` whole tiles (c, c+G, ... below sk_tile0), then stream-K
// iterations [b, e) covering relative stream-K tiles j0 .. j0 + nseg - dp - 1.
struct CtaWork {
  int dp, j0, nseg, units;
  int64_t b, e;
};

__device__ __forceinline__ CtaWork cta_work(const GemmParams& p, int c, int kt) {
  CtaWork w;
  w.dp = c < p.sk_tile0 ? (p.sk_tile0 - c + p.sk_grid - 1) / p.sk_grid : 0;
  w.b = p.sk_iters > 0 ? sk_bound(p, c) : 0;
  w.e = p.sk_iters > 0 ? sk_bound(p, c + 1) : 0;
  w.j0 = (int)(w.b / kt);
  w.nseg = w.dp + (w.e > w.b ? (int)((w.e - 1) / kt) - w.j0 + 1 : 0);
  w.units = w.dp * kt + (int)(w.e - w.b);
  return w;
}

// Segment s of a CTA's work: K tiles [kb, ke) of output tile `tile`; slot -1
// when the segment is the tile's whole K range (result goes to C).
struct Segment {
  int tile, kb, ke, slot;
};

__device__ __forceinline__ Segment cta_segment(const GemmParams& p, const CtaWork& w, int c, int s, int kt) {
  Segment g;
  if (s < w.dp) {
    g.tile = s * p.sk_grid + c;
    g.kb = 0;
    g.ke = kt;
    g.slot = -1;
  } else {
    const int j = w.j0 + (s - w.dp);
    const int64_t t0 = (int64_t)j * kt;
    g.tile = p.sk_tile0 + j;
    g.kb = (int)(max(w.b, t0) - t0);
    g.ke = (int)(min(w.e, t0 + kt) - t0);
    g.slot = (g.kb == 0 && g.ke == kt) ? -1 : sk_slot(p, c, j, kt);
  }
  return g;
}
// ---- CTA pairs (clusters of two CTAs on one TPC, tcgen05 cta_group::2)

constexpr uint16_t kPairMask = 0x3;  // both CTAs of the cluster

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t c;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(c));
  return c;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Pair TMEM allocation: one warp of each CTA of the pair executes these.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Arrives on the barrier at offset `bar` in both CTAs once every tcgen05.mma
// this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(kPairMask)
      : "memory");
}

// The shared::cluster address of this CTA's shared-memory offset `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// Arrive on the barrier at offset `bar` of CTA `rank` of this cluster.  The
// default (release, CTA scope) semantics suffice and cost no fence wait: what
// an arrival publishes is already ordered before it by the arriving warp --
// tensor-memory stores and loads by tcgen05.wait + tcgen05.fence, shared-memory
// operand writes by fence.proxy.async -- and the consumer is the tensor core,
// ordered after the issuer's wait by tcgen05.fence::after_thread_sync.  A
// cluster-scope release would also wait for the warp's outstanding global
// stores (the previous tile's C) on every arrival.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(map_to_rank(bar, rank)) : "memory");
}

// Product and origin (first row, first column) of tile `tile` of bm x bn tiles.
__device__ __forceinline__ void tile_origin_of(const GemmParams& p, int tile, int bm, int bn, int& prod, int& m0,
                                               int& n0) {
  const int tiles = p.tiles_m * p.tiles_n;
  prod = tile / tiles;
  int tm, tn;
  tile_coords(tile - prod * tiles, p.tiles_m, p.tiles_n, tm, tn);
  m0 = tm * bm;
  n0 = tn * bn;
}

}  // namespace tc
}  // namespace sgemm_impl
