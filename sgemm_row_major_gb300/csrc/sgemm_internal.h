// sgemm_internal.h -- host-side declarations shared by the translation units of libsgemm.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "sgemm.h"

namespace sgemm_impl {

// Everything a GEMM kernel needs besides its tensor maps.
//
// A call computes `batch` independent products; product b reads
// A + b*stride_a, B + b*stride_b and updates C + b*stride_c.  Grid: x =
// batch * tiles_m * tiles_n (CTA x works on product x / tiles, output tile
// x % tiles), y = K slices.
struct GemmParams {
  int M = 0, N = 0, K = 0;
  float alpha = 1.0f, beta = 0.0f;
  const float* A = nullptr;  // the generic kernel's operands; the tensor-core kernels' NaN repair reads them
  const float* B = nullptr;
  float* C = nullptr;        // final output (split == 1) ...
  float* ws = nullptr;       // ... or the partial-sum workspace [batch][split][M][ws_ld] (split > 1)
  int64_t lda = 0, ldb = 0, ldc = 0, ws_ld = 0;
  int64_t stride_a = 0, stride_b = 0, stride_c = 0;  // elements between consecutive products
  int ta = 0, tb = 0;            // 1: op(A) / op(B) is the transpose of the stored matrix
  int batch = 1;
  int za = 0, zb = 0;            // TMA kernels: 1 = the map's third coordinate is the product index
  int k_tiles_per_split = 0;     // K tiles (of the kernel's BK) per slice
  int tiles_m = 0, tiles_n = 0;  // output tiles of one product
  int c_vec = 0;                 // 1: C (every product) is 16-byte aligned and ldc % 4 == 0
  // Persistent schedule of the tensor-core kernel (kernel_tf32x3.cu): sk_grid
  // CTAs; CTA c takes whole tiles c, c + sk_grid, ... below sk_tile0, then an
  // even share of the sk_iters K tiles of output tiles sk_tile0 .. (all tiles
  // - 1); partial tiles go to slots of BM*BN floats in ws (2 per CTA).
  int sk_grid = 0, sk_tile0 = 0;
  int64_t sk_iters = 0;
  int repair = 1;                // tensor-core kernels: compute NaN sums again in FP32 (0: the TF32-input GEMM)
  uint64_t timeout_ns = 0;       // limit of every in-kernel wait
  unsigned* fault = nullptr;     // device fault word (bits of FaultBits), see fault_word()
  // Extents (elements from the base pointer) of the buffers, for the bounds checks of the debug
  // build (device_utils.cuh, in_range); the normal build does not read them.
  int64_t a_elems = 0, b_elems = 0, c_elems = 0, ws_elems = 0;
  unsigned long long* bounds = nullptr;  // debug build: first bounds violation (site << 48 | offset)
};

// Elements a row-major matrix of `rows` x `cols` (row stride ld) spans from its first element,
// over `batch` matrices `stride` elements apart (0 when empty).
inline int64_t matrix_extent(int64_t rows, int64_t cols, int64_t ld, int64_t batch, int64_t stride) {
  if (rows <= 0 || cols <= 0 || batch <= 0) return 0;
  return (batch - 1) * stride + (rows - 1) * ld + cols;
}

// Fills the extents of GemmParams from its own shape, op flags, leading dimensions, strides and
// batch, and the workspace size; `bounds` is the device's bounds word (bounds_word()).
inline void set_extents(GemmParams* p, int64_t ws_bytes, unsigned long long* bounds) {
  p->a_elems = p->ta ? matrix_extent(p->K, p->M, p->lda, p->batch, p->stride_a)
                     : matrix_extent(p->M, p->K, p->lda, p->batch, p->stride_a);
  p->b_elems = p->tb ? matrix_extent(p->N, p->K, p->ldb, p->batch, p->stride_b)
                     : matrix_extent(p->K, p->N, p->ldb, p->batch, p->stride_b);
  p->c_elems = matrix_extent(p->M, p->N, p->ldc, p->batch, p->stride_c);
  p->ws_elems = ws_bytes / 4;
  p->bounds = bounds;
}

// Tensor maps of the operands of a TMA-fed kernel: 3-D {contiguous, rows,
// product} float32 maps over the stored A and B, boxes of the kernel's tile
// (A: bm x bk of op(A), B: bk x bn of op(B)), 128-byte swizzle where a box
// row is 32 floats of K (K-major tiles), none otherwise.  A map whose stride
// is 0 or whose call has one product gets a product extent of 1 and its z flag
// (GemmParams::za / zb) is 0.  Returns the encode error.
cudaError_t encode_operand_maps(bool ta, bool tb, int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
                                int64_t stride_a, const float* B, int64_t ldb, int64_t stride_b, int batch,
                                int bm, int bn, int bk, CUtensorMap* mapA, CUtensorMap* mapB, int* za, int* zb);

// Copies the tensor-core kernel's schedule from a plan (no-op for other
// variants); the pair kernel's scheduling unit is the cluster of 2 CTAs.
inline void set_schedule(const sgemm_plan_t& plan, GemmParams* p) {
  const bool pairs = plan.variant == SGEMM_VARIANT_TC_PAIR || plan.variant == SGEMM_VARIANT_TC_PRESPLIT ||
                     plan.variant == SGEMM_VARIANT_TC_TF32 || plan.variant == SGEMM_VARIANT_TC_BF16;
  if (plan.variant != SGEMM_VARIANT_TC_TF32X3 && plan.variant != SGEMM_VARIANT_TC_GROUPED &&
      plan.variant != SGEMM_VARIANT_TC_SKINNY && !pairs)
    return;
  p->sk_grid = (int)(pairs ? plan.grid_x / 2 : plan.grid_x);
  p->sk_iters = plan.sk_iters;
  p->sk_tile0 = (int)plan.dp_tiles;
}

// Split-operand arrays of the TC_PRESPLIT variant: op(A) and op(B) as rows of
// K contiguous floats (row stride split_ldk(K)), hi and lo parts, one set per
// product whose operand differs (a stride of 0 shares one).
inline int64_t split_ldk(int64_t K) { return (K + 3) / 4 * 4; }
inline int64_t round256(int64_t bytes) { return (bytes + 255) / 256 * 256; }
struct SplitLayout {
  int64_t slots = 0;             // stream-K partial-sum slots (bytes, first in the workspace)
  int64_t a_products = 1, b_products = 1;
  int64_t a_bytes = 0, b_bytes = 0;  // one part (hi or lo) of op(A) / op(B), all products
  int parts = 2;                 // hi and lo (3xTF32), or hi only (the TF32-input GEMM)
  int64_t total() const { return round256(slots) + parts * (round256(a_bytes) + round256(b_bytes)); }
};
inline SplitLayout split_layout(int64_t M, int64_t N, int64_t K, int64_t batch, int64_t stride_a, int64_t stride_b,
                                int64_t slot_bytes, int parts = 2) {
  SplitLayout l;
  l.slots = slot_bytes;
  l.parts = parts;
  l.a_products = (batch > 1 && stride_a != 0) ? batch : 1;
  l.b_products = (batch > 1 && stride_b != 0) ? batch : 1;
  l.a_bytes = l.a_products * M * split_ldk(K) * 4;
  l.b_bytes = l.b_products * N * split_ldk(K) * 4;
  return l;
}

// TMA box extents one CTA of a plan loads per K tile: rows of op(A) and
// columns of op(B) (a CTA of a pair covers half of the tile's rows and loads
// half of its B columns).
inline void operand_boxes(const sgemm_plan_t& plan, int* bm, int* bn) {
  const bool pair = plan.variant == SGEMM_VARIANT_TC_PAIR;
  *bm = pair ? plan.tile_m / 2 : plan.tile_m;
  *bn = pair ? plan.tile_n / 2 : plan.tile_n;
}

// Shapes of the TMA-fed SIMT kernel.
enum class TmaTile { k128x128, k64x256 };

struct GenericTileShape {
  int bm, bn, bk, threads;
};
GenericTileShape generic_tile_shape();

// Launchers: enqueue one kernel on `stream`, return the launch error.
// TMA-fed kernel, one entry per operand layout (kernel_tma_{nn,nt,tn,tt}.cu).
#define SGEMM_DECLARE_TMA_OP(op)                                                                   \
  cudaError_t launch_tma_op_##op(TmaTile tile, const CUtensorMap& mapA, const CUtensorMap& mapB, \
                                 const GemmParams& p, int split, cudaStream_t stream);            \
  cudaError_t prepare_tma_op_##op();
SGEMM_DECLARE_TMA_OP(nn)
SGEMM_DECLARE_TMA_OP(nt)
SGEMM_DECLARE_TMA_OP(tn)
SGEMM_DECLARE_TMA_OP(tt)
#undef SGEMM_DECLARE_TMA_OP
// 3xTF32 tensor-core kernel (kernel_tf32x3.cu), 128x128x32 tiles, any op,
// persistent data-parallel + stream-K schedule (GemmParams::sk_*), then the
// fixup kernel over the sk_tiles stream-K tiles when any of them is shared.
// `group` G > 1 (2 or 4): products with M, N <= 128/G, G to a tile
// block-diagonally (tile t = products G*t .. G*t+G-1; tensor maps with boxes
// 128/G wide; whole tiles only, no stream-K).
cudaError_t prepare_tf32x3();
cudaError_t launch_tf32x3(bool transA, bool transB, int group, const CUtensorMap& mapA, const CUtensorMap& mapB,
                          const GemmParams& p, cudaStream_t stream);
cudaError_t launch_streamk_fixup(const GemmParams& p, int sk_tiles, cudaStream_t stream);
// 3xTF32 on CTA pairs (kernel_tc_pair.cu): 256x128x32 tiles, clusters of 2,
// p.sk_grid clusters, the schedule of the one-CTA kernel over pair tiles;
// then the fixup over the sk_tiles stream-K pair tiles when any is shared.
cudaError_t prepare_tc_pair();
cudaError_t tc_pair_max_clusters(int* clusters);  // co-resident clusters of the pair kernel on this device
cudaError_t launch_tc_pair(bool transA, bool transB, const CUtensorMap& mapA, const CUtensorMap& mapB,
                           const GemmParams& p, cudaStream_t stream);
cudaError_t launch_pair_fixup(const GemmParams& p, int sk_tiles, cudaStream_t stream);
// 3xTF32 on split operands (kernel_presplit.cu): the split pass (per operand:
// rows x K of op(X), from a stored layout whose rows run along K or not, any
// alignment; lo == nullptr writes hi only), then
// the CTA-pair GEMM on 256x256x32 tiles with four maps over the split arrays,
// then the fixup over the sk_tiles stream-K pair tiles when any is shared.
cudaError_t prepare_presplit();
// Where a split pass stands in its call's launch chain: the first of the call (lets the next
// launch start early), a dependent of the pass before it (a programmatic dependent launch that
// completes only after that pass), or alone.
enum class SplitOrder { kAlone, kFirst, kDependent };
cudaError_t launch_split_operand(const float* src, int64_t ld, int64_t stride, bool k_contig, int rows, int K,
                                 int products, float* hi, float* lo, int64_t ldk, int sm_count, cudaStream_t stream,
                                 unsigned* fault = nullptr, unsigned long long* bounds = nullptr,
                                 int64_t src_elems = 0, SplitOrder order = SplitOrder::kAlone);
cudaError_t launch_presplit_gemm(const CUtensorMap& mapAh, const CUtensorMap& mapAl, const CUtensorMap& mapBh,
                                 const CUtensorMap& mapBl, const GemmParams& p, cudaStream_t stream);
cudaError_t launch_presplit_fixup(const GemmParams& p, int sk_tiles, cudaStream_t stream, int k_tile = 32);
// The TF32-input GEMM: the same CTA-pair kernel with one part per operand (maps over the rounded
// copies, written by launch_split_operand with lo == nullptr) and one tensor-core product per k;
// its stream-K tiles go through launch_presplit_fixup (p.repair = 0).
cudaError_t launch_tf32_gemm(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p,
                             cudaStream_t stream);
// The BF16-input GEMM: the same CTA-pair kernel over maps of BF16 arrays (64 K per tile, kind::f16
// MMAs), written by launch_round_bf16 (out: rows of ldk BF16 values, ldk a multiple of 8); its
// stream-K tiles go through launch_presplit_fixup with k_tile = 64.
cudaError_t launch_bf16_gemm(const CUtensorMap& mapA, const CUtensorMap& mapB, const GemmParams& p,
                             cudaStream_t stream);
cudaError_t launch_round_bf16(const float* src, int64_t ld, bool k_contig, int rows, int K, void* out, int64_t ldk,
                              int sm_count, cudaStream_t stream, unsigned* fault, unsigned long long* bounds,
                              int64_t src_elems, SplitOrder order);
// Map over a BF16 array of `rows` rows of K values (row stride ldk elements): box {64, 128, 1}, 128-byte swizzle.
cudaError_t encode_bf16_map(const void* base, int64_t K, int64_t rows, int64_t ldk, CUtensorMap* map);
// sgemm_plan() for a caller that cannot provide the split arrays of TC_PRESPLIT
// (sgemm_noalloc): that variant, chosen or forced by override, is planned as TC_PAIR.
// pair_clusters as in sgemm_plan_for_device().
int plan_without_split_arrays(char transA, char transB, int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                              int64_t lda, const float* B, int64_t ldb, float beta, const float* C, int64_t ldc,
                              int sm_count, int pair_clusters, sgemm_plan_t* plan);
// Map over a split array: {K, rows, products} float32, row stride ldk, box {32, box_rows, 1}, 128-byte
// swizzle.
cudaError_t encode_split_map(const float* base, int64_t K, int64_t rows, int64_t ldk, int64_t products,
                             CUtensorMap* map, int box_rows = 128);
// Map over one row-major matrix of `outer` rows x `inner` contiguous floats (row stride ld), box
// {box_inner, box_outer, 1}; 128-byte swizzle when box rows are 32 floats.
cudaError_t encode_matrix_map(const float* base, int64_t inner, int64_t outer, int64_t ld, int box_inner,
                              int box_outer, CUtensorMap* map);

// The short-side kernel (kernel_skinny.cu).  long_contig: the long operand is stored long side
// contiguous; trans_c: C is the transpose of the kernel's (long x short) result.  mapL: the long
// operand as stored (box 128 x 32 floats); mapSh / mapSl: the short operand's hi / lo split arrays
// (box 32 x 64, swizzled).
cudaError_t prepare_skinny();
cudaError_t launch_skinny_gemm(bool long_contig, bool trans_c, const CUtensorMap& mapL, const CUtensorMap& mapSh,
                               const CUtensorMap& mapSl, const GemmParams& p, cudaStream_t stream);
cudaError_t launch_skinny_fixup(bool trans_c, const GemmParams& p, int sk_tiles, cudaStream_t stream);
cudaError_t launch_generic_gemm(bool transA, bool transB, const GemmParams& p, int split,
                                cudaStream_t stream);
cudaError_t launch_splitk_reduce(const GemmParams& p, int split, cudaStream_t stream);
cudaError_t launch_scale(const GemmParams& p, cudaStream_t stream);
cudaError_t launch_wait_selftest(uint64_t timeout_ns, unsigned* fault, cudaStream_t stream);
cudaError_t launch_clock_snapshot(unsigned long long* out, int slots, int sm_count, cudaStream_t stream);

// Keeps e as this thread's last CUDA error (sgemm_last_cuda_error) and returns SGEMM_ERR_CUDA.
int record_cuda_failure(cudaError_t e);
int& t_last_cuda_error_slot();
// The limit of every in-kernel wait: SGEMM_WAIT_TIMEOUT_MS (default 2000 ms), read once.
uint64_t wait_timeout_ns();
// Co-resident CTA-pair clusters on the current device, or 0 when the pair kernel cannot be
// co-scheduled there (or the query fails): the planner then leaves out the CTA-pair kernels.
int pair_clusters_or_none();
// Returns the memory pool of sgemm_host() on device `dev` to the driver down to keep_bytes.
cudaError_t trim_host_pool(int dev, size_t keep_bytes);

// Device address of the current device's fault word (looked up once per device).
cudaError_t fault_word(unsigned** ptr);
// Device address of the current device's bounds word (debug build: first bounds violation).
cudaError_t bounds_word(unsigned long long** ptr);
// Reads and clears the bounds word (synchronous).
cudaError_t take_bounds(unsigned long long* word);
// Launches the bounds self-test: one check of an index past its limit (never dereferenced).
cudaError_t launch_bounds_selftest(unsigned* fault, unsigned long long* word, cudaStream_t stream);
// Reads and clears the current device's fault word (synchronous).
cudaError_t take_faults(unsigned* bits);

}  // namespace sgemm_impl
