/*
 * sgemm.h -- C ABI of libsgemm, a single-precision GEMM for NVIDIA GB300 (sm_103a).
 *
 * Operation (BLAS SGEMM; itan.pw "CUDA NVIDIA 4090 高性能計算", 概要, with the
 * row-major element definition of klklkl10086.github.io "Sgemm单精度矩阵乘法",
 * 问题定义):
 *
 *     C = alpha * op(A) * op(B) + beta * C,     op(X) = X or X^T,
 *
 * on ROW-MAJOR float32 matrices: op(A) is M x K, op(B) is K x N, C is M x N.
 *
 * Layout (CBLAS row-major conventions; ld = row stride of the STORED matrix,
 * in elements):
 *   transA 'N': A stored M x K,  op(A)_ik = A[i*lda + k],  lda >= max(1, K)
 *   transA 'T': A stored K x M,  op(A)_ik = A[k*lda + i],  lda >= max(1, M)
 *   transB 'N': B stored K x N,  op(B)_kj = B[k*ldb + j],  ldb >= max(1, N)
 *   transB 'T': B stored N x K,  op(B)_kj = B[j*ldb + k],  ldb >= max(1, K)
 *   C_ij at C[i*ldc + j], ldc >= max(1, N)
 * 'n'/'t' are accepted, and 'C'/'c' mean 'T' (the data are real).
 *
 * Ownership: A, B, C are caller-owned DEVICE pointers on the current CUDA
 * device; the library never frees or retains them.  The library owns only
 * internal state: a per-device stream-ordered memory pool for its workspace
 * (split-K / stream-K partial sums and, for SGEMM_VARIANT_TC_PRESPLIT, the
 * split copies of op(A) and op(B): 4 x 4 bytes per element of each, at most
 * 4 GiB; allocated and freed in stream order on the caller's stream),
 * per-device kernel attributes, and a per-device fault word.  The pool keeps
 * the memory a call frees for later calls (so steady-state calls allocate
 * nothing): the largest workspace any call needed stays reserved for the
 * library until the process exits or sgemm_release_workspace() returns it.
 *
 * Semantics of special values (BLAS conventions; the pages do not say):
 *   - M == 0 or N == 0: nothing is done, SGEMM_OK.
 *   - beta == 0: C is not read (NaN/Inf in C do not propagate).
 *   - alpha == 0 or K == 0: A and B are not read; C = beta * C.
 *   - Unaligned pointers or leading dimensions are NOT errors; they take a
 *     slower path.  C overlapping A or B is undefined.
 *
 * Arithmetic: the default kernel (16-byte aligned A and B, lda % 4 == 0,
 * ldb % 4 == 0) runs on the tensor cores with each float split into two
 * TF32 parts (3 products per term, partial sums folded in FP32 every 32 k);
 * results meet |C - C_exact| <= (K+2) 2^-24 (|alpha| sum|a b| + |beta c|) and
 * are deterministic, but are not the IEEE FP32 FMA sums of a SIMT loop.
 * Inputs the split cannot carry -- +-Inf, and finite values of magnitude
 * >= (2 - 2^-11) 2^127, whose TF32 part would round to Inf -- make the
 * tensor-core sums they enter NaN; every NaN sum is computed again with FP32
 * FMAs (k ascending), so the results are those of IEEE FP32 arithmetic:
 * +-Inf where the definition gives +-Inf, NaN for Inf * 0, Inf - Inf and NaN
 * inputs, and finite values within the bound above.  As in any FP32
 * accumulation, products or partial sums beyond FLT_MAX overflow to +-Inf.
 * Scaling A and B by powers of two scales C exactly, as in FP32 arithmetic,
 * down to products near the FP32 subnormal range (products and sums in that
 * range are kept; measured exact).  Tiny INPUTS are the exception: TF32's
 * smallest step is 2^-136, so an input of magnitude below 2^-115 reaches the
 * tensor cores only to within 2^-137 (its remainder below TF32's range is
 * dropped), which adds up to 2^-137 * sum_k(|b_k| over the k whose a_k is
 * that small, and |a_k| over the k whose b_k is) to an element's error; that
 * exceeds the bound above only when the whole dot product is of that order.
 * The FP32 FFMA kernels
 * (IEEE operations throughout) are selected with
 * sgemm_set_variant_override(SGEMM_VARIANT_TMA_128x128 or
 * SGEMM_VARIANT_TMA_64x256, 0).  Operands TMA cannot load (a base not 16-byte
 * aligned, lda or ldb not a multiple of 4) take the split-operand tensor-core
 * kernel from 2 * 640^3 FLOP on (its split pass rewrites them aligned), the
 * FP32 FFMA generic kernel below that.
 *
 * Errors: invalid arguments return -(argument index) (1 = transA ... 14 =
 * stream) before anything is launched, and C is untouched.  CUDA launch or
 * allocation failures return SGEMM_ERR_CUDA / SGEMM_ERR_NOMEM (the CUDA
 * error code is kept per thread, see sgemm_last_cuda_error).  Execution is
 * asynchronous: sgemm() returns once the work is enqueued on `stream`;
 * kernel faults appear at the caller's next synchronisation.  Every wait
 * inside a kernel is bounded; a wait that gives up sets the device fault
 * word, which sgemm_sync_status() reports as SGEMM_ERR_TIMEOUT.
 */
#ifndef SGEMM_H
#define SGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *`; NULL = legacy default stream */

enum sgemm_status {
    SGEMM_OK = 0,
    SGEMM_ERR_CUDA = 1,        /* a CUDA runtime call failed (see sgemm_last_cuda_error) */
    SGEMM_ERR_TIMEOUT = 2,     /* a bounded in-kernel wait gave up (reported by sgemm_sync_status) */
    SGEMM_ERR_NOMEM = 3,       /* the call's workspace (partial sums, split operands) could not be allocated */
    SGEMM_ERR_UNSUPPORTED = 4, /* a dimension or leading dimension >= 2^31, or no usable device */
    SGEMM_ERR_SCRATCH_LIMIT = 5,/* sgemm_noalloc: the problem needs more scratch than its static array */
    SGEMM_ERR_BOUNDS = 6       /* debug build: a kernel index fell outside its buffer (reported by
                                  sgemm_sync_status; the access was skipped) */
    /* negative values: -(index of the invalid argument), BLAS xerbla style */
};

/* Kernel variants, as reported by sgemm_plan() and accepted by sgemm_set_variant_override(). */
enum sgemm_variant {
    SGEMM_VARIANT_AUTO = 0,       /* override only: let the planner choose */
    SGEMM_VARIANT_NONE = 1,       /* M == 0 or N == 0: no launch */
    SGEMM_VARIANT_SCALE = 2,      /* alpha == 0 or K == 0: C = beta * C */
    SGEMM_VARIANT_GENERIC = 3,    /* any alignment: 64x64 tiles, predicated loads */
    SGEMM_VARIANT_TMA_128x128 = 4,/* TMA-fed SIMT FFMA, 128x128x32 tiles, 4-stage mbarrier ring */
    SGEMM_VARIANT_TMA_64x256 = 5, /* same kernel, 64x256 tiles for short M */
    SGEMM_VARIANT_TC_TF32X3 = 6,  /* tcgen05 tensor cores, 3xTF32 split, 128x128x32 tiles */
    SGEMM_VARIANT_SMALL = 7,      /* M, N <= 64 in a large batch: one CTA per product, FP32 FFMA */
    SGEMM_VARIANT_TC_GROUPED = 8, /* M, N <= 64 in a batch: 3xTF32 tensor cores, 2 (M, N <= 32: 4) products
                                     per 128x128 tile, block-diagonally; tile_m = tile_n = 128 / group */
    SGEMM_VARIANT_TC_PAIR = 9,    /* 3xTF32 tensor cores on CTA pairs (clusters of 2 on one TPC): 256x128x32
                                     tiles, each CTA 128 rows and half of the tile's B columns */
    SGEMM_VARIANT_TC_PRESPLIT = 10,/* 3xTF32 with A and B split once per call into TF32 hi / FP32 lo arrays
                                      (in the workspace), then CTA pairs on 256x256x32 tiles reading both
                                      parts from shared memory */
    SGEMM_VARIANT_TC_TF32 = 11,   /* sgemm_tf32() only: A and B rounded to TF32 once per call (in the
                                      workspace), one tensor-core product per k on CTA pairs, 256x256x32
                                      tiles */
    SGEMM_VARIANT_TC_SKINNY = 12, /* one short side (M <= 64 or N <= 64), one product: the short operand
                                     split once per call into hi / lo arrays (in the workspace), the long
                                     one split in the kernel; 3xTF32 on tiles of 128 along the long side x
                                     64 along the short one (tile_m = 128 and tile_n = 64 name those
                                     sides, whichever of M and N is short) */
    SGEMM_VARIANT_TC_BF16 = 13    /* sgemm_bf16() only: A and B rounded to BF16 once per call (in the
                                     workspace), one kind::f16 tensor-core product per 16 k on CTA pairs,
                                     256x256x64 tiles */
};

/*
 * C = alpha * op(A) * op(B) + beta * C on row-major float32 matrices (see above).
 * Returns SGEMM_OK once the work is enqueued on `stream`, or an error status.
 */
int sgemm(char transA, char transB, int64_t M, int64_t N, int64_t K,
          float alpha, const float *A, int64_t lda,
          const float *B, int64_t ldb,
          float beta, float *C, int64_t ldc,
          struct CUstream_st *stream);

/*
 * Caller-supplied workspace: the same operation as sgemm() with its workspace
 * -- the partial sums of a split K (split-K slices, stream-K tiles shared by
 * several CTAs) and, for SGEMM_VARIANT_TC_PRESPLIT, the TF32 hi / FP32 lo
 * copies of op(A) and op(B) -- in memory the caller owns, so a call
 * allocates nothing, has no size limit and captures into a CUDA graph as
 * kernels only.
 *
 * sgemm_workspace_size() stores in *bytes the workspace sgemm_ex() needs for
 * these arguments on the current device (0: none; equal to the
 * workspace_bytes of sgemm_plan() with sm_count <= 0).  Arguments 1-13 are
 * checked as in sgemm() (C is only inspected); -14: bytes is NULL.
 *
 * sgemm_ex(): arguments 1-13 and 16 (stream) as in sgemm(); `workspace` is a
 * device pointer, 16-byte aligned, to at least that many bytes, which the
 * call uses in stream order on `stream` (the caller must not touch it, nor
 * share it with another call that may run at the same time, until the call's
 * work on the stream is done).  -14: workspace NULL although needed, or not
 * 16-byte aligned; -15: workspace_bytes smaller than needed.  Nothing is
 * launched on an argument error.
 */
int sgemm_workspace_size(char transA, char transB, int64_t M, int64_t N, int64_t K,
                         float alpha, const float *A, int64_t lda,
                         const float *B, int64_t ldb,
                         float beta, const float *C, int64_t ldc, size_t *bytes);
int sgemm_ex(char transA, char transB, int64_t M, int64_t N, int64_t K,
             float alpha, const float *A, int64_t lda,
             const float *B, int64_t ldb,
             float beta, float *C, int64_t ldc,
             void *workspace, size_t workspace_bytes,
             struct CUstream_st *stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char *sgemm_status_string(int status);

/* cudaError_t of the last CUDA failure seen by a libsgemm call on this thread (0 = none). */
int sgemm_last_cuda_error(void);

/*
 * Synchronises `stream`, then reads and clears the current device's fault
 * word.  Returns SGEMM_ERR_TIMEOUT if a kernel's bounded wait gave up since
 * the last call, SGEMM_ERR_CUDA if the synchronisation failed, else SGEMM_OK.
 */
int sgemm_sync_status(struct CUstream_st *stream);

/* What sgemm() would launch for these arguments. */
typedef struct sgemm_plan_t {
    int variant;             /* enum sgemm_variant */
    int tile_m, tile_n, tile_k;
    int stages;              /* shared-memory pipeline depth (0 when no GEMM kernel) */
    int threads;             /* threads per CTA of the GEMM kernel */
    int split_k;             /* number of K slices (1 = no split) */
    int kernel_launches;     /* kernels one sgemm() call launches */
    int64_t grid_x, grid_y;  /* CTAs of the GEMM kernel: tiles x K slices */
    int64_t workspace_bytes; /* split-K / stream-K partial sums (+ TC_PRESPLIT: split operands), from the pool */
    int64_t smem_bytes;      /* dynamic shared memory per CTA */
    /* Tensor-core kernel only (persistent CTAs, grid_x of them): the first
     * dp_tiles output tiles are taken whole, round robin (CTA c: tiles c,
     * c + grid_x, ...); the sk_iters K tiles of the last sk_tiles output tiles
     * are then shared evenly by all CTAs (stream-K); split_k is the most CTAs
     * that share one output tile.  SGEMM_VARIANT_TC_PAIR: the same schedule
     * over 256 x 128 tiles with clusters of two CTAs as the unit (grid_x / 2
     * clusters; split_k counts clusters); SGEMM_VARIANT_TC_PRESPLIT: likewise
     * over 256 x 256 tiles, and kernel_launches counts the split passes of A
     * and B.  SGEMM_VARIANT_TC_GROUPED: every tile is
     * whole and holds 128 / tile_m products (tile_m = tile_n = 64: two, 32:
     * four), so dp_tiles = ceil(batch_count / (128 / tile_m)).  For
     * SGEMM_VARIANT_SMALL grid_x is the persistent grid (products dealt round
     * robin) and tile_k its K chunk. */
    int64_t dp_tiles;
    int64_t sk_tiles;
    int64_t sk_iters;
} sgemm_plan_t;

/*
 * Fills *plan with the launch sgemm() would make for these arguments on a
 * device with `sm_count` SMs (sm_count <= 0: query the current device).
 * Pure host logic when sm_count > 0 (the device is then assumed to co-schedule
 * sm_count / 2 CTA-pair clusters, one per TPC); validates arguments like
 * sgemm().  Pointers are only inspected for alignment and NULL.
 */
int sgemm_plan(char transA, char transB, int64_t M, int64_t N, int64_t K,
               float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb,
               float beta, const float *C, int64_t ldc,
               int sm_count, sgemm_plan_t *plan);

/*
 * The plan for a device described by its SM count (> 0, else -14) and the
 * number of clusters of two CTAs of the CTA-pair kernels it can hold at once
 * (>= 0, else -15; the device's own figure comes from an occupancy query,
 * which gives less than sm_count / 2 under an SM limit such as MPS, and 0 when
 * such a cluster cannot be scheduled at all: the CTA-pair and split-operand
 * kernels are then never chosen, and a forced one falls back to one CTA per
 * tile).  plan == NULL: -16.  Pure host logic.
 */
int sgemm_plan_for_device(char transA, char transB, int64_t M, int64_t N, int64_t K,
                          float alpha, const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          float beta, const float *C, int64_t ldc,
                          int sm_count, int pair_clusters, sgemm_plan_t *plan);

/*
 * Returns to the driver the pooled workspace memory of the current device
 * (sgemm(), sgemm_strided_batched() and sgemm_host() buffers) beyond
 * keep_bytes.  Memory of calls still running is not released; call it when
 * the streams that ran libsgemm work are idle.  SGEMM_ERR_CUDA on failure.
 */
int sgemm_release_workspace(size_t keep_bytes);

/*
 * Process-wide override of the planner, for tests and benchmarks:
 * variant = SGEMM_VARIANT_AUTO restores automatic choice; split_k = 0 keeps
 * the planner's split, >= 1 forces it (clamped to the number of K tiles).
 * A forced TMA variant whose alignment rules the operands break falls back
 * to GENERIC.  Returns SGEMM_OK or -1 for an unknown variant.
 */
int sgemm_set_variant_override(int variant, int split_k);

/*
 * Self-test of the bounded-wait machinery: launches one CTA that waits on a
 * shared-memory mbarrier nothing will ever complete, with a limit of
 * `timeout_us` microseconds (1..10,000,000), synchronises `stream` and reports
 * what the kernel recorded.  Returns SGEMM_ERR_TIMEOUT when the wait gave up
 * and the fault word was set as designed (the expected outcome), SGEMM_OK if
 * it did not, or SGEMM_ERR_CUDA.  Clears the fault word afterwards.
 */
int sgemm_selftest_wait_timeout(unsigned timeout_us, struct CUstream_st *stream);

/*
 * sgemm_strided_batched -- batch_count independent products in one call
 * (the FC-layer use of SGEMM: itan.pw "CUDA NVIDIA 4090 高性能計算", 概要,
 * names fully connected and convolution layers as what SGEMM serves):
 *
 *     C_b = alpha * op(A_b) * op(B_b) + beta * C_b,   b = 0 .. batch_count-1,
 *     A_b = A + b*strideA,  B_b = B + b*strideB,  C_b = C + b*strideC,
 *
 * strides in ELEMENTS, every product with the shapes, leading dimensions and
 * layout rules of sgemm().  The first 13 arguments are sgemm()'s, so a
 * negative status names the same argument; then 14 strideA, 15 strideB,
 * 16 strideC, 17 batch_count, 18 stream.
 *   - strideA or strideB may be 0 (one matrix shared by every product) or
 *     smaller than a matrix (overlapping operands are only read).
 *   - With batch_count > 1 the C matrices must not overlap:
 *     strideC >= (M-1)*ldc + N, else -16.  Negative strides: -14/-15/-16.
 *   - batch_count < 0: -17; batch_count == 0 (or M == 0 or N == 0): nothing
 *     is done, SGEMM_OK.
 *   - The arithmetic, special values and error behaviour of each product are
 *     those of sgemm(); one call launches one GEMM kernel for all products
 *     (plus the split-K reduction when the products are too few to fill the
 *     GPU).  The fast paths need strides that are multiples of 4 floats (and
 *     non-overlapping operands or a 0 stride); other strides take the
 *     any-alignment kernel.
 *   - Products with M, N <= 64 (a batch of at least one per SM) run two to a
 *     tensor-core tile, M, N <= 32 four to a tile (SGEMM_VARIANT_TC_GROUPED):
 *     same arithmetic and bounds as the tensor-core path of sgemm().
 */
int sgemm_strided_batched(char transA, char transB, int64_t M, int64_t N, int64_t K,
                          float alpha, const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          float beta, float *C, int64_t ldc,
                          int64_t strideA, int64_t strideB, int64_t strideC,
                          int64_t batch_count, struct CUstream_st *stream);

/* What sgemm_strided_batched() would launch (grid_x counts the tiles of all
 * products, workspace_bytes the partial sums of all products); argument
 * checks as there, sm_count as in sgemm_plan(); plan == NULL gives -19. */
int sgemm_plan_strided_batched(char transA, char transB, int64_t M, int64_t N, int64_t K,
                               float alpha, const float *A, int64_t lda,
                               const float *B, int64_t ldb,
                               float beta, const float *C, int64_t ldc,
                               int64_t strideA, int64_t strideB, int64_t strideC,
                               int64_t batch_count, int sm_count, sgemm_plan_t *plan);

/*
 * Debug build (libsgemm_debug.so, the same sources compiled with
 * -DSGEMM_DEBUG_BOUNDS; the pages suggest checking every access, youngju.dev
 * "CUDA architecture visualized", よくある落とし穴): every global-memory index
 * of the kernels, and the shared- and tensor-memory offsets of the splitters,
 * is checked against its buffer's extent before the access.  A violation skips
 * the access (nothing traps, nothing is touched out of bounds), sets a bit that
 * sgemm_sync_status() reports as SGEMM_ERR_BOUNDS, and keeps the first
 * violation for sgemm_bounds_report(): *site (1 C, 2 workspace, 3 A or a split
 * source, 4 B, 5 split arrays, 6 shared memory, 7 tensor memory, 8 self-test)
 * and *offset (elements, bytes or columns from the buffer's start); both 0
 * when there was none; reading clears it (-1 / -2: site / offset NULL).
 * sgemm_debug_bounds_enabled() is 1 in the debug library, 0 in libsgemm.so.
 * sgemm_selftest_bounds() runs one check of an index one past its limit (never
 * dereferenced): in the debug library the next sgemm_sync_status() returns
 * SGEMM_ERR_BOUNDS and the report gives site 8, offset 64; in libsgemm.so
 * nothing is recorded.
 */
int sgemm_bounds_report(unsigned *site, long long *offset);
int sgemm_debug_bounds_enabled(void);
int sgemm_selftest_bounds(struct CUstream_st *stream);

/*
 * Measurement aid: enqueues on `stream` a tiny kernel whose CTAs (four per
 * SM) write, for the SM each runs on, the SM's cycle counter and the global
 * nanosecond timer to out[2 * smid] and out[2 * smid + 1].  `out` is a device
 * buffer of 2 * slots unsigned 64-bit words (slots >= the SM count covers
 * every SM; SMs with smid >= slots are skipped, entries of SMs no CTA ran on
 * are left as they were).  Two snapshots around a stretch of work give each
 * SM's average clock over it (cycles / ns); nothing is changed on the GPU.
 * -1: out is NULL; -2: slots < 1.
 */
int sgemm_clock_snapshot(unsigned long long *out, int slots, struct CUstream_st *stream);

/*
 * sgemm_tf32 -- reduced-precision inputs, FP32 accumulation: the tensor-core
 * format for FP32 data that youngju.dev "CUDA architecture visualized"
 * (テンソルコア) names.  Computes
 *     C = alpha * op(tf32(A)) * op(tf32(B)) + beta * C
 * where tf32(x) rounds x to 10 explicit significand bits, to nearest with
 * ties away from zero (a finite x whose rounding carries past FLT_MAX gives
 * +-Inf; +-Inf and NaN stay), and the products (exact in FP32) are summed in
 * FP32.  Contract: |C - C_t| <= (K+2) 2^-24 (|alpha| sum|a_t b_t| + |beta c|)
 * per element against that expression evaluated exactly on the rounded inputs
 * (C_t), so the result differs from sgemm()'s by up to about 2^-11 relative
 * per product -- this entry point trades FP32 accuracy for speed; sgemm()'s
 * contract is unchanged.  Arguments, conventions, ownership, errors and
 * asynchrony as sgemm(); any alignment.  Each operand is rounded once per
 * call into a pooled workspace (4 bytes per element of op(A) and op(B), rows
 * padded to a multiple of 4 floats), then CTA pairs compute 256x256 tiles with
 * one tensor-core product per k (SGEMM_VARIANT_TC_TF32).  Needs a device
 * where clusters of two CTAs can be co-scheduled, and K <= 2097120:
 * SGEMM_ERR_UNSUPPORTED otherwise.
 */
int sgemm_tf32(char transA, char transB, int64_t M, int64_t N, int64_t K,
               float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb,
               float beta, float *C, int64_t ldc,
               struct CUstream_st *stream);

/* What sgemm_tf32() would launch (sm_count as in sgemm_plan(); plan == NULL: -15). */
int sgemm_tf32_plan(char transA, char transB, int64_t M, int64_t N, int64_t K,
                    float alpha, const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    float beta, const float *C, int64_t ldc,
                    int sm_count, sgemm_plan_t *plan);

/*
 * sgemm_bf16 -- as sgemm_tf32, with BF16 inputs: the other tensor-core input
 * format youngju.dev "CUDA architecture visualized" (テンソルコア) names for
 * FP32-range data.  Computes
 *     C = alpha * op(bf16(A)) * op(bf16(B)) + beta * C
 * where bf16(x) rounds x to 7 explicit significand bits, to nearest with ties
 * to even (a finite x whose rounding carries past (2 - 2^-7) 2^127 gives
 * +-Inf; +-Inf and NaN stay), and the products (exact in FP32) are summed in
 * FP32.  Contract: |C - C_b| <= (K+2) 2^-24 (|alpha| sum|a_b b_b| + |beta c|)
 * per element against that expression evaluated exactly on the rounded inputs
 * (C_b): the result differs from sgemm()'s by up to about 2^-8 relative per
 * product.  Arguments, conventions, ownership, errors and asynchrony as
 * sgemm(); any alignment.  Each operand is rounded once per call into a
 * pooled workspace (2 bytes per element of op(A) and op(B), rows padded to a
 * multiple of 8 values), then CTA pairs compute 256x256 tiles, 64 k per
 * tile, with tcgen05.mma kind::f16 (SGEMM_VARIANT_TC_BF16).  Needs a device
 * where clusters of two CTAs can be co-scheduled, and K <= 2097120:
 * SGEMM_ERR_UNSUPPORTED otherwise.
 */
int sgemm_bf16(char transA, char transB, int64_t M, int64_t N, int64_t K,
               float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb,
               float beta, float *C, int64_t ldc,
               struct CUstream_st *stream);

/* What sgemm_bf16() would launch (sm_count as in sgemm_plan(); plan == NULL: -15). */
int sgemm_bf16_plan(char transA, char transB, int64_t M, int64_t N, int64_t K,
                    float alpha, const float *A, int64_t lda,
                    const float *B, int64_t ldb,
                    float beta, const float *C, int64_t ldc,
                    int sm_count, sgemm_plan_t *plan);

/*
 * sgemm_host -- the same operation with A, B and C in HOST memory (same
 * layout rules and argument checks as sgemm(); page-locked memory gives full
 * copy speed, pageable memory works but its copies are staged by the driver
 * and device-to-host copies then block the calling thread).  B is copied to
 * the device once; op(A) and C move in row blocks of C on two library-owned
 * streams, so copies of one block overlap the GEMM of the other.  Device
 * buffers come from a library-owned stream-ordered pool.  Asynchronous on
 * `stream`: the work starts after what is already on `stream`, and `stream`
 * waits for all of it; keep the host buffers alive and do not read C until
 * `stream` has completed.  Calls are serialised per device.
 */
int sgemm_host(char transA, char transB, int64_t M, int64_t N, int64_t K,
               float alpha, const float *A, int64_t lda,
               const float *B, int64_t ldb,
               float beta, float *C, int64_t ldc,
               struct CUstream_st *stream);

/*
 * sgemm_noalloc -- the same operation, arguments and results as sgemm(), for
 * callers that cannot allocate device memory during the call.  (The pages
 * have no counterpart; this is a library convenience.)
 *
 * sgemm() may grow its memory pool to hold split-K partial sums.  A caller
 * that has already given nearly all device memory to its own allocator, or
 * latency-critical code that cannot absorb a pool growing mid-run, cannot
 * allow that.  sgemm_noalloc() calls no cudaMalloc, cudaFree or other
 * allocating routine: the partial sums (split-K slices, or the stream-K
 * slots of the tensor-core kernel: 2 x 64 KiB per CTA, 19 MiB on 152 SMs)
 * go to a fixed scratch array of
 * SGEMM_NOALLOC_SCRATCH_BYTES compiled into the library, one per device,
 * held by every GPU that loads the library until the process exits.
 *
 * Where sgemm() would split operands into workspace arrays, sgemm_noalloc()
 * runs the kernel the planner takes without them: the CTA-pair kernel
 * (SGEMM_VARIANT_TC_PAIR) for SGEMM_VARIANT_TC_PRESPLIT, the one-CTA kernel's
 * rules (SGEMM_VARIANT_TC_TF32X3 or TC_PAIR) for SGEMM_VARIANT_TC_SKINNY:
 * the same error bounds, possibly different rounding.
 *
 * Limit: a problem whose split-K partial sums need more than
 * SGEMM_NOALLOC_SCRATCH_BYTES (see sgemm_plan_t.workspace_bytes) is rejected
 * with SGEMM_ERR_SCRATCH_LIMIT before anything is launched; C is untouched.
 * The first call on a device does a one-time set-up there (it looks up the
 * array's device address and sets kernel attributes); make that first call
 * before any stream capture (a set-up that fails returns SGEMM_ERR_CUDA and
 * is tried again by the next call).  The plan is sgemm()'s for the same
 * device (the same co-resident cluster count), except for the substitution
 * above.  All calls on a device share the one array:
 * calls whose kernels can overlap on the GPU (e.g. on unordered streams) race
 * on it, so order them.  CUDA failures return SGEMM_ERR_CUDA (the error code
 * is kept for sgemm_last_cuda_error(), as for sgemm()); in-kernel waits
 * use sgemm()'s limit (SGEMM_WAIT_TIMEOUT_MS).
 */
#define SGEMM_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB per device */

int sgemm_noalloc(char transA, char transB, int64_t M, int64_t N, int64_t K,
                  float alpha, const float *A, int64_t lda,
                  const float *B, int64_t ldb,
                  float beta, float *C, int64_t ldc,
                  struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_H */
