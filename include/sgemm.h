/*
 * sgemm.h -- C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * The operation is C = alpha * A * B + beta * C on row-major FP32 matrices,
 * computed with plain FP32 fused multiply-add (no tensor cores, no TF32):
 * - "Optimizing Matrix Multiply on CUDA, Part 1", section "Counting the Work":
 *   C[i][j] is the dot product of row i of A and column j of B.
 * - "GEMM from Scratch", Module 02 ("One Thread Per Output"): row-major
 *   operands A[x*K+i], B[i*N+y], C[x*N+y] and the epilogue
 *   alpha*tmp + beta*C[x*N+y].
 * - "Optimizing CUDA matmul, steps 4 to 6", section "The honest target":
 *   plain FP32 in, FP32 accumulate, FP32 out, no TF32 path.
 *
 * Layout: element (i, j) of a row-major matrix X with leading dimension ldx
 * lives at X[i * ldx + j]; ldx counts elements and may exceed the row length.
 * A is M x K (lda >= max(1, K)), B is K x N (ldb >= max(1, N)), C is M x N
 * (ldc >= max(1, N)).
 *
 * Conventions the pages leave open (BLAS practice):
 * - beta == 0: C is write-only; whatever C held (NaN included) is ignored.
 * - alpha == 0 or K == 0: A and B are not read; C = beta * C.
 * - M == 0 or N == 0: nothing is done.
 * - Any summation order of the K products is allowed; for a given shape,
 *   leading dimensions and pointer alignment the result is bitwise
 *   reproducible from call to call.
 *
 * All entry points return an sgemm_status_t.  Validation errors are returned
 * before any work is queued.  Calls are asynchronous with respect to the
 * host; results are ready once the given stream has been synchronised.
 */
#ifndef GB300_SGEMM_H
#define GB300_SGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SGEMM_API __attribute__((visibility("default")))
#else
#define SGEMM_API
#endif

typedef int sgemm_status_t;

enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = 1,    /* a size, leading dimension or pointer is invalid  */
    SGEMM_ERR_ALLOC = 2,          /* internal workspace could not be allocated        */
    SGEMM_ERR_TMA = 3,            /* a TMA tensor map could not be encoded            */
    SGEMM_ERR_LAUNCH = 4,         /* a kernel launch or CUDA runtime call failed      */
    SGEMM_ERR_DEVICE_TIMEOUT = 5, /* a bounded device-side wait gave up (see below)   */
    SGEMM_ERR_NO_DEVICE = 6,      /* no CUDA device, or it is not sm_103              */
    SGEMM_ERR_UNSUPPORTED = 7,    /* the request names something this build lacks     */
    SGEMM_ERR_SCRATCH_LIMIT = 8   /* beyond what sgemm_run_skinny_noalloc's fixed buffer takes */
};

/*
 * sgemm_run -- C = alpha * A * B + beta * C on the GPU.
 *
 * A, B, C: device pointers owned by the caller.  A and B are only read; C is
 *   read (when beta != 0) and written.  C must not overlap A or B.  Any
 *   4-byte-aligned pointers are accepted; 16-byte-aligned pointers with
 *   leading dimensions that are multiples of 4 take the fastest path.
 * stream: a cudaStream_t (NULL = the legacy default stream).  All work is
 *   queued on it; the call does not synchronise.
 * Internal workspace (partial tiles for K-split schedules) is allocated by
 *   the library on first use per (device, stream) and kept until
 *   sgemm_release_workspace().  Concurrent calls on one stream are ordered by
 *   the stream; calls on different streams use different workspaces.
 * Returns SGEMM_ERR_INVALID_ARG if M, N or K < 0, a leading dimension is below
 *   its minimum, or a pointer the operation must dereference is NULL or not
 *   4-byte aligned; SGEMM_ERR_LAUNCH if a launch fails.  A bounded device wait
 *   that gave up is reported by sgemm_device_status().
 */
SGEMM_API sgemm_status_t sgemm_run(int64_t M, int64_t N, int64_t K, float alpha,
                         const float *A, int64_t lda, const float *B, int64_t ldb,
                         float beta, float *C, int64_t ldc, void *stream);

/* Activation applied last by sgemm_run_epilogue. */
enum {
    SGEMM_ACT_NONE = 0, /* identity                                            */
    SGEMM_ACT_RELU = 1  /* x < 0 ? 0 : x  (a NaN stays NaN, -0 stays -0)       */
};

/*
 * sgemm_run_epilogue -- C = act(alpha * A * B + beta * C + bias) on the GPU,
 * the bias and the activation applied in the GEMM's own epilogue, with no
 * extra pass over C ("GEMM from Scratch", end of Module 08, "When to just
 * call the library": fusing an epilogue or activation into the product is
 * the reason given for writing one's own GEMM).
 *
 * bias: NULL, or a device pointer to N floats (4-byte aligned, owned by the
 *   caller, only read); bias[j] is added to every element of column j, as a
 *   linear layer's bias is added to each row of X * W.
 * activation: one of SGEMM_ACT_*.  Other values return SGEMM_ERR_INVALID_ARG.
 * Each element is rounded as fl(fl(alpha * acc + beta * c) + bias[j]) and the
 * activation is exact.  Everything else (arguments, layout, workspace,
 * asynchrony, errors) is as for sgemm_run, which is this call with
 * bias = NULL and SGEMM_ACT_NONE.  When alpha == 0 or K == 0 the result is
 * act(beta * C + bias); when M == 0 or N == 0 nothing is done.
 */
SGEMM_API sgemm_status_t sgemm_run_epilogue(int64_t M, int64_t N, int64_t K, float alpha,
                                  const float *A, int64_t lda, const float *B, int64_t ldb,
                                  float beta, float *C, int64_t ldc, const float *bias,
                                  int activation, void *stream);

/*
 * sgemm_run_host -- the same operation on HOST matrices.
 *
 * A, B, C are host pointers (pinned memory gives full copy bandwidth).  The
 * call copies A, B (and C when beta != 0) to device buffers it owns, runs
 * sgemm_run on `stream`, copies C back and synchronises `stream` before
 * returning, so C holds the result on return.  From M = 1024 on, when each
 * block keeps enough work for the tiled kernel, the rows of A and C are cut
 * into two to four blocks: B goes in first, then block i + 1 is copied in and
 * block i - 1 out (on two internal streams, after the work already queued on
 * `stream`) while block i is computed.  Device buffers are
 * kept for reuse until sgemm_release_workspace().
 */
SGEMM_API sgemm_status_t sgemm_run_host(int64_t M, int64_t N, int64_t K, float alpha,
                              const float *A, int64_t lda, const float *B, int64_t ldb,
                              float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_run_skinny_noalloc -- the skinny-M product (M <= 16) with no device
 * allocation at all.  (The pages have no counterpart; this is a library
 * convenience.)
 *
 * For callers that cannot call cudaMalloc: code running while a framework's
 * caching allocator owns the device memory, loops that must not allocate after
 * start-up, or code that must not put a synchronising allocation between
 * queued work.  sgemm_run allocates its stream-K workspace on first use; this
 * entry point takes partial sums, tickets and its error word from one fixed
 * 5 MiB + 16 KiB buffer compiled into the library as a __device__ array,
 * which every GPU that loads the library holds until the process exits.
 *
 * Same arguments, layout and conventions as sgemm_run (device pointers owned
 * by the caller, queued on `stream`, no host synchronisation), with limits:
 * M <= 16; N <= 1,048,576 (4096 slabs of 256 columns); A and B 16-byte
 * aligned with lda and ldb multiples of 4.  Requests beyond them return
 * SGEMM_ERR_SCRATCH_LIMIT before any work is queued.  Sizes no kernel of the
 * library takes (K or N above 2^30) return SGEMM_ERR_INVALID_ARG, as from
 * sgemm_run; a K so deep that the kernel's position counter would overflow
 * (about 2^18 * 32 rows per 256-column slab) returns SGEMM_ERR_UNSUPPORTED.
 * The plan uses at most 160 CTAs in total (one per SM), so a GPU with more
 * than 160 SMs leaves the others idle.  The first call on each device looks
 * up the buffer's device address (no work is queued by that set-up, but make
 * the first call before any stream capture).  Every call shares the one
 * buffer: calls that overlap on the GPU (different streams, or concurrent
 * host threads) race and must be ordered by the caller.  Each call clears
 * the tickets it uses before its kernel runs.  A bounded device wait that
 * gives up is recorded in the buffer's own error word, which no call clears:
 * read it with sgemm_skinny_noalloc_status(), not sgemm_device_status().
 */
SGEMM_API sgemm_status_t sgemm_run_skinny_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                                  const float *A, int64_t lda, const float *B,
                                                  int64_t ldb, float beta, float *C, int64_t ldc,
                                                  void *stream);

/*
 * sgemm_skinny_noalloc_status -- synchronise `stream`, then read and clear
 * the error word of sgemm_run_skinny_noalloc's fixed buffer on the current
 * device.  Returns SGEMM_ERR_DEVICE_TIMEOUT if a call since the last read
 * gave up a bounded device wait (the C it wrote is then undefined; the next
 * call is valid, since each call clears its tickets first),
 * SGEMM_ERR_LAUNCH if the stream reports a CUDA error, SGEMM_ERR_NO_DEVICE
 * without an sm_103 device, else SGEMM_OK.  Allocates nothing.  (A library
 * convenience; the pages have no counterpart.)
 */
SGEMM_API sgemm_status_t sgemm_skinny_noalloc_status(void *stream);

/* Human-readable name of a status code (a static string). */
SGEMM_API const char *sgemm_status_string(sgemm_status_t status);

/*
 * sgemm_device_status -- synchronise `stream`, then read and clear the
 * library's device error word on the current device.  Returns
 * SGEMM_ERR_DEVICE_TIMEOUT if any kernel since the last call gave up a
 * bounded wait (its output is then undefined; the library resets its own
 * workspace counters so later calls are valid), SGEMM_ERR_LAUNCH if the
 * stream reports a CUDA error, else SGEMM_OK.
 */
SGEMM_API sgemm_status_t sgemm_device_status(void *stream);

/*
 * sgemm_plan_describe -- host-only: write into buf (NUL-terminated, at most
 * len bytes) the plan sgemm_run would choose for these sizes, leading
 * dimensions and pointer addresses on a GPU with `num_sms` SMs (0 = query the
 * current device).  The text is one line of key=value pairs: kernel variant,
 * tile, grid, data-parallel tiles, stream-K tiles and share, estimated
 * busiest-SM cost.  Touches no device memory.  Returns SGEMM_ERR_INVALID_ARG
 * on bad sizes, SGEMM_ERR_NO_DEVICE if num_sms == 0 and no device is present.
 */
SGEMM_API sgemm_status_t sgemm_plan_describe(int64_t M, int64_t N, int64_t K,
                                   int64_t lda, int64_t ldb, int64_t ldc,
                                   uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
                                   float beta, int num_sms, char *buf, size_t len);

/*
 * sgemm_set_plan_override -- testing and benchmarking hook, process-wide.
 * variant: -1 = automatic; otherwise one of SGEMM_VARIANT_*.
 * splits: for the stream-K variants (and the mid-size ones), 0 = automatic,
 *   else the number of k-iterations each CTA takes in the stream-K region is
 *   chosen so that tiles split into about `splits` pieces.
 * Returns SGEMM_ERR_INVALID_ARG for an unknown variant.
 */
enum {
    SGEMM_VARIANT_AUTO = -1,
    SGEMM_VARIANT_GENERIC = 0,   /* any alignment: 64x64 tile, bounds-checked loads  */
    SGEMM_VARIANT_TILE = 1,      /* TMA + FFMA2 128x256 tile, whole tiles only        */
    SGEMM_VARIANT_STREAMK = 2,   /* same kernel, data-parallel waves + stream-K tail  */
    SGEMM_VARIANT_SKINNY = 3,    /* small-M streaming kernel (HBM-bound shapes)       */
    SGEMM_VARIANT_MID = 4,       /* cp.async + FFMA2 128x128 tile, any alignment,     */
                                 /* data-parallel waves + stream-K tail               */
    SGEMM_VARIANT_MID64 = 5,     /* the same kernel with 64x128 tiles                 */
    SGEMM_VARIANT_KSPLIT = 6,    /* cp.async + FFMA2 64x128 tile per CTA, K split     */
                                 /* over four warp groups inside the CTA              */
    SGEMM_VARIANT_NARROW = 7,    /* N <= 4: a warp per row of A (A x products)        */
    SGEMM_VARIANT_KSPLIT64 = 8,  /* the split-K kernel with 64x64 tiles (8 k-groups)   */
    SGEMM_VARIANT_SMALL = 9      /* 32x32 tiles, K split over four thread groups      */
};
SGEMM_API sgemm_status_t sgemm_set_plan_override(int variant, int splits);

/*
 * sgemm_set_wait_timeout_ns -- testing hook: the limit (nanoseconds of GPU
 * global time) every bounded device-side wait uses; 0 restores the default
 * (one second).  skip_loads_from >= 0 makes the copy producer of the tiled
 * kernels stop issuing loads at that k-iteration of each CTA, so the waits
 * for them run out (a flag that nothing sets); -1 disables it.
 */
SGEMM_API sgemm_status_t sgemm_set_wait_timeout_ns(uint64_t timeout_ns, int skip_loads_from);

/*
 * sgemm_set_tile_config -- tuning hook, process-wide: the form of the
 * multiply-add in the tiled kernel, its number of TMA ring stages and the
 * height of each thread's micro-tile.
 * fma_mode: 0 = one FFMA per product; 1 = packed pairs along n with the A
 *   value duplicated in registers; 2 = packed pairs along n with A stored
 *   duplicated in shared memory; 3 = packed pairs along m with the B value
 *   duplicated in registers (default).
 * stages: 3 or 4 (default 3).
 * micro_m: 16 (256 threads of 16 x 8); the only height this build contains.
 * All forms compute the same IEEE FP32 products and sums.  Returns
 * SGEMM_ERR_INVALID_ARG for a combination this build does not contain.
 */
SGEMM_API sgemm_status_t sgemm_set_tile_config(int fma_mode, int stages, int micro_m);

/*
 * sgemm_run_3xtf32 -- the same operation, C = alpha * A * B + beta * C, on
 * the tensor cores by split-precision emulation ("3xTF32"): each FP32 operand
 * x is split into TF32 parts hi = tf32(x) and lo = tf32(x - hi) (round to
 * nearest), and a * b is taken as hi_a*hi_b + hi_a*lo_b + lo_a*hi_b,
 * accumulated in FP32.  A separate entry point: sgemm_run never takes it,
 * because the FP32 contract excludes TF32 arithmetic
 * ("Optimizing CUDA matmul, steps 4 to 6", section "The honest target");
 * tensor cores are the route the pages name past FP32-core parity ("GEMM from
 * Scratch", Module 07; "Optimizing Matrix Multiply on CUDA, Part 2", section
 * "Looking Back").
 *
 * Arguments, layout, ownership and errors are those of sgemm_run; pointers
 * need only 4-byte alignment.  A split pass writes hi and lo copies of B
 * (transposed to K-major) into a per-(device, stream) workspace of
 * 8 * K' * ceil(N/w)*w bytes, K' = ceil(K/32)*32 and w the tile width (64 to
 * 256) chosen for the shape; A is split tile by tile inside the kernel (A not
 * 16-byte aligned, or lda not a multiple of 4, is first copied to aligned
 * rows in the same workspace: 4 * M * ceil(K/4)*4 more bytes).  A product
 * cut into s K ranges (see sgemm_set_3xtf32_config) adds 4 * s * M' * N'
 * bytes for the ranges' raw tiles (M', N' rounded up to the tile).  The
 * workspace is kept until sgemm_release_workspace().
 * Accuracy: measured within the FFMA path's bound
 * 2 * K * 2^-24 * (|alpha| (|A||B|)ij + |beta| |Cij|) on the test
 * distributions; no worst-case proof (the tensor core's accumulation rounding
 * is not documented).  Products with K < 64 or M <= 16 run the FFMA kernels
 * (the split's own error, up to about 3 * 2^-22 |a b| per product, would use
 * up the bound of a short sum, and such shapes gain nothing from the tensor
 * cores).  Non-finite values in A or B give NaN in the outputs they reach
 * (hi - x is not finite); |x| at or above (2 - 2^-11) * 2^127 rounds to Inf
 * in the split.
 * Results are bitwise reproducible for a given shape.
 */
SGEMM_API sgemm_status_t sgemm_run_3xtf32(int64_t M, int64_t N, int64_t K, float alpha,
                                          const float *A, int64_t lda, const float *B,
                                          int64_t ldb, float beta, float *C, int64_t ldc,
                                          void *stream);

/*
 * sgemm_run_3xtf32_epilogue -- sgemm_run_3xtf32 with the epilogue of
 * sgemm_run_epilogue: C = act(alpha * A * B + beta * C + bias), bias a
 * device vector of N floats (or NULL), activation SGEMM_ACT_NONE or
 * SGEMM_ACT_RELU, each element rounded as fl(fl(alpha*acc + beta*c) + bias_j)
 * before the activation.  Argument checks and errors are those of
 * sgemm_run_epilogue; accuracy that of sgemm_run_3xtf32.
 */
SGEMM_API sgemm_status_t sgemm_run_3xtf32_epilogue(int64_t M, int64_t N, int64_t K, float alpha,
                                                   const float *A, int64_t lda, const float *B,
                                                   int64_t ldb, float beta, float *C, int64_t ldc,
                                                   const float *bias, int activation, void *stream);

/*
 * sgemm_plan_describe_3xtf32 -- host-only: write into buf (NUL-terminated, at
 * most len bytes) what sgemm_run_3xtf32 would do for these sizes, A's leading
 * dimension and address on a GPU with `num_sms` SMs (0 = query the current
 * device), under the current sgemm_set_3xtf32_config settings: "path=ffma"
 * (the FFMA kernels take the call), or "path=tensor" followed by the K slice,
 * ring stages, CTAs per SM, whether A is split in the kernel, the tile width,
 * the K split, the K slices and the CTA count.  Touches no device memory.
 * Returns SGEMM_ERR_INVALID_ARG on bad sizes, SGEMM_ERR_NO_DEVICE if
 * num_sms == 0 and no device is present.
 */
SGEMM_API sgemm_status_t sgemm_plan_describe_3xtf32(int64_t M, int64_t N, int64_t K, int64_t lda,
                                                    uint64_t a_addr, int num_sms, char *buf,
                                                    size_t len);

/*
 * sgemm_set_3xtf32_config -- tuning hook, process-wide, for the 3xTF32 kernel.
 * bk: the K depth of one pipeline stage, 16 (64-byte swizzled rows, the
 *   default) or 32 (two stages of 128-byte rows, one CTA per SM).
 * a_in_kernel: 1 = the kernel loads A itself and splits each A tile in
 *   shared memory; 0 = a split pass writes A's hi and lo parts first;
 *   -1 (default) = 1 when M*N >= 48 * 2^20 and A's rows start on 128-byte
 *   lines (A 128-byte aligned, lda a multiple of 32), else 0.
 * splits: the number of K ranges each output tile is cut into, 1 to 8, or
 *   0 (default) = chosen per call from a cost model of whole waves: deep
 *   products with few tiles are cut so that more SMs work, and a reduction
 *   kernel adds the ranges' raw tiles in range order, then applies alpha and
 *   beta.  A count that leaves a range under 16 K slices is not taken.
 * ctas_per_sm: 1 = one CTA per SM with a 4-stage ring; 2 = two CTAs per SM
 *   with 2 stages each (bk 16 only), so that one CTA's epilogue and start-up
 *   overlap the other's MMAs; 0 (default) = 2 when the launch has more CTAs
 *   than the GPU has SMs, else 1.
 * For a given split count all forms compute the same products in the same
 * order (bitwise equal results).  SGEMM_ERR_INVALID_ARG for other values.
 */
SGEMM_API sgemm_status_t sgemm_set_3xtf32_config(int bk, int a_in_kernel, int splits,
                                                 int ctas_per_sm);

/* Free every workspace and host-path buffer the library holds on all devices. */
SGEMM_API sgemm_status_t sgemm_release_workspace(void);

#ifdef __cplusplus
}
#endif

#endif /* GB300_SGEMM_H */
