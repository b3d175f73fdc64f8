/*
 * sgemm.h -- C ABI of a single-precision GEMM library for one NVIDIA GB300
 * (compute capability 10.3, sm_103a).
 *
 * One call computes, on the caller's CUDA stream,
 *
 *     C = alpha * op(A) * op(B) + beta * C          op(X) = X or X^T
 *
 * for FP32 row-major matrices.  This is the product C(MxN) = A(MxK) x B(KxN) of
 * "CUDA矩阵乘法性能优化实战：从朴素内核到寄存器分块与Nsight剖析" (section 1.1, and
 * the matmul_naive/matmul_tiled kernels of sections 2.1 and 3.2, whose
 * signature matmul(A, B, C, M, N, K) this generalises), in the
 * D = alpha * A * B^T + beta * C form of the cloud.baidu.com article 9456745
 * (naive vs 2D block-tiled shared-memory matmul, naive-implementation
 * paragraph), with both operands optionally transposed.
 *
 * Layout (row-major throughout; every leading dimension counts elements):
 *   op(A) is M x K.  transA = N: A is stored M x K, lda >= max(1, K).
 *                    transA = T: A is stored K x M, lda >= max(1, M).
 *   op(B) is K x N.  transB = N: B is stored K x N, ldb >= max(1, N).
 *                    transB = T: B is stored N x K, ldb >= max(1, K).
 *   C is M x N, ldc >= max(1, N).
 * transA / transB accept 0 / 1 (SGEMM_OP_N / SGEMM_OP_T) or the characters
 * 'N', 'n', 'T', 't'.
 *
 * Pointers: A, B and C are DEVICE pointers (cudaMalloc'd, or any allocation the
 * device can address) on the current device.  The caller owns all of them; the
 * library never frees, keeps or reallocates them.  C must not overlap A or B.
 * Device memory of the library's own, per device, all of it under a limit the
 * caller sets with sgemm_set_scratch_limit() (initially the value of the
 * environment variable SGEMM_SCRATCH_LIMIT in bytes, else no limit):
 *   - a stream-K workspace (two 128 x 256 FP32 partial tiles per SM, ~40 MB
 *     on 152 SMs, plus 16 KiB of arrival counters), allocated the first time a
 *     product is split by stream-K;
 *   - an operand scratch buffer (grown in 64 MiB steps, at most 2 GiB),
 *     allocated the first time a product copies an operand ahead (a
 *     transpose, an aligning copy or a 3xTF32 split, see sgemm());
 * both kept until exit or until a lower limit frees them.  Calls on different
 * streams that use them are ordered by events.  A product whose buffer would
 * not fit under the limit runs without it (whole tiles instead of stream-K
 * splits, operands read in place), with the same result contract.  With a
 * limit of 0 the library allocates no device memory at all: what it owns is
 * then one status word per device (a __device__ variable) and host-side state
 * (tensor-map cache, events, kernel attributes).  sgemm_noalloc() never
 * allocates (see there).
 *
 * Environment: SGEMM_SCRATCH_LIMIT=<bytes> sets every device's initial scratch
 * limit (see sgemm_set_scratch_limit); SGEMM_VERBOSE=1 makes each CUDA-core
 * product print the plan it queued (kernel form, tile, grid, how split tiles
 * are finished) to stderr.  Both are read once.
 *
 * Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 * default stream).  Every call returns as soon as its work is queued; results
 * are ready once the stream reaches that point.  Argument errors are detected
 * on the host before anything is queued, and then nothing is launched.  A
 * pending error left by earlier, unrelated CUDA runtime calls is cleared
 * before the call's launches, so it does not fail this call.  The product
 * kernels are launched as programmatic dependents of whatever kernel precedes
 * them on the stream (cudaLaunchAttributeProgrammaticStreamSerialization): one
 * may be scheduled while that kernel finishes, but it reads and writes memory
 * only after griddepcontrol.wait, i.e. once that kernel has completed and its
 * writes are visible -- the stream's order is kept for every caller.
 *
 * CUDA graphs: sgemm(), sgemm_ex(), sgemm_strided_batched() and
 * sgemm_transpose() may be captured.  Inside a capture the library allocates
 * nothing: a product whose stream-K workspace or transpose scratch does not
 * exist yet (or is too small) runs without it; and once a capture has used
 * the scratch it is never freed (graphs hold its address): an eager product
 * that needs a larger one gets a new buffer of at least twice the size and
 * the old one is kept until exit.  Uses of these buffers inside graphs are
 * ordered against every other use through external event nodes, so graph
 * launches and eager calls on other streams may be mixed freely.
 *
 * Numerics: FP32 inputs and outputs; each output's K products are accumulated
 * in FP32 (FFMA) by the CUDA-core kernels, or from TF32 splits in FP32 by the
 * 3xTF32 tensor-core kernel.  The result matches the FP64-accumulated product
 * within a relative Frobenius error of 1e-5 and an absolute elementwise error of
 * 1e-4 * sqrt(K) for inputs of unit scale, and bit for bit when every input and
 * every partial sum is an integer below 2^24 in magnitude.  Denormals: no
 * kernel family flushes them to zero; the CUDA-core families keep subnormal
 * inputs, partial sums and results exactly as FP32 arithmetic does, and the
 * tensor-core family rounds subnormal inputs to TF32's subnormal spacing (see
 * SGEMM_ALGO_TC_3XTF32).  Degenerate cases follow BLAS: M == 0 or N == 0 does
 * nothing; K == 0 or alpha == 0 sets C = beta * C without reading A or B;
 * beta == 0 never reads C (NaN or garbage there is overwritten).
 */
#ifndef DENSE_FP32_MATRIX_10_GB300_SGEMM_H_
#define DENSE_FP32_MATRIX_10_GB300_SGEMM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SGEMM_API __attribute__((visibility("default")))
#else
#define SGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sgemm_op {
  SGEMM_OP_N = 0, /* op(X) = X   */
  SGEMM_OP_T = 1  /* op(X) = X^T */
} sgemm_op_t;

typedef enum sgemm_status {
  SGEMM_SUCCESS = 0,
  SGEMM_ERR_INVALID_VALUE = 1,  /* bad op, negative or too large M/N/K, leading
                                   dimension too small, NULL pointer with a
                                   nonzero extent, unknown algorithm */
  SGEMM_ERR_ALIASING = 2,       /* C's byte range overlaps A's or B's */
  SGEMM_ERR_UNSUPPORTED = 3,    /* no CUDA device, or not compute capability 10.3;
                                   or the requested algorithm cannot take these
                                   arguments (e.g. TMA with an unaligned ld) */
  SGEMM_ERR_LAUNCH = 4,         /* a CUDA call failed while queuing the work */
  SGEMM_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up a bounded wait (reported
                                   by sgemm_last_device_status) */
  SGEMM_ERR_SCRATCH_LIMIT = 6,  /* kept for ABI stability; no call returns it
                                   (sgemm_noalloc runs whole tiles instead
                                   when its array is too small) */
  SGEMM_ERR_DEVICE_BOUNDS = 7   /* only in a library built with
                                   SGEMM_DEBUG_BOUNDS=1: a kernel formed a
                                   shared- or global-memory index outside its
                                   tile, stage or matrix and skipped the access
                                   (reported by sgemm_last_device_status) */
} sgemm_status_t;

/*
 * Which kernel family runs.  SGEMM_ALGO_AUTO picks by shape, layout and
 * alignment; the others force one family (for tests and measurement).
 */
typedef enum sgemm_algo {
  SGEMM_ALGO_AUTO = 0,
  SGEMM_ALGO_SIMT_TMA = 1,     /* CUDA cores, FFMA, 8x8 outputs per thread; a TMA
                                  producer warp fills a multi-stage ring of
                                  swizzled shared-memory tiles.  Needs A and B
                                  16-byte aligned and lda, ldb multiples of 4. */
  SGEMM_ALGO_SIMT_CPASYNC = 2, /* same consumer warps; producer warps fill the
                                  ring with 4-byte cp.async.  Any alignment/ld. */
  SGEMM_ALGO_TC_3XTF32 = 3,    /* tcgen05 tensor cores, TMEM accumulator, each
                                  FP32 operand split into two TF32 parts and
                                  three products accumulated.  Large products
                                  split both operands ahead into library
                                  scratch (two extra launches) and run on CTA
                                  pairs (clusters of two, cta_group::2 MMAs
                                  on 256-row tiles).  Subnormals are not
                                  flushed (subnormal partial sums and results
                                  are kept), but a subnormal input is kept
                                  only to within 2^-137, half the spacing of
                                  TF32 subnormals: its bits below that are
                                  lost (exact when its significant bits fit
                                  TF32's 10-bit mantissa). */
  SGEMM_ALGO_NAIVE = 4,        /* one thread per output, operands read straight
                                  from global memory (the pages' first kernel;
                                  for comparison only) */
  SGEMM_ALGO_SMEM_TILED = 5,   /* 16x16 shared-memory tiles, one output per
                                  thread (the pages' second kernel; comparison) */
  SGEMM_ALGO_SMALL = 6,        /* small and skinny products: one launch, no
                                  workspace; one CTA per 32x32 tile of C, K split
                                  across its eight warps and their partial tiles
                                  added in a fixed order.  Any alignment/ld. */
  SGEMM_ALGO_REG_2X2 = 7,      /* the pages' third kernel (register tiling,
                                  "CUDA矩阵乘法性能优化实战..." sections 5.2-5.3):
                                  16x16 threads, 2x2 outputs held in registers
                                  per thread (32x32 tile), k-major shared tiles
                                  read with float2, float2 global loads where
                                  aligned; any layout (comparison only) */
  SGEMM_ALGO_REG_4X4 = 8       /* the same with 4x4 outputs per thread (64x64
                                  tile) and float4 loads (comparison only) */
} sgemm_algo_t;

/*
 * C = alpha * op(A) * op(B) + beta * C, kernel chosen automatically.
 * Returns SGEMM_SUCCESS once the work is queued on `stream`, or an error code
 * (see sgemm_status_t) with nothing queued.  Thread-safe.
 * Small products -- M * N * K <= 2^26, K <= 1024 and at most 608 tiles of
 * 32 x 32 -- run SGEMM_ALGO_SMALL: one launch, any layout, no workspace.
 * Large products whose op(A) or op(B) is k-contiguous (A stored M x K, or B
 * stored N x K) and that fill the GPU with 128 x 256 tiles first copy that
 * operand transposed into library scratch (one transpose launch each) and
 * then run with both operands m/n-contiguous; the result is bit-identical to
 * the in-kernel path.  Products of M * N * K >= 2^27 whose A or B is not
 * TMA-eligible (base not 16-byte aligned, or lda / ldb not a multiple of 4)
 * first copy that operand into 16-byte aligned scratch rows (one launch for
 * both; transposed instead where the rule above transposes it) and run the
 * SGEMM_ALGO_SIMT_TMA kernel, again bit-identical to that kernel on aligned
 * copies of the operands; smaller ones run SGEMM_ALGO_SIMT_CPASYNC in place.
 * sgemm_last_launch_count() reports all launches.
 */
SGEMM_API sgemm_status_t sgemm(int transA, int transB, int64_t M, int64_t N, int64_t K,
                     float alpha, const float *A, int64_t lda,
                     const float *B, int64_t ldb,
                     float beta, float *C, int64_t ldc, void *stream);

/*
 * As sgemm(), with the kernel family forced by `algo` (SGEMM_ALGO_AUTO gives
 * exactly sgemm()).  Returns SGEMM_ERR_UNSUPPORTED, with nothing queued, when
 * that family cannot take these arguments.
 */
SGEMM_API sgemm_status_t sgemm_ex(int transA, int transB, int64_t M, int64_t N, int64_t K,
                        float alpha, const float *A, int64_t lda,
                        const float *B, int64_t ldb,
                        float beta, float *C, int64_t ldc, void *stream,
                        sgemm_algo_t algo);

/*
 * Strided batch: for b = 0 .. batch-1,
 *     C_b = alpha * op(A_b) * op(B_b) + beta * C_b,
 * with A_b = A + b*strideA, B_b = B + b*strideB, C_b = C + b*strideC (strides
 * in elements, >= 0).  Attention's Q K^T, which the cloud.baidu.com article
 * 9456745 (introduction) names among the main uses of a GEMM kernel, is such
 * a batch of small products, one per head -- here one launch for the whole
 * batch instead of one per product.  A stride of 0 shares that operand
 * across the batch (e.g. one weight matrix for every product).
 * Layout and leading dimensions per product are as for sgemm().  When batch > 1
 * the C_b must not overlap one another (strideC >= (M-1)*ldc + N), and the
 * address range covered by all C_b must not meet the range covered by all A_b
 * or all B_b (else SGEMM_ERR_ALIASING; inputs may overlap each other, e.g.
 * sliding windows).  batch < 0 or a negative stride is SGEMM_ERR_INVALID_VALUE;
 * batch == 0, M == 0 or N == 0 do nothing; K == 0 or alpha == 0 scale every
 * C_b by beta.  Runs the CUDA-core kernels -- TMA loads (a 3-D tensor map per
 * strided operand) when bases, leading dimensions and strides are multiples of
 * 16 bytes and the map encodes, cp.async otherwise -- with the k-iterations of
 * the batch's tiles spread by stream-K like a single product's.  A
 * k-contiguous op(B) (transB = T) stored as dense consecutive blocks
 * (strideB == N * ldb) of products with at least 1024 rows is first copied
 * transposed, for the whole batch at once, into the library's operand
 * scratch (one more launch; skipped when the scratch limit does not admit
 * it).  batch * tiles per product must stay below 2^31
 * (SGEMM_ERR_UNSUPPORTED).
 */
SGEMM_API sgemm_status_t sgemm_strided_batched(int transA, int transB, int64_t M, int64_t N,
                                               int64_t K, float alpha, const float *A, int64_t lda,
                                               int64_t strideA, const float *B, int64_t ldb,
                                               int64_t strideB, float beta, float *C, int64_t ldc,
                                               int64_t strideC, int64_t batch, void *stream);

/*
 * Matrix transpose: out[c * ld_out + r] = in[r * ld_in + c] for r < rows,
 * c < cols -- the workload of "现代 CUDA 工具箱实战：从朴素代码到硬件极限的优化之路"
 * (hankli.space, widened from N x N to rows x cols with leading dimensions).
 * in is rows x cols (ld_in >= cols), out is cols x rows (ld_out >= rows), both
 * row-major device memory owned by the caller; elements of out outside the
 * cols x rows block are not written.  Values are copied bit for bit.
 * Errors: negative sizes or short leading dimensions -> INVALID_VALUE; in and
 * out overlapping (including in place) -> ALIASING; rows == 0 or cols == 0 do
 * nothing.  One launch, queued on `stream`; memory-bound (2 * rows * cols * 4
 * bytes), 16-byte vector accesses when both bases and leading dimensions are
 * 16-byte aligned.
 */
SGEMM_API sgemm_status_t sgemm_transpose(int64_t rows, int64_t cols, const float *in,
                                         int64_t ld_in, float *out, int64_t ld_out, void *stream);

/*
 * The family SGEMM_ALGO_AUTO would run for these arguments, or -1 if the
 * arguments are invalid.  Host only: queues nothing and touches no device
 * memory (it reads the device's SM count once).
 */
SGEMM_API int sgemm_select_algo(int transA, int transB, int64_t M, int64_t N, int64_t K,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      float alpha, float beta, const float *C, int64_t ldc);

/*
 * Number of kernel launches the last successful sgemm()/sgemm_ex() call on the
 * calling host thread queued (0 for M == 0 or N == 0).
 */
SGEMM_API int sgemm_last_launch_count(void);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word, in which a kernel records that it gave up a bounded wait (or, in a
 * SGEMM_DEBUG_BOUNDS=1 build, that it caught an out-of-range index).  Returns
 * SGEMM_SUCCESS, SGEMM_ERR_DEVICE_TIMEOUT, SGEMM_ERR_DEVICE_BOUNDS, or
 * SGEMM_ERR_LAUNCH if the synchronisation itself failed.  On an error it also
 * zeroes the stream-K arrival counters, which a kernel that gave up may have
 * left mid-count.
 */
SGEMM_API sgemm_status_t sgemm_last_device_status(void *stream);

/*
 * Caps, for the current device, the device memory that sgemm(), sgemm_ex()
 * and sgemm_strided_batched() may allocate for the library's own use (the
 * stream-K workspace and the operand scratch described at the top of this
 * file); `bytes` = UINT64_MAX removes the cap, 0 forbids any allocation.
 * Products queued afterwards that would need a buffer above the cap run
 * without it, with the same result contract.  If the library already holds
 * more than `bytes`, this call frees those buffers -- after the device has
 * finished the work queued on it (cudaFree waits for it) -- except buffers
 * that a captured CUDA graph may still use, which stay until exit (and keep
 * counting against the cap).  Returns SGEMM_SUCCESS, SGEMM_ERR_UNSUPPORTED
 * (no usable device) or SGEMM_ERR_LAUNCH (freeing failed).
 * Not part of the pages' interface: it exists so that callers whose own
 * allocator owns the device memory can hold the library to the ownership
 * contract "the caller owns all device memory" (limit 0).
 */
SGEMM_API sgemm_status_t sgemm_set_scratch_limit(uint64_t bytes);

/*
 * The current device's scratch limit and the bytes of device memory the
 * library holds there now (either pointer may be NULL).  The fixed array of
 * sgemm_noalloc() is not counted.  Returns SGEMM_SUCCESS or
 * SGEMM_ERR_UNSUPPORTED.
 */
SGEMM_API sgemm_status_t sgemm_get_scratch_limit(uint64_t *limit, uint64_t *held);

/*
 * Sets the limit, in nanoseconds of %globaltimer, that every wait inside the
 * library's kernels observes before it gives up and records
 * SGEMM_ERR_DEVICE_TIMEOUT (default 2e9 = 2 s; 0 restores the default).
 * Affects launches queued after the call, from any thread.
 */
SGEMM_API void sgemm_set_wait_budget_ns(uint64_t budget_ns);

/*
 * Queues one tiny kernel whose single thread waits on a shared-memory mbarrier
 * that nothing will ever complete, with the same bounded wait the GEMM kernels
 * use and a budget of `budget_ns`.  It lets a test watch the give-up path end
 * in SGEMM_ERR_DEVICE_TIMEOUT (read with sgemm_last_device_status) without
 * faulting or hanging anything.  Returns SGEMM_ERR_LAUNCH if queuing failed.
 */
SGEMM_API sgemm_status_t sgemm_selftest_wait_timeout(uint64_t budget_ns, void *stream);

/*
 * Size of the fixed device array that sgemm_noalloc uses as scratch: 20 MiB,
 * i.e. two 128 x 128 FP32 partial tiles for each of up to 160 CTAs.
 */
#define SGEMM_NOALLOC_SCRATCH_BYTES (20u * 1024u * 1024u)

/*
 * sgemm_noalloc -- the same product as sgemm(), guaranteed not to allocate
 * device memory.  (The pages have no counterpart; this is an entry point for
 * callers that may not let a library allocate.)
 *
 * sgemm() allocates its stream-K workspace with cudaMalloc the first time a
 * product needs one (unless sgemm_set_scratch_limit forbids it, and then
 * splits no tiles).  Callers that cannot allow a library to allocate but
 * still want split tiles -- programs whose own pool or caching allocator owns
 * the device memory, latency-sensitive loops (cudaMalloc may synchronise the
 * device and can fail under memory pressure), services with a fixed, audited
 * memory footprint -- call this instead.  Its scratch is a __device__ array
 * of SGEMM_NOALLOC_SCRATCH_BYTES, reserved on a device by the set-up below and
 * held until the process exits; the call itself makes no cudaMalloc, cudaFree
 * or other allocating call.
 *
 * Arguments, layout, numerics and degenerate cases are those of sgemm(); it
 * runs the CUDA-core kernels (128 x 128 or 128 x 64 tiles) and updates
 * sgemm_last_launch_count() like sgemm().  A product whose split tiles would
 * need more than the array holds runs whole tiles only.
 * Set-up: the first call on a device -- any call with valid arguments, an
 * empty one (M = 0) included -- looks up the array's device address and loads
 * every kernel this entry point launches, with that device current.  Under
 * CUDA's lazy module loading (the default since CUDA 12.2) that is when the
 * runtime reserves the array and the kernels' code on the device.  Make this
 * first call before handing the rest of the device's memory to your own pool
 * and before any stream capture.
 * Sharing: all calls use the one array and leave its contents behind; nothing
 * in it needs clearing between calls, but calls that overlap on the GPU (on
 * streams not ordered with each other) race on it.
 */
SGEMM_API sgemm_status_t sgemm_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                       float alpha, const float *A, int64_t lda,
                                       const float *B, int64_t ldb,
                                       float beta, float *C, int64_t ldc, void *stream);

/* Static English text for a status code (never NULL). */
SGEMM_API const char *sgemm_status_string(sgemm_status_t status);

/* Static name of an algorithm ("auto", "simt_tma", ...), or "unknown". */
SGEMM_API const char *sgemm_algo_name(sgemm_algo_t algo);

/* Library version as "major.minor.patch". */
SGEMM_API const char *sgemm_version(void);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* DENSE_FP32_MATRIX_10_GB300_SGEMM_H_ */
