/*
 * qm.h — C ABI of libqm: the GGML Q4_0 x f32 quantized matmul, the Q4_0
 * dequant and the Q8_0 dequant and quantize, as hand-written CUDA kernels for
 * sm_103a (GB300).
 *
 * Operations (defined in "fuel-vulkan-kernels — quantized (GGML) kernel
 * contracts", fuel-dispatch 0.20.71, kernel-contracts/vulkan/quantized.fkc.md):
 *
 *   Q4_0 block: 18 bytes for 32 elements.  Bytes 0-1: the scale d, IEEE
 *   binary16, little-endian.  Bytes 2-17: 16 quant bytes; element j (0..15) is
 *   the low nibble of quant byte j and element j+16 its high nibble.  Element
 *   value = (nibble - 8) * d, nibble unsigned 0..15   (section "dequant_q4_0").
 *
 *   Matmul: C[m][n] = sum over k of A[m][k] * W[n][k], A f32 row-major [M][K],
 *   W a row-major [N][K/32] stream of Q4_0 blocks (row n holds blocks
 *   n*K/32 .. n*K/32 + K/32 - 1), C f32 row-major [M][N], K a multiple of 32
 *   (sections "qmatvec_q4_0" and "matmul_q4_0_tiled").  M = 1..8 runs the
 *   decode-regime GEMV kernels, M >= 9 the prefill GEMM.  The sum is taken in
 *   f32 in an order of the kernel's choosing; results agree with the exact
 *   sum to |error| <= 1e-5 * sum_k |A[m][k] * W[n][k]| + 1e-7 per element.
 *   The same call on the same inputs gives bitwise the same C (no atomics).
 *
 * Conventions for every entry point:
 *   - Pointers are device memory owned by the caller (cudaMalloc'd, managed,
 *     or mapped host memory with a device address).  Work is enqueued on
 *     `stream` (a cudaStream_t passed as void*; NULL means the legacy default
 *     stream) on the current device, and results are visible once that
 *     stream has been synchronized; no entry point but qm_device_status
 *     synchronizes.  Calls are thread-safe.
 *   - Memory: no entry point allocates device memory, and none writes
 *     anything but its outputs (and, for qm_matmul_q4_0_noalloc, its fixed
 *     scratch array).  The prefill GEMM splits A into bf16 pieces inside the
 *     kernel.  Where a GEMM or GEMV splits K over S CTAs (too few output tiles
 *     or rows to fill the SMs), S is 2, 4 or 8 and the S CTAs form a
 *     thread-block cluster that adds the partial sums in its shared memory;
 *     where those clusters would not all be resident at once, K is not split.
 *     The first call on a device sets kernel attributes and queries the
 *     device (host-side state only); after it, calls on any stream, including
 *     one being captured into a CUDA graph, enqueue kernels and nothing else.
 *   - Launch: the fast kernels are launched with programmatic dependent
 *     launch, so one may start its prologue while the previous kernel on the
 *     stream finishes; it reads and writes memory only after that kernel has
 *     completed, so stream order is kept exactly as for ordinary launches.
 *   - Operands are contiguous; no strides, offsets or broadcasts.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     failed check returns a negative status and leaves memory untouched.
 *   - An output never aliases an input: overlapping byte ranges are rejected.
 */
#ifndef QM_H
#define QM_H

#include <stdint.h>

#if defined(__GNUC__)
#define QM_API __attribute__((visibility("default")))
#else
#define QM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define QM_OK 0
#define QM_ERR_NULL (-1)        /* a required pointer is NULL                    */
#define QM_ERR_SHAPE (-2)       /* negative size, K % 32 != 0, or a size whose
                                   byte count does not fit in int64              */
#define QM_ERR_ALIGN (-3)       /* wq not 2-byte aligned, or A/C/out not 4-byte  */
#define QM_ERR_ALIAS (-4)       /* an output overlaps an input                   */
#define QM_ERR_CUDA (-5)        /* a CUDA call or kernel launch failed           */
#define QM_ERR_TIMEOUT (-6)     /* a kernel gave up a bounded wait (see
                                   qm_device_status)                             */
#define QM_ERR_UNSUPPORTED (-7) /* the forced algorithm cannot run this shape    */
#define QM_ERR_POINTER (-8)     /* a pointer is not device memory of the current
                                   device                                        */
#define QM_ERR_TOO_LARGE (-9)   /* beyond the fixed scratch of
                                   qm_matmul_q4_0_noalloc (M > 8)               */

/* Algorithms for qm_matmul_q4_0_algo. */
#define QM_ALGO_AUTO 0      /* what qm_matmul_q4_0 picks: GEMV_PK for M <= 2 and
                               N <= 1024, GEMV for M <= 8, otherwise GEMM_TC
                               where it applies, else GEMM_SIMT              */
#define QM_ALGO_GEMV 1      /* decode-regime GEMV on tensor cores (mma.sync, bf16
                               pieces, f32 sums); M 1..8                         */
#define QM_ALGO_GEMM_SIMT 2 /* prefill GEMM on FP32 FMA; any M >= 1              */
#define QM_ALGO_GEMV_SIMT 3 /* decode-regime GEMV on FP32 FMA; M 1..8             */
#define QM_ALGO_GEMM_TC 4   /* prefill GEMM on tcgen05 tensor cores (split bf16);
                               needs K % 256 == 0 and 16-byte aligned A and wq  */
#define QM_ALGO_GEMV_PK 5   /* decode-regime GEMV on packed FP32 FMA
                               (fma.rn.f32x2), one weight row per lane; M 1..2 */

/* Library version: major * 10000 + minor * 100 + patch. */
QM_API int qm_version(void);

/* A static, human-readable string for a status code. */
QM_API const char* qm_status_string(int status);

/*
 * qm_dequant_q4_0 — section "dequant_q4_0": out[32*b + j] = (q_j(b) - 8) * d(b)
 * for every block b < n_blocks and j < 32.
 *   wq       : n_blocks * 18 bytes of Q4_0 blocks, 2-byte aligned (16-byte
 *              aligned takes the fast path).
 *   n_blocks : number of blocks, >= 0.  0 enqueues nothing.
 *   out      : n_blocks * 32 floats, 4-byte aligned (16-byte aligned takes the
 *              fast path); must not overlap wq.
 * Exact: the product of an integer in [-8, 7] and a binary16 scale is
 * representable in f32, so the result is bit-identical to the definition,
 * including the sign of zero (q = 8 with d < 0 gives -0.0), infinities
 * (q != 8 with d = +-inf) and NaN (q = 8 with d infinite, or d NaN).
 * Returns QM_OK or a negative status.
 */
QM_API int qm_dequant_q4_0(const void* wq, int64_t n_blocks, float* out, void* stream);

/*
 * qm_dequant_q8_0 — section "dequant_q8_0": out[32*b + j] = qs_j(b) * d(b)
 * for every block b < n_blocks and j < 32.  A Q8_0 block is 34 bytes: the
 * scale d (IEEE binary16, little-endian) in bytes 0-1, then 32 signed 8-bit
 * quants qs_0 .. qs_31.
 *   wq       : n_blocks * 34 bytes, any alignment (16-byte aligned, with a
 *              16-byte aligned out, takes the fast path).
 *   n_blocks : number of blocks, >= 0.  0 enqueues nothing.
 *   out      : n_blocks * 32 floats, 4-byte aligned; must not overlap wq.
 * Exact: an 8-bit integer times a binary16 scale is representable in f32, so
 * the result is bit-identical to the definition, including the sign of zero,
 * infinities and NaN.  Returns QM_OK or a negative status.
 */
QM_API int qm_dequant_q8_0(const void* wq, int64_t n_blocks, float* out, void* stream);

/*
 * qm_quantize_q8_0 — section "quantize_q8_0": each block of 32 consecutive
 * elements of x becomes one 34-byte Q8_0 block with d = max|x| / 127 and
 * qs = round(x / d).  Where the section is silent this library takes:
 *   - f32 arithmetic; d = max|x| / 127 and each x / d are single correctly
 *     rounded f32 divisions; NaN elements do not raise the max;
 *   - the stored scale is d narrowed to binary16, round to nearest even
 *     (values from 65520 up become infinity);
 *   - round() takes halfway cases away from zero; qs is clamped to
 *     [-127, 127] (this binds only when d is an f32 subnormal);
 *   - qs = 0 where d is 0 or x / d is NaN.
 *   x          : n_elements floats, 4-byte aligned (16-byte aligned, with a
 *                16-byte aligned out, takes the fast path).
 *   n_elements : >= 0 and a multiple of 32, else QM_ERR_SHAPE.  0 enqueues
 *                nothing.
 *   out        : n_elements / 32 * 34 bytes, any alignment; must not overlap x.
 * Deterministic: every block depends only on its own 32 inputs.
 * Returns QM_OK or a negative status.
 */
QM_API int qm_quantize_q8_0(const float* x, int64_t n_elements, void* out, void* stream);

/*
 * qm_matmul_q4_0 — C = A x dequant(W)^T (see the header comment).
 *   A  : M*K floats, row-major [M][K], 4-byte aligned.
 *   wq : N*(K/32) Q4_0 blocks = N*K*9/16 bytes, row-major [N][K/32], 2-byte
 *        aligned.  Rows are 16-byte aligned, and the fastest GEMV path is
 *        taken, when wq is 16-byte aligned and K % 256 == 0.
 *   C  : M*N floats, row-major [M][N], 4-byte aligned; must overlap neither A
 *        nor wq.  Every element of C is written.
 *   M, N, K : M, N >= 0; K >= 0 with K % 32 == 0.
 * M == 0 or N == 0 enqueues nothing.  K == 0 sets C to +0.0 (the empty sum).
 * Returns QM_OK or a negative status.
 */
QM_API int qm_matmul_q4_0(const float* A, const void* wq, float* C, int64_t M,
                   int64_t N, int64_t K, void* stream);

/*
 * qm_matmul_q4_0_algo — qm_matmul_q4_0 with the algorithm forced (QM_ALGO_*),
 * for tests and benchmarks.  Returns QM_ERR_UNSUPPORTED when the algorithm
 * cannot run the shape (a GEMV with M > 8), QM_ERR_SHAPE for an unknown
 * algorithm number.
 */
QM_API int qm_matmul_q4_0_algo(const float* A, const void* wq, float* C, int64_t M,
                        int64_t N, int64_t K, int algo, void* stream);

/*
 * qm_device_status — synchronizes `stream` and reads the library's device
 * error word for the current device.  Kernels that wait on asynchronous
 * copies give up after a bounded number of polls, set this word and return
 * early (their output is then incomplete).  Returns QM_OK if the word is
 * clear, QM_ERR_TIMEOUT if a wait gave up, QM_ERR_CUDA if the synchronize or
 * the read failed.  With clear != 0 the word is reset after reading.
 */
QM_API int qm_device_status(void* stream, int clear);

/*
 * qm_selftest_wait_timeout — exercises the failure path of the bounded waits
 * without faulting or hanging anything.  No counterpart on the kernel-contract
 * pages; it exists so that tests can check, on a real GPU, that a wait which
 * runs out is reported and that the context stays usable.  Enqueues on
 * `stream` one kernel in which a single thread waits on an mbarrier that
 * nothing completes, giving up after 65536 polls; it then sets the device
 * error word and returns.  The next qm_device_status on the stream returns
 * QM_ERR_TIMEOUT (and, with clear != 0, resets the word, after which
 * qm_device_status returns QM_OK again).  No memory is read or written but the
 * error word.  Returns QM_OK, or QM_ERR_CUDA if the launch failed.
 */
QM_API int qm_selftest_wait_timeout(void* stream);

/*
 * qm_matmul_q4_0_noalloc — the decode-regime product C = A x dequant(W)^T for
 * M = 1..8, for callers that cannot call cudaMalloc.  No counterpart on the
 * kernel-contract pages: it exists for code that must not allocate device
 * memory at call time, such as a custom allocator or memory-pool callback,
 * a process running under a hard device-memory cap, or a runtime that owns
 * all device memory.  It meets the partial sums of a split K in a fixed array
 * compiled into the library (qm_matmul_q4_0 adds them up inside thread-block
 * clusters instead, and allocates nothing either), and allocates nothing,
 * ever.
 *   Arguments, layouts, alignment and aliasing rules: as qm_matmul_q4_0.
 *   Limit: M <= 8 (the GEMV regime); M > 8 returns QM_ERR_TOO_LARGE.  The
 *   array holds 1 MB of partial sums and 4096 row-group counters; when a
 *   shape's split would not fit, the kernel splits K less (down to not at
 *   all), so every N and K within the other limits is accepted.
 *   Memory: every GPU that loads the library holds the array (about 1 MB)
 *   until the process exits.
 *   Set-up: the first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress) with that device current, and looks it up
 *   again when the device's current context has changed (after
 *   cudaDeviceReset); make that first call, and the first call after a reset,
 *   before any stream capture.
 *   Sharing: all calls use the same array, which keeps the last call's
 *   contents; a call clears the counters it needs before its kernel runs.
 *   Calls that overlap on the GPU (different streams, or concurrent graph
 *   launches) race on the array and may produce wrong results: order them.
 * Returns QM_OK or a negative status.
 */
QM_API int qm_matmul_q4_0_noalloc(const float* A, const void* wq, float* C, int64_t M,
                                  int64_t N, int64_t K, void* stream);

/*
 * qm_matmul_q4_0_q8act — the decode-regime product with the activations
 * quantized to Q8_0 first: C = A' x dequant(W)^T, A' = dequant_q8_0(
 * quantize_q8_0(A)) row by row (the GEMV fused with a preceding activation
 * quantization, the "act-quant fusion" item of "vulkan: shader and sequencing
 * efficiency backlog"; quantize_q8_0 with the readings of qm_quantize_q8_0).
 * A is read as f32 and quantized on chip; nothing but C is written.  Each
 * block of 32 then factors exactly into integers (d_a d_w (sum q qs - 8 sum
 * qs)), so the product runs on integer dot products, with one f32 rounding per
 * block; results agree with the exact product of A' and W to |error| <= 1e-5 *
 * sum_k |A'[m][k] * W[n][k]| + 1e-7, and infinities and NaN (a scale past
 * binary16's range) by class.  It is NOT the product with A: quantization
 * moves each activation by up to about half its block's step, max|x| / 254.
 *   A, wq, C, M, N, K, stream, alignment and aliasing: as qm_matmul_q4_0.
 *   M = 1..8 (M > 8 returns QM_ERR_TOO_LARGE); K % 256 == 0 with 16-byte
 *   aligned A and wq takes the staged kernel, other shapes a generic one.
 * Returns QM_OK or a negative status.
 */
QM_API int qm_matmul_q4_0_q8act(const float* A, const void* wq, float* C, int64_t M, int64_t N,
                                int64_t K, void* stream);

/*
 * qm_gemv_q4_0_list — a list of decode-regime products C_p = A_p x
 * dequant(W_p)^T (sections "qmatvec_q4_0" and "matmul_q4_0_tiled"; the
 * GEMV's cost is streaming the weight blocks once), all with the same M, in
 * one persistent launch where the shapes allow it: a decode step's chain of
 * projections without a fixed launch price per projection.
 *   problems : host array of `count` descriptors (read before the call
 *              returns).  Each problem follows the rules of qm_matmul_q4_0
 *              (operands, layouts, alignment, no output overlapping its own
 *              inputs).  wait_for is -1, or an index j below the problem's own:
 *              the problem's A is read only after problems 0..j have written
 *              their C (this is how a problem consumes an earlier one's
 *              output).  reserved must be 0.
 *   count    : >= 0.  M : >= 0, the rows of every A and C.
 *   counters : device memory of `count` uint32 (4-byte aligned, overlapping
 *              no operand) that the launch uses to count finished problems;
 *              it is cleared on `stream` before each launch that needs it.
 *              May be NULL: dependencies are then honoured by ending the
 *              launch before every problem that waits on one inside it.
 * Results are those of calling qm_matmul_q4_0 on the problems in list order.
 * Problems that neither wait on one another nor share memory may run in any
 * order; so no output may overlap another problem's weights, and an output
 * that overlaps another problem's activations or output (or whose
 * activations another problem's output overlaps) needs the later of the two
 * to wait for the earlier (QM_ERR_ALIAS otherwise).  The persistent kernel
 * takes M = 1, K % 2048 == 0, K <= 14336 and 16-byte aligned A and wq; other
 * problems run one by one through qm_matmul_q4_0's kernels, in list order on
 * the same stream.  Deterministic, like qm_matmul_q4_0.
 * Returns QM_OK or a negative status (nothing is enqueued when a check fails).
 */
typedef struct qm_gemv_problem {
    const float* A;   /* [M][K] f32, row-major                         */
    const void* wq;   /* [N][K/32] Q4_0 blocks                          */
    float* C;         /* [M][N] f32, row-major                          */
    int64_t N;
    int64_t K;
    int32_t wait_for; /* -1, or read A after problems 0..wait_for       */
    int32_t reserved; /* 0                                              */
} qm_gemv_problem;

QM_API int qm_gemv_q4_0_list(const qm_gemv_problem* problems, int64_t count, int64_t M,
                             uint32_t* counters, void* stream);

/*
 * qm_gemv_q4_0_q8act_list — qm_gemv_q4_0_list for the act-quant product of
 * qm_matmul_q4_0_q8act: every problem computes C_p = dequant_q8_0(
 * quantize_q8_0(A_p)) x dequant(W_p)^T, each activation vector quantized on
 * chip, in one persistent launch where the shapes allow it (M = 1, K % 2048
 * == 0, K <= 14336, 16-byte aligned A and wq); other problems run through
 * qm_matmul_q4_0_q8act in list order.  Arguments, ordering (wait_for,
 * counters), aliasing rules and errors: as qm_gemv_q4_0_list; M > 8 returns
 * QM_ERR_TOO_LARGE.  Precision: as qm_matmul_q4_0_q8act.
 */
QM_API int qm_gemv_q4_0_q8act_list(const qm_gemv_problem* problems, int64_t count, int64_t M,
                                   uint32_t* counters, void* stream);

/*
 * qm_gemm_plan — the work items the prefill GEMM on tensor cores
 * (QM_ALGO_GEMM_TC) takes for (M, N, K) on a device with sm_count SMs on
 * which fit2, fit4 and fit8 thread-block clusters of 2, 4 and 8 of its CTAs
 * can be resident at once.  Host only: touches no device and enqueues nothing;
 * meant for tests and tuning.
 *   out: 8 int64 values {tile width (112, 128 or 256), n-tiles, tiles, whole-tile
 *        items, s_rem K ranges of each later tile, 1 if the later tiles are
 *        split into 128-column halves instead, items (= CTAs), 1 if the K
 *        ranges add up through a cluster}.
 *   M, N >= 1, K a positive multiple of 256 (the shapes QM_ALGO_GEMM_TC takes).
 * Returns QM_OK, QM_ERR_NULL or QM_ERR_SHAPE.
 */
QM_API int qm_gemm_plan(int64_t M, int64_t N, int64_t K, int sm_count, int fit2, int fit4, int fit8,
                        int64_t* out);

/*
 * qm_gemv_plan — the launch plan the decode GEMV (QM_ALGO_GEMV, packed = 0;
 * QM_ALGO_GEMV_PK, packed = 1) takes for (M, N, K) on a device with sm_count
 * SMs and smem_optin bytes of opt-in shared memory per CTA.  With noalloc = 0
 * the plan of qm_matmul_q4_0, which adds a split K up through thread-block
 * clusters of 2, 4 or 8 CTAs, fit2, fit4 and fit8 of which can be resident
 * at once on that device; with noalloc = 1 the plan of
 * qm_matmul_q4_0_noalloc, whose split K meets in its fixed scratch array
 * (the fit counts are then ignored).  Host only: touches no device and
 * enqueues nothing; meant for tests and tuning.
 *   out: 13 int64 values {RG row groups, U units of 256 k, S K ranges, rps row
 *        groups per row block, c units per stage, hs warps per tile, rbpc row
 *        blocks per CTA, nu_max units in the largest K range, stages, grid
 *        CTAs, dynamic shared memory bytes, W consumer warps, 1 if the K
 *        ranges add up through a cluster}.
 *   M 1..8 (1..2 when packed), N >= 1, K a positive multiple of 256, fit
 *   counts >= 0.
 * Returns QM_OK, QM_ERR_NULL, QM_ERR_SHAPE, or QM_ERR_UNSUPPORTED when no
 * plan fits (the library then runs the generic GEMV).
 */
QM_API int qm_gemv_plan(int64_t M, int64_t N, int64_t K, int packed, int sm_count, int smem_optin,
                        int fit2, int fit4, int fit8, int noalloc, int64_t* out);

/*
 * qm_launch_count — the number of kernels this library has enqueued in this
 * process (all devices, all threads), for accounting in benchmarks.
 */
QM_API uint64_t qm_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* QM_H */
