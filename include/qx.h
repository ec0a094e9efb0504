/*
 * qx.h -- C ABI of the GB300 (sm_103a) block-quantised GEMV / GEMM library.
 *
 * The library computes the decode-time matrix-vector product of GGUF-style
 * block-quantised weight rows (Q4_K, Q6_K, Q8_0) with one activation vector,
 * in two methods (llamay docs, "Backends and hardware", section "Accelerate is
 * not bit-identical": dequantising the weights to float and quantising the
 * activation to int8 are two methods, not one method and its rounding error):
 *
 *   QX_MODE_F32  -- the weights are dequantised on the fly and dotted with an
 *                   f32 activation (llambda.lisp README, "Features &
 *                   Architecture": the f32 FMA GEMV over Q4_K_M / Q6_K).
 *   QX_MODE_W4A8 -- the activation is quantised to int8 once per matmul and
 *                   the weight rows are never materialised; per-block integer
 *                   dot products are scaled per block (llamay, "Backends and
 *                   hardware", section "CPU": the W4A8 fused dot product; and
 *                   section "CUDA": an integer dot for the W4A8 inner product).
 *
 * It also runs the same contraction at prefill batch sizes on the tensor
 * cores (llamay, section "CUDA": a tensor-core prefill kernel, whose missing
 * piece was staging the next weight tile behind the current multiply).
 *
 * Conventions shared by every entry point:
 *   - Weights are a row-major array of blocks; row r starts at byte
 *     r * qx_row_bytes(fmt, cols).  Block layouts are the GGUF ones:
 *       Q4_K 256 weights / 144 B: d f16, dmin f16, 12 B of packed 6-bit
 *            scales and mins, 128 B of 4-bit quants; w = d*sc*q - dmin*m.
 *       Q6_K 256 weights / 210 B: ql[128] (low 4 bits), qh[64] (high 2 bits),
 *            scales[16] int8 (one per 16 weights), d f16 last;
 *            w = d*sc*(q - 32).
 *       Q8_0 32 weights / 34 B: d f16, 32 int8 quants; w = d*q.
 *   - Every pointer named "device" is device memory owned by the caller.  The
 *     library keeps no per-call state.  Per device it holds: one cached
 *     device-property query, the device error word (below), and the
 *     QX_CHAIN_MAX_JOBS + 1 arrival counters of qx_gemv_chain_noalloc (file-
 *     scope device arrays, present on every GPU that loads the library).  No
 *     entry point of this header allocates device memory; the one allocation
 *     in the library is the short-lived buffer of the measurement hook
 *     qx_debug_mma_rate (qx_debug.h).
 *   - Calls are asynchronous on stream `s` (NULL = the legacy default stream)
 *     and run on the current device.  Argument, shape and alignment errors
 *     return before anything is launched or written; a failed launch returns
 *     QX_ERR_CUDA.
 *   - Alignment: W, the f32 activation x and the qx_act_q8 buffers must be
 *     16-byte aligned; the outputs y, Y and P 4-byte aligned.
 *   - Only compute capability 10.3 (GB300) is served.  Any other device is
 *     declined with QX_ERR_UNSUPPORTED_DEVICE rather than run through another
 *     kernel (llamay, section "CUDA": below its minimum capability the
 *     backend declines at open with a message naming the reason).
 *   - Kernels bound every wait.  A wait that runs out sets a device error
 *     word and the kernel returns; qx_device_check() reports it.
 */
#ifndef QX_H
#define QX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* qx_stream_t;

/* Format tags (the GGML type ids, a naming convention only), and
 * QX_Q6_K_SOA: Q6_K repacked at load time by qx_repack (see there). */
typedef enum { QX_Q8_0 = 8, QX_Q4_K = 12, QX_Q6_K = 14, QX_Q6_K_SOA = 142 } qx_fmt;

typedef enum { QX_MODE_F32 = 0, QX_MODE_W4A8 = 1, QX_MODE_W4A8_FUSED = 2 } qx_mode;

/*
 * Launch flag, OR'd into the mode argument of qx_gemv and qx_gemv_multi.
 * QX_FLAG_PDL: programmatic dependent launch.  The launch may start while the
 * previous kernel in the stream is still running: it begins streaming its
 * weights at once and reads x (and writes y) only after that kernel has
 * completed and its memory is visible.  The caller guarantees that the
 * previous kernel in the stream does not write W.
 */
#define QX_FLAG_PDL 0x100

/* Status codes.  0 is success; every error is negative. */
typedef int qx_status;
#define QX_OK 0
#define QX_ERR_ARG (-1)                /* null pointer, bad count, bad path       */
#define QX_ERR_FMT (-2)                /* unknown format                          */
#define QX_ERR_SHAPE (-3)              /* cols not whole blocks, size out of range */
#define QX_ERR_ALIGN (-4)              /* a pointer is not 16-byte aligned        */
#define QX_ERR_MODE (-5)               /* unknown mode, or mode/format mismatch   */
#define QX_ERR_CUDA (-6)               /* a CUDA runtime call or launch failed    */
#define QX_ERR_DEVICE_TIMEOUT (-7)     /* a kernel's bounded wait ran out         */
#define QX_ERR_UNSUPPORTED_DEVICE (-8) /* current device is not compute 10.3      */

/* Largest activation width served (columns per row). */
#define QX_MAX_COLS 32768
/* Largest number of matrices in one qx_gemv_multi call. */
#define QX_MAX_MULTI 8

/*
 * An int8-quantised activation, m rows of `cols` values, in caller-owned
 * device buffers (llamay, "Backends and hardware", section "CPU": the
 * activation is quantised to int8 once per matmul):
 *   q   [m, cols]      int8, row-major
 *   d   [m, cols/32]   f32 scale of each block of 32
 *   sum [m, cols/32]   int32 sum of the 32 quants of each block
 * The struct itself lives in host memory.
 */
typedef struct {
    int8_t* q;
    float* d;
    int32_t* sum;
    int64_t m;
    int64_t cols;
} qx_act_q8;

/*
 * Quantise x (device, f32 [m, cols] row-major) per block of 32:
 *   d = amax / 127 (f32, correctly rounded), q = round-half-even(x / d)
 *   (correctly rounded f32 quotient) clamped to [-127, 127], q = 0 when
 *   d == 0, sum = sum of q.
 * Writes out->q, out->d, out->sum (device buffers sized for m x cols) and
 * sets out->m = m, out->cols = cols.  cols must be a positive multiple of 32
 * (QX_ERR_SHAPE), m >= 1.  Non-finite inputs are not checked; their outputs
 * are unspecified.  The launch uses programmatic dependent launch: it may
 * start while the previous kernel in the stream drains, but reads x and
 * writes the outputs only after that kernel has completed (plain stream
 * order), so a following qx_gemv with QX_FLAG_PDL streams its weights early.
 */
qx_status qx_quantize_act_q8(const float* x, int64_t m, int64_t cols, qx_act_q8* out, qx_stream_t s);

/*
 * y[r] = sum_i w[r, i] * x[i] for r in [0, rows)  (device y, f32 [rows]).
 *   mode QX_MODE_F32 : x is `const float*`, device, f32 [cols]; y is within
 *                      1e-4 * sum_i |w[r, i] * x[i]| of the exact sum.  Q6_K
 *                      and QX_Q6_K_SOA rows of 2048 or 4096 columns, and
 *                      Q4_K rows of 256 to 4096 columns (except launches of
 *                      at most 192 KB per SM with QX_FLAG_PDL), run the
 *                      products on the tensor pipe: the quants exact in
 *                      bf16, x scaled per 256 columns by a power of two and
 *                      split into bf16 hi + lo, so each product carries at
 *                      most 2^-17 of its magnitude for every x within 2^-100
 *                      of its 256-column block's largest (Q4_K's min term
 *                      d_min m sum(x) is taken per 32 columns in f32); both
 *                      Q6_K layouts give bit-identical y.  The others
 *                      dequantise each quant to f32 and use one FMA per
 *                      weight.
 *   mode QX_MODE_W4A8: x is `const qx_act_q8*` (host struct) with m == 1 and
 *                      cols == cols, produced by qx_quantize_act_q8; y is the
 *                      per-block-scaled sum of exact integer partial sums.
 *   mode QX_MODE_W4A8_FUSED: x is `const float*`, device, f32 [cols]; the
 *                      launch quantises it itself with the arithmetic of
 *                      qx_quantize_act_q8 (identical int8 codes) and then
 *                      computes exactly what QX_MODE_W4A8 computes.
 * mode may carry QX_FLAG_PDL.
 * cols must be a positive multiple of the block width (256 for Q4_K/Q6_K,
 * 32 for Q8_0) and at most QX_MAX_COLS; rows >= 1.  The lanes cover rows of
 * up to 32768 columns for Q4_K / Q6_K in W4A8 mode, 24576 for Q4_K / Q6_K in
 * f32 mode, and 8192 for Q8_0; wider rows return QX_ERR_SHAPE.
 */
qx_status qx_gemv(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const void* x, float* y,
                  qx_mode mode, qx_stream_t s);

/*
 * n independent GEMVs over one activation in a single launch, e.g. the Q, K
 * and V projections, or gate and up: y[k] = W[k] . x for k in [0, n).  The
 * activation is read (and in QX_MODE_W4A8_FUSED quantised) once for all n
 * matrices: the pages quantise it to int8 once per matmul (llamay docs,
 * "Backends and hardware", section "CPU"), and matrices that share one input
 * are one matmul over their stacked rows, whose rows are independent
 * (llambda.lisp README, "Features & Architecture": the GEMV's outer loop runs
 * in parallel with isolated writes).
 * fmt, W, rows and y are host arrays of n entries; W[k] and y[k] are device
 * pointers.  All entries share cols, x and mode; 1 <= n <= QX_MAX_MULTI.
 * Entries of different formats are run as one launch per format.
 */
qx_status qx_gemv_multi(int n, const qx_fmt* fmt, const void* const* W, const int64_t* rows, int64_t cols,
                        const void* x, float* const* y, qx_mode mode, qx_stream_t s);

/*
 * Prefill: Y[m, r] = sum_i w[r, i] * x'[m, i] for every row m of the
 * quantised activation X (X->m rows, X->cols == cols), with Y device f32
 * [X->m, rows] row-major.  The rows of X are independent W4A8 GEMVs (colibri
 * GPU_BACKENDS.md, XDNA lane: C = A x B is row-independent, so padding the
 * batch to a tile is legitimate and padded rows are never written).
 */
qx_status qx_gemm_prefill(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* X, float* Y,
                          qx_stream_t s);

/*
 * qx_gemm_prefill with a forced path:
 *   0 = automatic (by measured time): path 1 for one row of X, path 4 for
 *       2 to 16 rows, path 3 above;
 *   1 = one W4A8 GEMV launch per row of X (bit-for-bit the qx_gemv result);
 *   2 = mma.sync tensor-core GEMM, Q4_K only (integer-valued f16 operands,
 *       exact per-sub-block integer sums, scales applied per sub-block);
 *   3 = tcgen05 tensor-core GEMM, every format: the W4A8 product is the dot
 *       product of the dequantised activation dx*q_x with the dequantised
 *       weight (llamay docs, "Backends and hardware", sections "CPU" and
 *       "CUDA"); both are formed inside the kernel, in shared memory, from
 *       the int8 codes and the raw weight blocks, each as two bf16 terms (hi
 *       + lo, 16 significant bits), and Y = Xh Wh^T + Xh Wl^T + Xl Wh^T is
 *       accumulated in f32 in tensor memory.  Each product's error is about
 *       2^-15 of its magnitude.  When the tiles (256 rows of X x 128 weight
 *       rows) leave a last wave over the SMs at most half full, that wave's
 *       tiles are split in two along K (a second launch, started beside the
 *       first by programmatic dependent launch; Y = the first half's sum plus
 *       the second's); when all the tiles fill at most half a wave, every
 *       tile is, and when they fill at most a quarter (K of 1024 columns or
 *       more; 512 for Q8_0) every tile is split in four (Y = (a0 + a1) +
 *       (a2 + a3)); so results depend on the shape and the GPU's SM count but
 *       not on the run.  No workspace: the call allocates nothing, may
 *       be captured in a CUDA graph on its first use and may run concurrently
 *       on several streams.  Shapes whose weights span 2 GiB or more (the
 *       copy engine's 32-bit coordinates) or more than 2^29 - 1 tiles
 *       return QX_ERR_SHAPE; path 0 takes path 1 for them.
 *   4 = small-batch GEMV (decode of several tokens at once: speculative or
 *       batched decode), every format, the weights streamed once per group
 *       of rows of X: groups of eight while five or more rows remain, then
 *       one of up to four.  Groups of five to eight rows against rows of up
 *       to 4096 columns in whole 256-column units whose bytes are a 16-byte
 *       multiple (Q4_K, Q8_0; Q6_K at 2048 and 4096 columns) run on the
 *       integer tensor path (mma.sync, the rows of X as the MMA's eight
 *       columns: exact integer partials per 32-column block, or per 16 for
 *       Q6_K, scaled in registers); the others on dp4a lanes, each holding
 *       its column slice of the group's codes and dotting every weight word
 *       with each row's (rows of up to 14336 columns, or 28672 for Q4_K /
 *       Q6_K when at most four rows of X remain; path 0 takes path 1 for
 *       wider rows).  Both: the same per-block integer dot products and
 *       scales as qx_gemv's W4A8 path, in a different f32 summation order
 *       (within the same tolerance, not bit-for-bit path 1).
 * A path that cannot serve the call returns QX_ERR_FMT rather than falling
 * back.
 */
qx_status qx_gemm_prefill_ex(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* X,
                             float* Y, int path, qx_stream_t s);

/*
 * The exact integer partial sums of the W4A8 product, written instead of y:
 * P[r, g] = sum over group g of q_w * q_x, with groups of 32 weights for Q4_K
 * (q_w the unsigned 4-bit quant) and Q8_0 (q_w the int8 quant), and groups of
 * 16 for Q6_K and QX_Q6_K_SOA (q_w = q - 32).  P is device int32
 * [rows, cols/32] or [rows, cols/16].  Computed by the same kernel code as qx_gemv's W4A8 path
 * (colibri GPU_BACKENDS.md: a numerics-matched integer GPU kernel).
 */
qx_status qx_gemv_partials(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* x,
                           int32_t* P, qx_stream_t s);

/*
 * A chain of dependent GEMVs in one launch.  Decode runs its GEMVs one after
 * another, each reading what an earlier one wrote (llamay docs, "Backends and
 * hardware": decode streams every weight once per token; VKNN wiki, "Running
 * an LLM on VKNN", section "Performance": the decode step is
 * weight-bandwidth-bound).  Separate launches pay a launch, a prologue and a
 * tail each; a chain streams the weights of job j + 1 while job j finishes.
 *
 * Job j computes y[k] = W[k] . x for its n entries (one format, shared cols
 * and x, like qx_gemv_multi) in W4A8 mode with the activation quantised
 * inside the launch (QX_MODE_W4A8_FUSED).  Job j + 1 reads its x only after
 * every write of job j has completed, so its x may be (part of) job j's y.
 */
#define QX_CHAIN_MAX_JOBS 128
#define QX_CHAIN_MAX_ENTRIES 4
typedef struct {
    qx_fmt fmt;
    int n;                                  /* entries, 1..QX_CHAIN_MAX_ENTRIES */
    const void* W[QX_CHAIN_MAX_ENTRIES];    /* device, 16-byte aligned          */
    int64_t rows[QX_CHAIN_MAX_ENTRIES];
    float* y[QX_CHAIN_MAX_ENTRIES];         /* device, f32 [rows], 4-byte aligned */
    int64_t cols;
    const float* x;                         /* device, f32 [cols], 16-byte aligned */
} qx_gemv_job;

/* Device scratch bytes a chain of n_jobs needs (arrival counters). */
size_t qx_gemv_chain_scratch_bytes(int n_jobs);

/*
 * Run jobs[0 .. n_jobs) in order as one cooperative launch (all CTAs
 * resident).  `scratch` is caller-owned device memory of at least
 * qx_gemv_chain_scratch_bytes(n_jobs) bytes, zero-filled before the first
 * call; a call that completes leaves it zero-filled again.  Calls that may
 * overlap on the GPU need separate scratch.  After QX_ERR_DEVICE_TIMEOUT the
 * scratch must be zero-filled again.  1 <= n_jobs <= QX_CHAIN_MAX_JOBS.
 */
qx_status qx_gemv_chain(int n_jobs, const qx_gemv_job* jobs, void* scratch, qx_stream_t s);

/*
 * qx_gemv_chain without caller scratch: for callers that cannot allocate
 * device memory where they run a chain -- code running during CUDA graph
 * capture, where cudaMalloc is not allowed; runtimes that only hand out
 * memory from a pool fixed at start-up; plug-ins that must not use the
 * process's allocator.  (The pages have no counterpart: this is a library
 * convenience, not part of the method.)
 *
 * Same jobs and results as qx_gemv_chain.  The arrival counters live in a
 * fixed array inside the library (QX_CHAIN_MAX_JOBS + 1 words on every GPU
 * that loads the library, held until the process exits); the call allocates
 * nothing, and clears the counters on stream s before each launch.
 *   - n_jobs above QX_CHAIN_MAX_JOBS (the array's capacity) returns
 *     QX_ERR_ARG before anything is launched.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture on the device.
 *   - Every call on a device shares the one array: calls that may overlap on
 *     the GPU (different streams without ordering) race and give wrong
 *     results.  Order them, or use qx_gemv_chain with separate scratch.
 */
qx_status qx_gemv_chain_noalloc(int n_jobs, const qx_gemv_job* jobs, qx_stream_t s);

/* Bytes of one row of `cols` weights, or 0 if fmt is unknown or cols is not
 * a positive multiple of the block width. */
size_t qx_row_bytes(qx_fmt fmt, int64_t cols);

/*
 * Load-time repack between the GGUF Q6_K layout and QX_Q6_K_SOA (llamay
 * docs, "Backends and hardware", section "Repacking is a per-device decision
 * now": block layouts are rewritten once, at load, for the device that runs
 * them).  A QX_Q6_K_SOA row of cols weights (nsb = cols / 256 super-blocks)
 * holds, for each super-block j, the 208 bytes ql[128], qh[64], scales[16]
 * of the GGUF block at bytes [208 j, 208 j + 208), then the nsb f16 d values
 * at byte 208 nsb, padded with zero bytes to a 16-byte multiple:
 * qx_row_bytes(QX_Q6_K_SOA, cols) = 208 nsb + 16 * ceil(2 nsb / 16) (the
 * GGUF row size when nsb is a multiple of 8).  Every field of every
 * super-block is then 16-byte aligned, which the GEMV lanes read with
 * vector loads; the values and the arithmetic are those of Q6_K, so
 * qx_gemv and qx_gemv_partials give the same bits on either layout.
 *   from, to: QX_Q6_K -> QX_Q6_K_SOA, or QX_Q6_K_SOA -> QX_Q6_K (the exact
 *             inverse: a round trip restores every byte).
 *   src, dst: device, rows * qx_row_bytes(from / to, cols) bytes, 16-byte
 *             aligned, not overlapping.
 * QX_Q6_K_SOA is served by qx_gemv, qx_gemv_multi, qx_gemv_partials and
 * prefill path 1 (and path 0, which then takes path 1); the other prefill
 * paths and qx_gemv_chain return QX_ERR_FMT for it.
 */
qx_status qx_repack(qx_fmt from, qx_fmt to, const void* src, int64_t rows, int64_t cols, void* dst,
                    qx_stream_t s);

/* Synchronise stream s, then read and clear the device error word of the
 * current device: QX_OK, QX_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran
 * out since the last check, or QX_ERR_CUDA if the synchronisation failed. */
qx_status qx_device_check(qx_stream_t s);

/* Static, NUL-terminated strings. */
const char* qx_status_string(qx_status st);
/* The CUDA call and error text behind the most recent QX_ERR_CUDA returned
 * on the calling thread ("" if none); valid until the next call on it. */
const char* qx_last_error(void);
const char* qx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QX_H */
