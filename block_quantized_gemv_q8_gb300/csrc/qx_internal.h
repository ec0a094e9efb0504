// qx_internal.h -- launch descriptors shared by the C-ABI layer (qx_api.cu)
// and the kernel translation units.  Host and device code; no CUDA types in
// the public header depend on it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qx.h"

namespace qx {

// Warps of a GEMV CTA: the consumers, then a producer warp whose lane 0
// issues the bulk copies, then (y outputs) a reducer warp that sums the
// consumers' per-lane partials of each row and writes y.  An SM partition
// holds 16K registers, so a kernel with up to 16 warps per SM (4 per
// partition) gets 128 registers a thread, one with 17 to 20 warps 96.  The
// f32-mode K-quant kernels run one CTA per SM with 12 consumer warps, the
// others two per SM with 8.
//
// The merged variant (Q6_K W4A8 with y outputs; taken for long launches, see
// gemv_geometry): 7 consumer warps and one warp that both produces and
// reduces, 16 warps per SM and so 128 registers (the standard Q6_K W4A8
// kernel is held to 96 and spills); rows of 14336 columns are then exactly
// two teams of 112 lanes.
// The f32-mode K-quant kernels have a merged variant too, for small launches
// under programmatic dependent launch: 8 warps of at most 128 registers, so
// that the next launch's CTA fits on the SM beside it (the standard f32
// kernel's 14 warps of 128 registers leave no room).
__host__ __device__ constexpr bool gemv_has_merged(int fmt, int mode, bool partials) {
    return !partials && ((mode == QX_MODE_W4A8 && (fmt == QX_Q6_K || fmt == QX_Q6_K_SOA)) ||
                         (mode == QX_MODE_F32 && fmt != QX_Q8_0));
}
__host__ __device__ constexpr int gemv_consumer_warps(int fmt, int mode, bool merged) {
    return merged ? 7 : ((mode == QX_MODE_F32 && fmt != QX_Q8_0) ? 12 : 8);
}
// Integer partials need no reducer warp; the merged variant has none either.
__host__ __device__ constexpr int gemv_threads(int fmt, int mode, bool partials, bool merged) {
    return 32 * (gemv_consumer_warps(fmt, mode, merged) + ((partials || merged) ? 1 : 2));
}
// Consumer warps per chain CTA (one CTA per SM), plus a producer and a reducer.
constexpr int kChainConsumerWarps = 10;
constexpr int kChainThreads = 32 * (kChainConsumerWarps + 2);
// Bytes read past the end of a shared-memory slot by the unaligned-word loads.
constexpr int kSlotPad = 16;

struct GemvEntry {
    const uint8_t* W;  // device, rows * row_bytes
    float* y;          // device, [rows]      (y output)
    int32_t* P;        // device, [rows, ng]  (partials output)
    int64_t rows;
    int64_t row0;      // first row of this entry in the concatenated row space
};

struct GemvParams {
    GemvEntry e[QX_MAX_MULTI];
    int n_entries;
    int64_t total_rows;
    int64_t cols;
    int64_t row_bytes;
    int quantum;      // rows per 16-byte-aligned row group
    int G;            // rows per pipeline stage
    int stages;       // pipeline depth (shared-memory slots)
    int slot_bytes;   // bytes per slot, including kSlotPad
    int team_lanes;   // lanes per team: a power of two <= 32, or L (teams packed across warps)
    int team_warps;   // 1 for sub-warp teams, else the warps a team touches (> 1)
    int nteams;       // teams per CTA
    int L;            // lanes with work per row (cols / columns-per-lane)
    int RS;           // floats per row of the per-lane partial-sum area
    int n_cta;
    int prewait;       // stages the producer issues before waiting on the preceding kernel
    int inflight;      // most stages in flight (issued, not landed) per CTA; 0: up to `stages`
    int merged;        // 1: the merged producer/reducer variant (gemv_has_merged)
    const float* x;    // f32 mode activation [cols]
    const int8_t* xq;  // W4A8 activation quants [cols]
    const float* xd;   // W4A8 activation scales [cols/32]
    const int32_t* xs; // W4A8 activation block sums [cols/32]
    const float* xf;   // W4A8 with in-kernel quantisation: f32 activation [cols]
    int bar_off;       // shared-memory byte offsets: mbarriers (full, empty, part),
    int red_off;       //   per-lane partial sums [stages][G][RS],
    int act_off;       //   quantised activation (in-kernel quantisation; the same
                       //   area as the partial sums, used before them)
    unsigned* err;     // device error word
    uint64_t wait_ns;  // bound on every wait
    // Batched launches (gemv_batch_kernel): rows m of a quantised activation
    // X, y[m * y_stride + r] for m < m_valid; the lanes hold mb rows (rows
    // m_valid .. mb - 1 repeat row m_valid - 1, unwritten).
    int mb;
    int m_valid;
    int64_t y_stride;
    // Row-group kernels (gemv_f32_mma_kernel): 16-row groups each consumer
    // warp takes per stage (the stage holds 16 P gq rows).
    int gq;
};

// Small-batch GEMV (one weight stream for several activation rows): rows of
// X per launch (four, or eight for 5..8 remaining rows), consumer warps (one
// CTA per SM: 16 warps of <= 128 registers), and columns per lane (64 for
// the K-quants with four rows, 32 otherwise, so that the rows' activation
// slices fit in registers).
constexpr int kBatchRows = 4;
constexpr int kBatchRowsWide = 8;
constexpr int kBatchConsumerWarps = 14;
constexpr int kBatchThreads = 32 * (kBatchConsumerWarps + 2);
__host__ __device__ constexpr int batch_cols_per_lane(int fmt, int mb) {
    return (fmt == QX_Q8_0 || mb > kBatchRows) ? 32 : 64;
}
// Small-batch GEMV on the integer tensor path (gemv_batch_mma_kernel): up to
// eight rows of X per launch, rows of at most 16 units of 256 columns (4096
// columns); 16 consumer warps, a producer and a reducer.
constexpr int kMmaBatchRows = 8;
constexpr int kMmaBatchMaxSuperBlocks = 16;
constexpr int kMmaBatchThreads = 32 * (16 + 2);
// f32-mode GEMV of Q6_K rows on the tensor pipe (gemv_f32_mma_kernel): the
// same geometry, rows of 2048 or 4096 columns.
constexpr int kF32MmaThreads = 32 * (16 + 2);

// Columns owned by one lane, per (format, mode).
__host__ __device__ constexpr int gemv_cols_per_lane(int fmt, int mode) {
    return fmt == QX_Q8_0 ? 32 : (mode == QX_MODE_W4A8 ? 128 : 64);
}

// A chain of dependent W4A8 GEMVs in one launch (qx_gemv_chain).
struct ChainEntry {
    const uint8_t* W;  // device, rows * row_bytes
    float* y;          // device, [rows]
    int64_t rows;
    int64_t row0;      // first row of this entry in the job's concatenated row space
};
struct alignas(16) ChainJob {
    ChainEntry e[QX_CHAIN_MAX_ENTRIES];
    const float* x;                      // f32 activation [cols], quantised in-kernel
    int64_t cols;
    int64_t row_bytes;
    int64_t total_rows;
    int fmt, n_entries, team_lanes, team_warps, nteams, quantum, G, L, RS;
};
static_assert(sizeof(ChainJob) % 16 == 0, "job descriptors are copied to shared memory in 16-byte words");

struct ChainParams {
    int n_jobs;
    int n_cta;
    int stages;
    int slot_bytes;
    int bar_off, red_off, act_off;
    int jobs_off;        // shared-memory copy of job[0 .. n_jobs), made once at kernel start
    int ranges_off;      // shared memory: this CTA's row range of every job (2 x int64 per job)
    int red_slot_floats; // floats of the partial-sum area per slot (most G * RS of any job)
    int64_t max_cols;    // widest activation (size of the quantised-activation area)
    unsigned* counters;  // caller scratch: [n_jobs + 1] arrival counters, zero on entry and exit
    unsigned* err;
    uint64_t wait_ns;
    int inflight;        // most stages in flight (issued, not landed); 0: up to `stages`
    ChainJob job[QX_CHAIN_MAX_JOBS];
};

// Row stride (floats) of the per-lane partial sums of a row of L lanes: a
// multiple of 4 (16-byte rows) with an odd number of 16-byte groups, so that
// the reducer's lanes (one row each) read distinct banks.
__host__ __device__ constexpr int partial_stride(int L) {
    return ((L + 3) / 4 % 2 == 1) ? (L + 3) / 4 * 4 : (L + 3) / 4 * 4 + 4;
}

// Rows a team computes per call, per (format, mode) (must match the kernels).
__host__ __device__ constexpr int gemv_rows_per_call(int fmt, int mode) {
    return fmt == QX_Q8_0 ? 2 : 1;
}

// Launchers (defined in the kernel translation units).
cudaError_t launch_actq8(const float* x, int64_t nblocks, int8_t* q, float* d, int32_t* sum, int sm_count,
                         cudaStream_t s);
cudaError_t launch_gemv(int fmt, int mode, bool partials, const GemvParams& p, size_t smem, cudaStream_t s,
                        bool pdl);
cudaError_t gemv_max_ctas_per_sm(int fmt, int mode, bool partials, bool merged, bool fused, size_t smem, int* out);
cudaError_t launch_gemv_batch(int fmt, const GemvParams& p, size_t smem, cudaStream_t s);
cudaError_t launch_gemv_batch_mma(int fmt, const GemvParams& p, size_t smem, cudaStream_t s);
cudaError_t launch_gemv_f32_mma(int fmt, const GemvParams& p, size_t smem, cudaStream_t s, bool pdl);
// Q6_K <-> QX_Q6_K_SOA (qx_repack.cu); row bytes of each side.
cudaError_t launch_repack_q6k(bool to_soa, const uint8_t* src, int64_t rows, int64_t nsb, int64_t src_row_bytes,
                              uint8_t* dst, int64_t dst_row_bytes, cudaStream_t s);
cudaError_t launch_timeout_probe(unsigned* err, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_chain(const ChainParams& p, size_t smem, cudaStream_t s);
cudaError_t launch_prefill_q4k(const uint8_t* W, int64_t N, int64_t K, const int8_t* xq, const float* xd,
                               const int32_t* xs, int64_t M, float* Y, cudaStream_t s);
cudaError_t chain_max_ctas_per_sm(size_t smem, int* out);
// Measurement builds (QX_TRACE): copy the chain kernel's timestamps to host.
cudaError_t chain_trace_read(void* host, size_t bytes);
// tcgen05 prefill (qx_tc.cu): both operands converted in shared memory, no
// workspace.  prefill_tc_serves: whether the kernel's 32-bit copy coordinates
// cover the shape.
bool prefill_tc_serves(int fmt, int64_t N, int64_t K, int64_t M, int64_t row_bytes);
cudaError_t launch_prefill_tc(int fmt, const uint8_t* W, int64_t N, int64_t K, int64_t row_bytes, const int8_t* xq,
                              const float* xd, int64_t M, float* Y, unsigned* err, int sm_count, cudaStream_t s);

}  // namespace qx
