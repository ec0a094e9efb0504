// qx_gemv.cu -- batch-1 GEMV over GGUF-style block-quantised rows (Q4_K,
// Q6_K, Q8_0) for sm_103a, in f32 mode and W4A8 mode.
//
// Decode is weight-bandwidth-bound (VKNN wiki, "Running an LLM on VKNN",
// section "Performance": one token streams every weight once and the wide
// lm_head is the largest single op), so the kernel is a weight stream:
//
//   * Each CTA owns a contiguous range of rows (rows are independent:
//     llambda.lisp README, "Features & Architecture", the GEMV's outer loop
//     runs in parallel with isolated, lock-free writes).  Its rows are
//     contiguous bytes, streamed in stages of G whole rows by 1-D bulk copies
//     (TMA) into a ring of shared-memory slots, issued by one producer warp
//     and completed on mbarriers.  G is a multiple of the number of rows
//     whose bytes make a 16-byte multiple, so every copy is 16-byte aligned.
//   * Consumer lanes own a fixed slice of columns for the whole kernel, so
//     the activation slice stays in registers.  A "team" of lanes covers one
//     row; teams take the rows of a stage in turn.  Each lane stores its
//     partial sum of a row to shared memory and moves on; a reducer warp adds
//     the partials of each row in a fixed lane order and writes y, so no
//     consumer ever waits on a cross-lane reduction.
//   * W4A8 (llamay docs, "Backends and hardware", sections "CPU" and
//     "CUDA"): per 32-weight sub-block (16 for Q6_K) the int8 x int4/int6/int8
//     products are summed exactly with dp4a, and only then scaled; the weight
//     rows are never materialised.
//   * f32 mode (llambda.lisp README, "Features & Architecture"): every quant
//     is converted exactly to f32 and fused-multiply-added with the f32
//     activation; the per-sub-block scale d*sc (and the Q4_K min term
//     dmin*m*sum(x)) is applied once per sub-block, which is the same sum
//     reassociated.
#include "qx_device.cuh"
#include "qx_internal.h"
#include "qx_lanes.cuh"
#include "qx_stage.cuh"

namespace qx {

namespace {

using namespace lanes;


// ----------------------------------------------------------------------------
// Work distribution (the row split and the stage walk: qx_stage.cuh)
// ----------------------------------------------------------------------------

// W4A8 kernels and Q8_0 kernels fit two CTAs per SM (<= 112 registers), so
// that with programmatic dependent launch the next GEMV's CTA can be resident
// next to this one and stream its weights while this one finishes.
template <int FMT, int MODE, bool MERGED>
constexpr int gemv_min_blocks() {
    return (MODE == QX_MODE_W4A8 || FMT == QX_Q8_0 || MERGED) ? 2 : 1;
}

// FUSED: W4A8 with the activation quantised in-kernel (p.xf set).
template <int FMT, int MODE, bool PART, bool MERGED, bool FUSED>
__global__ void __launch_bounds__(gemv_threads(FMT, MODE, PART, MERGED), gemv_min_blocks<FMT, MODE, MERGED>())
    gemv_kernel(const __grid_constant__ GemvParams p) {
    using LaneT = Lane<FMT, MODE>;
    constexpr int NW = gemv_consumer_warps(FMT, MODE, MERGED);
    constexpr bool kMerged = MERGED;
    static_assert(!MERGED || gemv_has_merged(FMT, MODE, PART), "no merged variant of this kernel");
    static_assert(!FUSED || (MODE == QX_MODE_W4A8 && !PART), "in-kernel quantisation is a W4A8 y-output variant");
    // Warps that may quantise an f32 activation in-kernel: all of them -- the
    // producer and the reducer have nothing else to do until the consumers
    // finish their first stage, which needs the quantised activation.  They
    // join only when that takes fewer rounds of two-lane block tasks than the
    // consumers alone (each round waits on its loads: the 14336-column
    // activation of a Llama-3.1-8B down projection, 4 rounds -> 3); a merged
    // producer/reducer warp always joins.  The Q4_K and Q8_0 kernels are
    // built without helpers: the extra code slowed their one-round launches
    // measurably (GB300, Llama-3.1-8B q/k/v launch 5.24 -> 5.30 us).
    constexpr int QW = NW + 1 + ((!PART && !kMerged) ? 1 : 0);
    constexpr bool kMayHelp = kMerged || FMT == QX_Q6_K || FMT == QX_Q6_K_SOA;
    const int ntask = static_cast<int>(2 * (p.cols / 32));
    const bool helpers =
        kMerged || (kMayHelp && (ntask + NW * 32 - 1) / (NW * 32) > (ntask + QW * 32 - 1) / (QW * 32));
    const int qthreads = helpers ? QW * 32 : NW * 32;  // threads that quantise (and sync around it)
    // Rounds of quantisation whose loads are in flight together: one (the
    // Llama-3.1-8B down projection's three rounds took 4.5 us one after the
    // other and 6.9 us with all loads in flight, GB300).
    constexpr int kQuantBatch = 1;
    static_assert(PART || LaneT::kRows == gemv_rows_per_call(FMT, MODE), "row count must match the host geometry");
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = p.stages;
    // full[s]: the slot's bytes have landed.  empty[s]: the consumers (and,
    // with a separate reducer warp, the reducer) are done with the slot and
    // its partials.  part[s] (y outputs): the consumers' partials of the
    // slot's rows are stored, and they are done with its bytes.
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + S;
    uint64_t* part = empty + S;
    float* red = reinterpret_cast<float*>(smem + p.red_off);  // [S][G][RS]; first the quantised activation

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = cta_row_begin(p, blockIdx.x), r1 = cta_row_begin(p, blockIdx.x + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], (PART || kMerged) ? NW : NW + 1);
            mbar_init(&part[s], NW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    // A producer or reducer warp's share of the in-kernel quantisation (W4A8
    // with an f32 activation), with the consumers' two barriers around it:
    // the codes are complete / every consumer holds its slice (see below).
    const auto quantise_share = [&]() {
        int8_t* sq = reinterpret_cast<int8_t*>(smem + p.act_off);
        float* sd = reinterpret_cast<float*>(sq + p.cols);
        int32_t* ss = reinterpret_cast<int32_t*>(sd + p.cols / 32);
        const int nblk = static_cast<int>(p.cols / 32);
        pdl_wait_prior_grid();  // the activation may come from the previous kernel
        quantize_all<kQuantBatch>(p.xf, nblk, threadIdx.x, qthreads, sq, sd, ss, FMT != QX_Q8_0);
        quantiser_barrier(qthreads);
        quantiser_barrier(qthreads);
    };

    if (warp == NW) {
        // ---------------- producer (and, merged, reducer) ---------------------
        // Lane 0 issues every bulk copy.  Weights are never written by the
        // preceding kernel, so the first p.prewait stages are fetched before
        // the programmatic dependency on it is resolved.  Then lane 0 refills
        // each slot once `empty` says its previous stage is done with -- or,
        // when this warp is also the reducer, right after the warp has reduced
        // that stage (the reducer is a slot's last user: the consumers are
        // done with its bytes once their partials are stored).
        const uint64_t policy = policy_evict_first();
        StageWalker wk{r0, r1, 0};
        int issued = 0;
        unsigned tail_slots = 0;  // slots whose bytes were last written by plain stores
        // Copies the next stage into its slot; false once the CTA's rows are exhausted.
        const auto issue_next = [&]() -> bool {
            int e, nrows;
            int64_t lrow;
            if (!wk.next(p, e, lrow, nrows)) return false;
            const int k = issued, slot = k % S;
            const uint8_t* src = p.e[e].W + lrow * p.row_bytes;
            const uint32_t bytes = static_cast<uint32_t>(int64_t(nrows) * p.row_bytes);
            const uint32_t abytes = bytes & ~15u;
            uint8_t* dst = smem + size_t(slot) * p.slot_bytes;
            if (bytes != abytes) {
                // The last < 16 bytes of a matrix whose size is not a 16-byte multiple.
                for (uint32_t t = abytes; t < bytes; ++t) dst[t] = src[t];
                tail_slots |= 1u << slot;
            } else if (tail_slots & (1u << slot)) {
                fence_proxy_async_smem();
                tail_slots &= ~(1u << slot);
            }
            mbar_arrive_expect_tx(&full[slot], abytes);
            if (abytes) bulk_g2s_evict_first(dst, src, abytes, &full[slot], policy);
            issued = k + 1;
            return true;
        };
        const auto issue_first_stages = [&]() {
            for (int k = 0; k < S; ++k) {
                if (k == p.prewait) pdl_wait_prior_grid();
                if (!issue_next()) break;
            }
        };
        // Keep the CTA alive until every copy it issued has landed (bounded;
        // on the normal path each wait returns at once or shortly).
        const auto drain = [&]() {
            for (int k = issued > S ? issued - S : 0; k < issued; ++k)
                mbar_wait_bounded(&full[k % S], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
        };
        // With a cap of p.inflight < S stages in flight, stage k is issued only
        // once stage k - p.inflight has landed.  Its slot is not reused before
        // stage k - p.inflight + S > k, so the phase parity below is that
        // stage's.  Fewer bytes queued in the memory system keep the latency
        // of every other load (activation, parameters) low.
        const auto landed_before = [&](int k) -> bool {
            if (p.inflight <= 0 || p.inflight >= S || k < p.inflight) return true;
            const int j = k - p.inflight;
            return mbar_wait_bounded(&full[j % S], (j / S) & 1, p.wait_ns, p.err, kErrTimeoutFull);
        };
        if constexpr (!kMerged) {
            const bool helps = FUSED && helpers;
            if (!helps) {
                if (lane != 0) return;
                int e, nrows;
                int64_t lrow;
                StageWalker pw{r0, r1, 0};
                for (int k = 0; pw.next(p, e, lrow, nrows); ++k) {
                    const int slot = k % S;
                    if (k == p.prewait) pdl_wait_prior_grid();
                    if (k >= S &&
                        !mbar_wait_bounded(&empty[slot], ((k / S) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                        break;
                    if (!landed_before(k)) break;
                    const uint8_t* src = p.e[e].W + lrow * p.row_bytes;
                    const uint32_t bytes = static_cast<uint32_t>(int64_t(nrows) * p.row_bytes);
                    const uint32_t abytes = bytes & ~15u;
                    uint8_t* dst = smem + size_t(slot) * p.slot_bytes;
                    if (bytes != abytes) {
                        for (uint32_t t = abytes; t < bytes; ++t) dst[t] = src[t];
                        tail_slots |= 1u << slot;
                    } else if (tail_slots & (1u << slot)) {
                        fence_proxy_async_smem();
                        tail_slots &= ~(1u << slot);
                    }
                    mbar_arrive_expect_tx(&full[slot], abytes);
                    if (abytes) bulk_g2s_evict_first(dst, src, abytes, &full[slot], policy);
                    issued = k + 1;
                }
                drain();
                return;
            }
            int e = 0, nrows = 0;
            int64_t lrow = 0;
            StageWalker pw{r0, r1, 0};
            const auto issue_stage = [&](int k) {
                const int slot = k % S;
                const uint8_t* src = p.e[e].W + lrow * p.row_bytes;
                const uint32_t bytes = static_cast<uint32_t>(int64_t(nrows) * p.row_bytes);
                const uint32_t abytes = bytes & ~15u;
                uint8_t* dst = smem + size_t(slot) * p.slot_bytes;
                if (bytes != abytes) {
                    for (uint32_t t = abytes; t < bytes; ++t) dst[t] = src[t];
                    tail_slots |= 1u << slot;
                } else if (tail_slots & (1u << slot)) {
                    fence_proxy_async_smem();
                    tail_slots &= ~(1u << slot);
                }
                mbar_arrive_expect_tx(&full[slot], abytes);
                if (abytes) bulk_g2s_evict_first(dst, src, abytes, &full[slot], policy);
                issued = k + 1;
            };
            // the first S stages (no slot to wait for), then the quantisation
            // share, then every later stage once its slot is released
            // (no more stages than may be in flight before the quantisation:
            // this warp takes part in it)
            int k = 0;
            bool more = true;
            const int first = (p.inflight > 0 && p.inflight < S) ? p.inflight : S;
            if (lane == 0) {
                for (; k < first && (more = pw.next(p, e, lrow, nrows)); ++k) {
                    if (k == p.prewait) pdl_wait_prior_grid();
                    issue_stage(k);
                }
            }
            __syncwarp();
            quantise_share();
            if (lane != 0) return;
            if (more) {
                for (; pw.next(p, e, lrow, nrows); ++k) {
                    if (k == p.prewait) pdl_wait_prior_grid();
                    if (k >= S &&
                        !mbar_wait_bounded(&empty[k % S], ((k / S) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                        break;
                    if (!landed_before(k)) break;
                    issue_stage(k);
                }
            }
            drain();
        } else {
            if (lane == 0) issue_first_stages();
            // The other lanes wait here for lane 0, and below for each refill,
            // so that the warp never sits in two different waits at once.
            __syncwarp();
            if constexpr (FUSED) quantise_share();
            else pdl_wait_prior_grid();  // y may be read by the previous kernel (a small launch fetches
                                         // its whole ring before this wait in issue_first_stages)
            StageWalker rw{r0, r1, 0};
            int e, nrows;
            int64_t lrow;
            for (int k = 0; rw.next(p, e, lrow, nrows); ++k) {
                const int slot = k % S;
                const bool landed = mbar_wait_bounded(&part[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull);
                if (!__all_sync(0xffffffffu, landed)) break;  // the whole warp leaves together
                reduce_stage(red + size_t(slot) * p.G * p.RS, p.RS, p.L, nrows, p.e[e].y + lrow, lane);
                __syncwarp();
                if (lane == 0) issue_next();
                __syncwarp();
            }
            if (lane == 0) drain();
        }
        return;
    }

    if constexpr (!PART && !kMerged) {
        if (warp == NW + 1) {
            // ---------------- reducer: row sums of every stage, in order -----
            if (FUSED && helpers) quantise_share();
            StageWalker wk{r0, r1, 0};
            int e, nrows;
            int64_t lrow;
            for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
                const int slot = k % S;
                if (!mbar_wait_bounded(&part[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
                reduce_stage(red + size_t(slot) * p.G * p.RS, p.RS, p.L, nrows, p.e[e].y + lrow, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            return;
        }
    }

    // ---------------- consumers ----------------------------------------------
    const Team tm = make_team(warp, lane, p.team_lanes, p.team_warps, p.nteams, p.L);

    LaneT X;
    const int8_t* q = p.xq;
    const float* d = p.xd;
    const int32_t* s = p.xs;
    pdl_wait_prior_grid();  // the activation may come from the previous kernel
    if constexpr (FUSED) {
        {
            // Quantise the f32 activation once per CTA into shared memory,
            // with the same code as qx_quantize_act_q8; two adjacent lanes
            // per block of 32; all consumer lanes (and a merged
            // producer/reducer warp) take part.
            int8_t* sq = reinterpret_cast<int8_t*>(smem + p.act_off);
            float* sd = reinterpret_cast<float*>(sq + p.cols);
            int32_t* ss = reinterpret_cast<int32_t*>(sd + p.cols / 32);
            const int nblk = static_cast<int>(p.cols / 32);
            quantize_all<kQuantBatch>(p.xf, nblk, threadIdx.x, qthreads, sq, sd, ss, FMT != QX_Q8_0);
            quantiser_barrier(qthreads);
            q = sq;
            d = sd;
            s = ss;
        }
    }
    // the quantised activation in shared memory has its 128-byte slices permuted
    if (tm.active) load_slice<MODE>(X, q, d, s, p.x, tm.slice, FMT != QX_Q8_0 && FUSED);
    if constexpr (FMT == QX_Q6_K_SOA) X.geometry(p.cols);
    if constexpr (MODE == QX_MODE_W4A8) {
        // the quantised activation shares its area with the partial sums
        if constexpr (FUSED) quantiser_barrier(qthreads);
    }

    const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
    const int64_t ng = p.cols / ((FMT == QX_Q6_K || FMT == QX_Q6_K_SOA) ? 16 : 32);
    StageWalker wk{r0, r1, 0};
    int e, nrows;
    int64_t lrow;
    for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
        const int slot = k % S;
        if (!mbar_wait_bounded(&full[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
        const uint8_t* sbuf = smem + size_t(slot) * p.slot_bytes;
        consume_stage<FMT, MODE, PART>(X, tm, sbuf, nrows, rb, red + size_t(slot) * p.G * p.RS, p.RS,
                                       PART ? p.e[e].P + lrow * ng : nullptr, ng);
        __syncwarp();
        if (lane == 0) {
            if constexpr (!PART) mbar_arrive(&part[slot]);
            if constexpr (!kMerged) mbar_arrive(&empty[slot]);
        }
    }
}

// ----------------------------------------------------------------------------
// Small-batch GEMV: Y[m, r] for MB (four or eight) rows of a quantised
// activation X (qx_gemm_prefill path 4).  The same weight stream as
// gemv_kernel (contiguous rows per CTA, bulk copies into a shared-memory
// ring, a producer lane, a reducer warp), read once for all rows of X:
// decode of several tokens at once (speculative or batched decode) is then
// still bound by the weight bytes, not by one stream per token.  One CTA per
// SM, 14 consumer warps.
// ----------------------------------------------------------------------------
template <int FMT, int MB>
__global__ void __launch_bounds__(kBatchThreads, 1) gemv_batch_kernel(const __grid_constant__ GemvParams p) {
    constexpr int NW = kBatchConsumerWarps;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + S;
    uint64_t* part = empty + S;
    float* red = reinterpret_cast<float*>(smem + p.red_off);  // [S][G * MB][RS]
    const size_t red_stage = size_t(p.G) * MB * p.RS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = cta_row_begin(p, blockIdx.x), r1 = cta_row_begin(p, blockIdx.x + 1);
    if (threadIdx.x == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(&full[k], 1);
            mbar_init(&empty[k], NW + 1);
            mbar_init(&part[k], NW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == NW) {
        // ---------------- producer: lane 0 issues every bulk copy -----------
        if (lane != 0) return;
        const uint64_t policy = policy_evict_first();
        unsigned tail_slots = 0;
        StageWalker pw{r0, r1, 0};
        int e, nrows, issued = 0;
        int64_t lrow;
        for (int k = 0; pw.next(p, e, lrow, nrows); ++k) {
            const int slot = k % S;
            if (k >= S && !mbar_wait_bounded(&empty[slot], ((k / S) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                break;
            const uint8_t* src = p.e[e].W + lrow * p.row_bytes;
            const uint32_t bytes = static_cast<uint32_t>(int64_t(nrows) * p.row_bytes);
            const uint32_t abytes = bytes & ~15u;
            uint8_t* dst = smem + size_t(slot) * p.slot_bytes;
            if (bytes != abytes) {
                // the last < 16 bytes of a matrix whose size is not a 16-byte multiple
                for (uint32_t t = abytes; t < bytes; ++t) dst[t] = src[t];
                tail_slots |= 1u << slot;
            } else if (tail_slots & (1u << slot)) {
                fence_proxy_async_smem();
                tail_slots &= ~(1u << slot);
            }
            mbar_arrive_expect_tx(&full[slot], abytes);
            if (abytes) bulk_g2s_evict_first(dst, src, abytes, &full[slot], policy);
            issued = k + 1;
        }
        for (int k = issued > S ? issued - S : 0; k < issued; ++k)
            mbar_wait_bounded(&full[k % S], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
        return;
    }
    if (warp == NW + 1) {
        // ---------------- reducer: (row, activation row) sums, in order -----
        pdl_wait_prior_grid();  // y may be read by the previous kernel
        StageWalker wk{r0, r1, 0};
        int e, nrows;
        int64_t lrow;
        for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
            const int slot = k % S;
            if (!mbar_wait_bounded(&part[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
            reduce_stage_batch<MB>(red + slot * red_stage, p.RS, p.L, nrows, p.e[e].y + lrow, p.y_stride,
                                   p.m_valid, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        return;
    }

    // ---------------- consumers ----------------------------------------------
    const Team tm = make_team(warp, lane, p.team_lanes, p.team_warps, p.nteams, p.L);
    pdl_wait_prior_grid();  // X may come from the previous kernel
    BatchLane<FMT, MB> X;
    if (tm.active) X.load(p.xq, p.xd, p.xs, p.cols, p.m_valid, tm.slice);
    const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
    StageWalker wk{r0, r1, 0};
    int e, nrows;
    int64_t lrow;
    for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
        const int slot = k % S;
        if (!mbar_wait_bounded(&full[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
        consume_stage_batch<FMT, MB>(X, tm, smem + size_t(slot) * p.slot_bytes, nrows, rb, red + slot * red_stage,
                                     p.RS);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&part[slot]);
            mbar_arrive(&empty[slot]);
        }
    }
}

// ----------------------------------------------------------------------------
// Small-batch Q4_K GEMV on the integer tensor path (mma.sync m16n8k32, u8
// weight quants x s8 activation codes, s32 partials): Y[m, r] for up to eight
// rows of a quantised activation X.  The eight rows of X are the MMA's N = 8
// columns, sixteen weight rows its M rows and one 32-column sub-block its K,
// so one MMA yields the integer partial P of 16 x 8 (weight row, row of X)
// pairs for one sub-block, and the scales apply in registers:
//     y[m, r] += d sc_j dx[m, j] P - dmin m_j dx[m, j] S[m, j]
// (the W4A8 sum of the batch-1 lanes, term by term).  The low nibbles of a
// weight word are one mask; the high nibbles enter as 16 q (a mask, no
// shift) and their scale carries the 1/16.  (The f16 form -- 1024 + q as an
// f16, two m16n8k16 MMAs per sub-block -- keeps the tensor pipe idler but
// needs more integer work per weight and measured slower.)
//
// Same weight stream as gemv_batch_kernel (a CTA's contiguous rows, a ring
// of stages, a producer warp, a reducer warp), but each stage is 16 P rows
// copied one row at a time to a padded stride (rows row_bytes + 16 apart,
// so that the eight row groups of a fragment load fall on different banks).
// Consumer warp w owns super-block w % nsb of row group w / nsb of every
// stage (nsb = cols / 256 <= 16, P = 16 / nsb groups a stage), so its slice
// of X (the MMA's B fragments) stays in registers for the whole launch.
// Each warp writes its 16 x 8 partial of a stage to shared memory; the
// reducer adds the nsb partials of each group and writes Y for the valid
// rows of X.
// ----------------------------------------------------------------------------
constexpr int kMmaBatchWarps = 16;

__device__ __forceinline__ void mma_s8s8_k32(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}
// m16n8k16: A rows gid, gid + 8 (one register each), B one register.
__device__ __forceinline__ void mma_u8s8_k16(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm("mma.sync.aligned.m16n8k16.row.col.s32.u8.s8.s32 {%0, %1, %2, %3}, {%4, %5}, {%6}, {%7, %7, %7, %7};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "r"(0));
}

__device__ __forceinline__ void mma_u8s8_k32(int (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.u8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(0));
}

// The 6-bit scales and mins of a Q4_K super-block header (d, dmin, 12 bytes)
// as bytes: sc of sub-blocks 0-3 and 4-7, m of 0-3 and 4-7.
struct Q4kSubScales {
    uint32_t sc[2], m[2];
    float d, nd, d16, nd16, dmin, ndmin;  // d, -2^23 d, d / 16, -2^23 d / 16, dmin, -2^23 dmin
    __device__ __forceinline__ explicit Q4kSubScales(const uint4 h) {
        sc[0] = h.y & 0x3F3F3F3Fu;
        m[0] = h.z & 0x3F3F3F3Fu;
        sc[1] = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        m[1] = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
        d = f16_bits_to_f32(h.x & 0xFFFFu);
        dmin = f16_bits_to_f32(h.x >> 16);
        d16 = d * 0.0625f;
        nd = d * -8388608.0f;
        nd16 = d16 * -8388608.0f;
        ndmin = dmin * -8388608.0f;
    }
    // a_j = d sc_j (/ 16 for odd j: the high nibbles enter as 16 q) and
    // b_j = dmin m_j, exact (an f16 times a 6-bit integer): byte -> 2^23 +
    // byte, then one FMA.
    __device__ __forceinline__ void ab(int j, float& a, float& b) const {
        const float fs = __int_as_float(__byte_perm(sc[j >> 2], 0x4B000000u, 0x7650u + uint32_t(j & 3)));
        const float fm = __int_as_float(__byte_perm(m[j >> 2], 0x4B000000u, 0x7650u + uint32_t(j & 3)));
        a = (j & 1) ? fmaf(d16, fs, nd16) : fmaf(d, fs, nd);
        b = fmaf(dmin, fm, ndmin);
    }
};

// One 256-column unit of a row (a Q4_K or Q6_K super-block, eight Q8_0
// blocks) against the warp's slice of X: rows gid and gid + 8 of the unit's
// 16-row group (ra, rb: their unit bases in shared memory), rows 2 t and
// 2 t + 1 of X; adds y[row][row of X] into ya2 (row gid) and yb2 (row gid + 8).
// bx: the unit's B fragments; act: its scale-table entries (see the kernel).
template <int FMT>
struct BatchMmaUnit;

// Q4_K: eight sub-blocks of 32, one m16n8k32 each (u8 quants: low nibbles as
// q, high nibbles as 16 q); table entry per sub-block (dx, dx, dx S, dx S).
template <>
struct BatchMmaUnit<QX_Q4_K> {
    static constexpr int kBytes = 144, kB = 16, kActPerUnit = 8;
    __device__ __forceinline__ static void load_b(const int8_t* xr, int t, bool live, uint32_t (&bx)[kB]) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int u = 0; u < 2; ++u)
                bx[2 * j + u] = live ? __ldg(reinterpret_cast<const uint32_t*>(xr + 32 * j + 16 * u + 4 * t)) : 0u;
    }
    __device__ __forceinline__ static void run(const uint8_t* ra, const uint8_t* rb, int t, const uint32_t (&bx)[kB],
                                               const float4* act, uint64_t& ya2, uint64_t& yb2) {
        const Q4kSubScales sa(*reinterpret_cast<const uint4*>(ra)), sbs(*reinterpret_cast<const uint4*>(rb));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t w[2][2];  // [half][row gid, gid + 8]: bytes 4 t .. 4 t + 3 of the half
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int o = 16 + 32 * c + 16 * u + 4 * t;
                w[u][0] = *reinterpret_cast<const uint32_t*>(ra + o);
                w[u][1] = *reinterpret_cast<const uint32_t*>(rb + o);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // sub-block 2 c (low nibbles), 2 c + 1 (high nibbles, as 16 q)
                const int j = 2 * c + h;
                // the partials P (16 P for high nibbles): rows gid, gid + 8 x rows 2 t, 2 t + 1 of X
                const uint32_t mask = h ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
                const uint32_t a[4] = {w[0][0] & mask, w[0][1] & mask, w[1][0] & mask, w[1][1] & mask};
                int d[4];
                mma_u8s8_k32(d, a, bx[2 * j], bx[2 * j + 1]);
                float aa, ba, ab, bb;
                sa.ab(j, aa, ba);
                sbs.ab(j, ab, bb);
                const float4 xv = act[4 * j];  // dx, dx, dx S, dx S of rows 2 t, 2 t + 1 of X
                const uint64_t dx2 = f32x2_pack(xv.x, xv.y), ds2 = f32x2_pack(xv.z, xv.w);
                ya2 = f32x2_fma(f32x2_pack(aa, aa), f32x2_mul(f32x2_pack(float(d[0]), float(d[1])), dx2), ya2);
                ya2 = f32x2_fma(f32x2_pack(-ba, -ba), ds2, ya2);
                yb2 = f32x2_fma(f32x2_pack(ab, ab), f32x2_mul(f32x2_pack(float(d[2]), float(d[3])), dx2), yb2);
                yb2 = f32x2_fma(f32x2_pack(-bb, -bb), ds2, yb2);
            }
        }
    }
};

// Q8_0: eight blocks of 34 bytes (d, 32 int8), one m16n8k32 each (s8 weights
// as stored, read at 2-byte-aligned offsets); table entry per block (dx, dx, -, -).
template <>
struct BatchMmaUnit<QX_Q8_0> {
    static constexpr int kBytes = 272, kB = 16, kActPerUnit = 8;
    __device__ __forceinline__ static void load_b(const int8_t* xr, int t, bool live, uint32_t (&bx)[kB]) {
        BatchMmaUnit<QX_Q4_K>::load_b(xr, t, live, bx);
    }
    __device__ __forceinline__ static void run(const uint8_t* ra, const uint8_t* rb, int t, const uint32_t (&bx)[kB],
                                               const float4* act, uint64_t& ya2, uint64_t& yb2) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint8_t* ba = ra + 34 * j;
            const uint8_t* bb = rb + 34 * j;
            const uint32_t a[4] = {lds_u32_a2(ba + 2 + 4 * t), lds_u32_a2(bb + 2 + 4 * t), lds_u32_a2(ba + 18 + 4 * t),
                                   lds_u32_a2(bb + 18 + 4 * t)};
            int d[4];
            mma_s8s8_k32(d, a, bx[2 * j], bx[2 * j + 1]);
            const float da = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(ba));
            const float db = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bb));
            const float4 xv = act[4 * j];
            const uint64_t dx2 = f32x2_pack(xv.x, xv.y);
            ya2 = f32x2_fma(f32x2_pack(da, da), f32x2_mul(f32x2_pack(float(d[0]), float(d[1])), dx2), ya2);
            yb2 = f32x2_fma(f32x2_pack(db, db), f32x2_mul(f32x2_pack(float(d[2]), float(d[3])), dx2), yb2);
        }
    }
};

// Q6_K (ql[128], qh[64], scales[16] int8, d): sixteen groups of 16 with their
// own scales, one m16n8k16 each (u8 q = 0..63; P = D - 32 S16, exact).  The
// two groups of one 32-column block share dx, so their partials are combined
// in integers first: sc_a (D_a - 32 S_a) + sc_b (D_b - 32 S_b) (|.| < 2^25).
// Table entry per group (dx, dx, S16, S16) with S16 the group's sum of codes
// (as integers in float bits).
template <>
struct BatchMmaUnit<QX_Q6_K> {
    static constexpr int kBytes = 210, kB = 16, kActPerUnit = 16;
    __device__ __forceinline__ static void load_b(const int8_t* xr, int t, bool live, uint32_t (&bx)[kB]) {
#pragma unroll
        for (int g = 0; g < 16; ++g)
            bx[g] = live ? __ldg(reinterpret_cast<const uint32_t*>(xr + 16 * g + 4 * t)) : 0u;
    }
    __device__ __forceinline__ static void run(const uint8_t* ra, const uint8_t* rb, int t, const uint32_t (&bx)[kB],
                                               const float4* act, uint64_t& ya2, uint64_t& yb2) {
        const float da = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(ra + 208));
        const float db = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rb + 208));
        const int8_t* sca = reinterpret_cast<const int8_t*>(ra + 192);
        const int8_t* scb = reinterpret_cast<const int8_t*>(rb + 192);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // words of elements 128 h + 32 tq + 16 u + 4 t .. + 3: ql for quarters 0 / 2 and 1 / 3, qh
            uint32_t ql[2][2][2], qh[2][2];  // [u][quarter parity][row], [u][row]
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int o = 16 * u + 4 * t;
#pragma unroll
                for (int qp = 0; qp < 2; ++qp) {
                    ql[u][qp][0] = lds_u32_a2(ra + 64 * h + 32 * qp + o);
                    ql[u][qp][1] = lds_u32_a2(rb + 64 * h + 32 * qp + o);
                }
                qh[u][0] = lds_u32_a2(ra + 128 + 32 * h + o);
                qh[u][1] = lds_u32_a2(rb + 128 + 32 * h + o);
            }
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {  // the 32-column block 4 h + tq: groups 8 h + 2 tq + u
                int p[4] = {0, 0, 0, 0};  // sum over its two groups of sc (D - 32 S16)
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int g = 8 * h + 2 * tq + u;
                    uint32_t a[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        a[r] = ((ql[u][tq & 1][r] >> (4 * (tq >> 1))) & 0x0F0F0F0Fu) |
                               (((qh[u][r] >> (2 * tq)) & 0x03030303u) << 4);
                    int d[4];
                    mma_u8s8_k16(d, a[0], a[1], bx[g]);
                    const float4 xv = act[4 * g];
                    const int s0 = __float_as_int(xv.z), s1 = __float_as_int(xv.w);
                    const int ka = sca[g], kb = scb[g];
                    p[0] += ka * (d[0] - 32 * s0);
                    p[1] += ka * (d[1] - 32 * s1);
                    p[2] += kb * (d[2] - 32 * s0);
                    p[3] += kb * (d[3] - 32 * s1);
                }
                const float4 xv = act[4 * (8 * h + 2 * tq)];
                const uint64_t dx2 = f32x2_pack(xv.x, xv.y);
                ya2 = f32x2_fma(f32x2_pack(da, da), f32x2_mul(f32x2_pack(float(p[0]), float(p[1])), dx2), ya2);
                yb2 = f32x2_fma(f32x2_pack(db, db), f32x2_mul(f32x2_pack(float(p[2]), float(p[3])), dx2), yb2);
            }
        }
    }
};

template <int FMT>
__global__ void __launch_bounds__(kMmaBatchThreads, 1) gemv_batch_mma_kernel(const __grid_constant__ GemvParams p) {
    using U = BatchMmaUnit<FMT>;
    constexpr int NW = kMmaBatchWarps;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + S;
    uint64_t* part = empty + S;
    const int nsb = static_cast<int>(p.cols / 256), P = NW / nsb;  // groups of 16 rows per stage
    float* red = reinterpret_cast<float*>(smem + p.red_off);          // [S][P][nsb][16 rows x 8]
    const int red_stage = P * nsb * 128;
    const int rstride = static_cast<int>(p.row_bytes) + 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = cta_row_begin(p, blockIdx.x), r1 = cta_row_begin(p, blockIdx.x + 1);
    if (threadIdx.x == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(&full[k], 1);
            mbar_init(&empty[k], NW + 1);
            mbar_init(&part[k], NW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == NW) {
        // ---------------- producer: one bulk copy per row, lanes in parallel -
        const uint64_t policy = policy_evict_first();
        const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
        StageWalker pw{r0, r1, 0};
        int e, nrows, issued = 0;
        int64_t lrow;
        for (int k = 0; pw.next(p, e, lrow, nrows); ++k) {
            const int slot = k % S;
            if (k >= S && !warp_wait_all(&empty[slot], ((k / S) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty)) break;
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], uint32_t(nrows) * rb);
            __syncwarp();
            uint8_t* dst = smem + size_t(slot) * p.slot_bytes;
            const uint8_t* src = p.e[e].W + lrow * p.row_bytes;
            for (int r = lane; r < nrows; r += 32)
                bulk_g2s_evict_first(dst + r * rstride, src + int64_t(r) * rb, rb, &full[slot], policy);
            issued = k + 1;
        }
        if (lane == 0)
            for (int k = issued > S ? issued - S : 0; k < issued; ++k)
                mbar_wait_bounded(&full[k % S], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
        return;
    }
    if (warp == NW + 1) {
        // ---------------- reducer: the nsb partials of each (row, row of X) --
        pdl_wait_prior_grid();  // y may be read by the previous kernel
        StageWalker wk{r0, r1, 0};
        int e, nrows;
        int64_t lrow;
        const int n = lane & 7;
        for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
            const int slot = k % S;
            if (!mbar_wait_bounded(&part[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
            const float* rs = red + size_t(slot) * red_stage;
            for (int gi = 0; gi < P && 16 * gi < nrows; ++gi) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const int rr = (lane >> 3) + 4 * kk, row = 16 * gi + rr;
                    float acc = 0.0f;
                    for (int sb = 0; sb < nsb; ++sb) acc += rs[(gi * nsb + sb) * 128 + rr * 8 + n];
                    if (n < p.m_valid && row < nrows) p.e[e].y[int64_t(n) * p.y_stride + lrow + row] = acc;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        return;
    }

    // ---------------- consumers ----------------------------------------------
    pdl_wait_prior_grid();  // X may come from the previous kernel
    const int sb = warp % nsb, gsub = warp / nsb;
    const bool active = gsub < P;
    const int gid = lane >> 2, t = lane & 3;
    const int nblk = static_cast<int>(p.cols / 32);
    // B fragments: X row gid, the warp's unit (in flight while the table below is filled)
    uint32_t bx[U::kB];
    U::load_b(p.xq + int64_t(gid) * p.cols + 256 * sb, t, active && gid < p.m_valid, bx);
    // Scales of X, per 32-column block (Q6_K: per 16-column group) q and
    // rows 2 t', 2 t' + 1 of X: act[q][t'] = (dx, dx, dx S, dx S) (Q6_K: the
    // group's code sums S16 as integers in the last two), zeros for rows past
    // m_valid; the consumer warps fill it once.
    float4* act = reinterpret_cast<float4*>(smem + p.act_off);
    const int nact = nblk * (U::kActPerUnit / 8);
    for (int i = threadIdx.x; i < nact * 4; i += NW * 32) {
        const int q = i >> 2, tt = i & 3;
        float v[4];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int n = 2 * tt + u;
            const bool ln = n < p.m_valid;
            if constexpr (FMT == QX_Q6_K) {
                const int64_t bi = int64_t(n) * nblk + (q >> 1);
                v[u] = ln ? __ldg(p.xd + bi) : 0.0f;
                int s16 = 0;
                if (ln) {
                    const uint4 c = __ldg(reinterpret_cast<const uint4*>(p.xq + int64_t(n) * p.cols + 16 * q));
                    s16 = __dp4a(int(c.x), 0x01010101, s16);
                    s16 = __dp4a(int(c.y), 0x01010101, s16);
                    s16 = __dp4a(int(c.z), 0x01010101, s16);
                    s16 = __dp4a(int(c.w), 0x01010101, s16);
                }
                v[2 + u] = __int_as_float(s16);
            } else {
                const int64_t bi = int64_t(n) * nblk + q;
                const float dx = ln ? __ldg(p.xd + bi) : 0.0f;
                v[u] = dx;
                v[2 + u] = (FMT == QX_Q4_K && ln) ? dx * float(__ldg(p.xs + bi)) : 0.0f;
            }
        }
        act[i] = make_float4(v[0], v[1], v[2], v[3]);
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NW * 32) : "memory");  // the consumer warps: the table is filled
    const float4* my_act = act + (U::kActPerUnit * sb) * 4 + t;  // entry q of the unit: my_act[4 q]
    StageWalker wk{r0, r1, 0};
    int e, nrows;
    int64_t lrow;
    for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
        const int slot = k % S;
        if (!mbar_wait_bounded(&full[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
        if (active && 16 * gsub < nrows) {
            const uint8_t* ra = smem + size_t(slot) * p.slot_bytes + (16 * gsub + gid) * rstride + U::kBytes * sb;
            uint64_t ya2 = f32x2_pack(0.0f, 0.0f), yb2 = ya2;  // rows gid, gid + 8; rows 2 t, 2 t + 1 of X
            U::run(ra, ra + 8 * rstride, t, bx, my_act, ya2, yb2);
            const float2 ya = f32x2_unpack(ya2), yb = f32x2_unpack(yb2);
            float* rs = red + size_t(slot) * red_stage + (gsub * nsb + sb) * 128;
            *reinterpret_cast<float2*>(rs + gid * 8 + 2 * t) = ya;
            *reinterpret_cast<float2*>(rs + (gid + 8) * 8 + 2 * t) = yb;
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&part[slot]);
            mbar_arrive(&empty[slot]);
        }
    }
}

// Largest shared memory (static + dynamic) a CTA may use on sm_103a.
constexpr int kMaxDynamicSmem = 227 * 1024;

// Raise the kernel's dynamic shared-memory limit to the maximum, once per
// kernel and device.  Occupancy and launches then depend only on the bytes
// each launch asks for.
template <int FMT, int MODE, bool PART, bool MERGED, bool FUSED>
cudaError_t configure_once() {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, gemv_kernel<FMT, MODE, PART, MERGED, FUSED>);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(gemv_kernel<FMT, MODE, PART, MERGED, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMaxDynamicSmem - static_cast<int>(fa.sharedSizeBytes));
    if (err == cudaSuccess) done[dev] = true;
    return err;
}

template <int FMT, int MODE, bool PART, bool MERGED, bool FUSED>
cudaError_t launch_one(const GemvParams& p, size_t smem, cudaStream_t s, bool pdl) {
    cudaError_t err = configure_once<FMT, MODE, PART, MERGED, FUSED>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_cta);
    cfg.blockDim = dim3(gemv_threads(FMT, MODE, PART, MERGED));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, MODE, PART, MERGED, FUSED>, p);
}

template <int FMT, int MODE, bool PART, bool MERGED, bool FUSED>
cudaError_t occupancy_one(size_t smem, int* out) {
    cudaError_t err = configure_once<FMT, MODE, PART, MERGED, FUSED>();
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, gemv_kernel<FMT, MODE, PART, MERGED, FUSED>,
                                                         gemv_threads(FMT, MODE, PART, MERGED), smem);
}

template <int FMT, int MB>
cudaError_t launch_batch_one(const GemvParams& p, size_t smem, cudaStream_t s) {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
        cudaFuncAttributes fa;
        if ((err = cudaFuncGetAttributes(&fa, gemv_batch_kernel<FMT, MB>)) != cudaSuccess) return err;
        err = cudaFuncSetAttribute(gemv_batch_kernel<FMT, MB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxDynamicSmem - static_cast<int>(fa.sharedSizeBytes));
        if (err != cudaSuccess) return err;
        done[dev] = true;
    }
    gemv_batch_kernel<FMT, MB><<<p.n_cta, kBatchThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_batch_mma_one(const GemvParams& p, size_t smem, cudaStream_t s) {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
        cudaFuncAttributes fa;
        if ((err = cudaFuncGetAttributes(&fa, gemv_batch_mma_kernel<FMT>)) != cudaSuccess) return err;
        err = cudaFuncSetAttribute(gemv_batch_mma_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxDynamicSmem - static_cast<int>(fa.sharedSizeBytes));
        if (err != cudaSuccess) return err;
        done[dev] = true;
    }
    gemv_batch_mma_kernel<FMT><<<p.n_cta, kMmaBatchThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_batch_mma(int fmt, const GemvParams& p, size_t smem, cudaStream_t s) {
    switch (fmt) {
        case QX_Q4_K: return launch_batch_mma_one<QX_Q4_K>(p, smem, s);
        case QX_Q6_K: return launch_batch_mma_one<QX_Q6_K>(p, smem, s);
        case QX_Q8_0: return launch_batch_mma_one<QX_Q8_0>(p, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv_batch(int fmt, const GemvParams& p, size_t smem, cudaStream_t s) {
    const bool wide = p.mb == kBatchRowsWide;
    if (!wide && p.mb != kBatchRows) return cudaErrorInvalidValue;
    switch (fmt) {
        case QX_Q4_K: return wide ? launch_batch_one<QX_Q4_K, kBatchRowsWide>(p, smem, s)
                                  : launch_batch_one<QX_Q4_K, kBatchRows>(p, smem, s);
        case QX_Q6_K: return wide ? launch_batch_one<QX_Q6_K, kBatchRowsWide>(p, smem, s)
                                  : launch_batch_one<QX_Q6_K, kBatchRows>(p, smem, s);
        case QX_Q8_0: return wide ? launch_batch_one<QX_Q8_0, kBatchRowsWide>(p, smem, s)
                                  : launch_batch_one<QX_Q8_0, kBatchRows>(p, smem, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv(int fmt, int mode, bool partials, const GemvParams& p, size_t smem, cudaStream_t s,
                        bool pdl) {
    const bool fused = p.xf != nullptr;
    if (fused && (mode != QX_MODE_W4A8 || partials)) return cudaErrorInvalidValue;
    if (p.merged) {
        if (fmt == QX_Q6_K && mode == QX_MODE_W4A8 && !partials)
            return fused ? launch_one<QX_Q6_K, QX_MODE_W4A8, false, true, true>(p, smem, s, pdl)
                         : launch_one<QX_Q6_K, QX_MODE_W4A8, false, true, false>(p, smem, s, pdl);
        if (fmt == QX_Q6_K_SOA && mode == QX_MODE_W4A8 && !partials)
            return fused ? launch_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, true, true>(p, smem, s, pdl)
                         : launch_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, true, false>(p, smem, s, pdl);
        if (mode == QX_MODE_F32 && !partials && !fused) {
            if (fmt == QX_Q4_K) return launch_one<QX_Q4_K, QX_MODE_F32, false, true, false>(p, smem, s, pdl);
            if (fmt == QX_Q6_K) return launch_one<QX_Q6_K, QX_MODE_F32, false, true, false>(p, smem, s, pdl);
            if (fmt == QX_Q6_K_SOA) return launch_one<QX_Q6_K_SOA, QX_MODE_F32, false, true, false>(p, smem, s, pdl);
        }
        return cudaErrorInvalidValue;
    }
    switch (fmt * 8 + mode * 4 + (partials ? 2 : 0) + (fused ? 1 : 0)) {
        case QX_Q4_K * 8 + 0: return launch_one<QX_Q4_K, QX_MODE_F32, false, false, false>(p, smem, s, pdl);
        case QX_Q4_K * 8 + 4: return launch_one<QX_Q4_K, QX_MODE_W4A8, false, false, false>(p, smem, s, pdl);
        case QX_Q4_K * 8 + 5: return launch_one<QX_Q4_K, QX_MODE_W4A8, false, false, true>(p, smem, s, pdl);
        case QX_Q4_K * 8 + 6: return launch_one<QX_Q4_K, QX_MODE_W4A8, true, false, false>(p, smem, s, pdl);
        case QX_Q6_K * 8 + 0: return launch_one<QX_Q6_K, QX_MODE_F32, false, false, false>(p, smem, s, pdl);
        case QX_Q6_K * 8 + 4: return launch_one<QX_Q6_K, QX_MODE_W4A8, false, false, false>(p, smem, s, pdl);
        case QX_Q6_K * 8 + 5: return launch_one<QX_Q6_K, QX_MODE_W4A8, false, false, true>(p, smem, s, pdl);
        case QX_Q6_K * 8 + 6: return launch_one<QX_Q6_K, QX_MODE_W4A8, true, false, false>(p, smem, s, pdl);
        case QX_Q8_0 * 8 + 0: return launch_one<QX_Q8_0, QX_MODE_F32, false, false, false>(p, smem, s, pdl);
        case QX_Q8_0 * 8 + 4: return launch_one<QX_Q8_0, QX_MODE_W4A8, false, false, false>(p, smem, s, pdl);
        case QX_Q8_0 * 8 + 5: return launch_one<QX_Q8_0, QX_MODE_W4A8, false, false, true>(p, smem, s, pdl);
        case QX_Q8_0 * 8 + 6: return launch_one<QX_Q8_0, QX_MODE_W4A8, true, false, false>(p, smem, s, pdl);
        case QX_Q6_K_SOA * 8 + 0: return launch_one<QX_Q6_K_SOA, QX_MODE_F32, false, false, false>(p, smem, s, pdl);
        case QX_Q6_K_SOA * 8 + 4: return launch_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, false, false>(p, smem, s, pdl);
        case QX_Q6_K_SOA * 8 + 5: return launch_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, false, true>(p, smem, s, pdl);
        case QX_Q6_K_SOA * 8 + 6: return launch_one<QX_Q6_K_SOA, QX_MODE_W4A8, true, false, false>(p, smem, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t gemv_max_ctas_per_sm(int fmt, int mode, bool partials, bool merged, bool fused, size_t smem, int* out) {
    if (fused && (mode != QX_MODE_W4A8 || partials)) return cudaErrorInvalidValue;
    if (merged) {
        if (fmt == QX_Q6_K && mode == QX_MODE_W4A8 && !partials)
            return fused ? occupancy_one<QX_Q6_K, QX_MODE_W4A8, false, true, true>(smem, out)
                         : occupancy_one<QX_Q6_K, QX_MODE_W4A8, false, true, false>(smem, out);
        if (fmt == QX_Q6_K_SOA && mode == QX_MODE_W4A8 && !partials)
            return fused ? occupancy_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, true, true>(smem, out)
                         : occupancy_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, true, false>(smem, out);
        if (mode == QX_MODE_F32 && !partials && !fused) {
            if (fmt == QX_Q4_K) return occupancy_one<QX_Q4_K, QX_MODE_F32, false, true, false>(smem, out);
            if (fmt == QX_Q6_K) return occupancy_one<QX_Q6_K, QX_MODE_F32, false, true, false>(smem, out);
            if (fmt == QX_Q6_K_SOA) return occupancy_one<QX_Q6_K_SOA, QX_MODE_F32, false, true, false>(smem, out);
        }
        return cudaErrorInvalidValue;
    }
    switch (fmt * 8 + mode * 4 + (partials ? 2 : 0) + (fused ? 1 : 0)) {
        case QX_Q4_K * 8 + 0: return occupancy_one<QX_Q4_K, QX_MODE_F32, false, false, false>(smem, out);
        case QX_Q4_K * 8 + 4: return occupancy_one<QX_Q4_K, QX_MODE_W4A8, false, false, false>(smem, out);
        case QX_Q4_K * 8 + 5: return occupancy_one<QX_Q4_K, QX_MODE_W4A8, false, false, true>(smem, out);
        case QX_Q4_K * 8 + 6: return occupancy_one<QX_Q4_K, QX_MODE_W4A8, true, false, false>(smem, out);
        case QX_Q6_K * 8 + 0: return occupancy_one<QX_Q6_K, QX_MODE_F32, false, false, false>(smem, out);
        case QX_Q6_K * 8 + 4: return occupancy_one<QX_Q6_K, QX_MODE_W4A8, false, false, false>(smem, out);
        case QX_Q6_K * 8 + 5: return occupancy_one<QX_Q6_K, QX_MODE_W4A8, false, false, true>(smem, out);
        case QX_Q6_K * 8 + 6: return occupancy_one<QX_Q6_K, QX_MODE_W4A8, true, false, false>(smem, out);
        case QX_Q8_0 * 8 + 0: return occupancy_one<QX_Q8_0, QX_MODE_F32, false, false, false>(smem, out);
        case QX_Q8_0 * 8 + 4: return occupancy_one<QX_Q8_0, QX_MODE_W4A8, false, false, false>(smem, out);
        case QX_Q8_0 * 8 + 5: return occupancy_one<QX_Q8_0, QX_MODE_W4A8, false, false, true>(smem, out);
        case QX_Q8_0 * 8 + 6: return occupancy_one<QX_Q8_0, QX_MODE_W4A8, true, false, false>(smem, out);
        case QX_Q6_K_SOA * 8 + 0: return occupancy_one<QX_Q6_K_SOA, QX_MODE_F32, false, false, false>(smem, out);
        case QX_Q6_K_SOA * 8 + 4: return occupancy_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, false, false>(smem, out);
        case QX_Q6_K_SOA * 8 + 5: return occupancy_one<QX_Q6_K_SOA, QX_MODE_W4A8, false, false, true>(smem, out);
        case QX_Q6_K_SOA * 8 + 6: return occupancy_one<QX_Q6_K_SOA, QX_MODE_W4A8, true, false, false>(smem, out);
        default: return cudaErrorInvalidValue;
    }
}

// ----------------------------------------------------------------------------
// Bounded-wait probe: one warp waits on an mbarrier that nothing completes.
// ----------------------------------------------------------------------------
__global__ void timeout_probe_kernel(unsigned* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    mbar_wait_bounded(&bar, 0, limit_ns, err, kErrTimeoutProbe);
}

cudaError_t launch_timeout_probe(unsigned* err, uint64_t limit_ns, cudaStream_t s) {
    timeout_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace qx
