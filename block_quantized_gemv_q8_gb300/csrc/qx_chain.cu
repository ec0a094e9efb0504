// qx_chain.cu -- a chain of dependent W4A8 GEMVs in one persistent launch.
//
// Decode runs its GEMVs one after another, each on the output of the
// previous step (llamay docs, "Backends and hardware": decode streams every
// weight once per token; VKNN wiki, "Running an LLM on VKNN", section
// "Performance": the decode step is weight-bandwidth-bound).  Launching each
// GEMV separately pays a launch, a prologue and a tail every time.  Here one
// cooperative launch (all CTAs resident) runs the whole chain:
//   * the producer warp of every CTA streams its rows of job 0, job 1, ...
//     into the shared-memory ring without pause -- weights never depend on
//     earlier jobs;
//   * the consumers store per-lane partial sums; the reducer warp of the CTA
//     adds them per row, writes y and, after the CTA's last row of job j,
//     counts the CTA on job j's arrival counter (caller scratch memory);
//   * the consumers of job j + 1 first wait until every CTA has finished job
//     j (that counter, bounded wait), then quantise job j + 1's activation
//     (which may be job j's output), load their slices and consume the
//     stages already in the ring.
// The ring keeps filling while the consumers wait, so the stream continues
// across job boundaries.  The last reducer to finish resets the counters to
// zero for the next call.
#include "qx_device.cuh"
#include "qx_internal.h"
#include "qx_lanes.cuh"

namespace qx {

namespace {

using namespace lanes;
constexpr int NW = kChainConsumerWarps;

#ifdef QX_TRACE
// Measurement builds only: %globaltimer stamps per (CTA, job, event).
constexpr int kTraceCtas = 160, kTraceEvents = 12;
__device__ unsigned long long g_trace[kTraceCtas * QX_CHAIN_MAX_JOBS * kTraceEvents];
__device__ __forceinline__ void stamp(int j, int ev) {
    if (blockIdx.x < kTraceCtas) g_trace[(blockIdx.x * QX_CHAIN_MAX_JOBS + j) * kTraceEvents + ev] = global_timer_ns();
}
#else
__device__ __forceinline__ void stamp(int, int) {}
#endif

// First row of CTA i in a job: an even split rounded down within its entry
// to a multiple of the alignment quantum (as in the single-launch kernel).
__device__ __forceinline__ int64_t job_row_begin(const ChainJob& j, int n_cta, int i) {
    if (i >= n_cta) return j.total_rows;
    const int64_t raw = j.total_rows * int64_t(i) / n_cta;
    int e = 0;
    while (e + 1 < j.n_entries && raw >= j.e[e + 1].row0) ++e;
    const int64_t local = raw - j.e[e].row0;
    return j.e[e].row0 + (local - local % j.quantum);
}

// Stages of one CTA in one job: at most G rows, never crossing an entry.
struct JobWalker {
    int64_t g, gend;
    int e;
    __device__ __forceinline__ bool next(const ChainJob& j, int& entry, int64_t& lrow, int& nrows) {
        if (g >= gend) return false;
        while (g >= j.e[e].row0 + j.e[e].rows) ++e;
        const int64_t entry_end = j.e[e].row0 + j.e[e].rows;
        const int64_t stop = gend < entry_end ? gend : entry_end;
        const int64_t n = stop - g < j.G ? stop - g : j.G;
        entry = e;
        lrow = g - j.e[e].row0;
        nrows = static_cast<int>(n);
        g += n;
        return true;
    }
};

__device__ __forceinline__ unsigned load_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Count one arrival, releasing every write this CTA made before it (the
// consumer barrier just before orders the other consumers' writes first).
__device__ __forceinline__ void arrive_release_gpu(unsigned* p) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(p) : "memory");
}

// Wait until *c >= target, for at most limit_ns; false (and an error code)
// when the wait runs out.  Polls without sleeping: one thread per CTA.
__device__ __forceinline__ bool wait_count(const unsigned* c, unsigned target, uint64_t limit_ns, unsigned* err) {
    if (load_acquire_gpu(c) >= target) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (load_acquire_gpu(c) >= target) return true;
        if ((it & 255u) == 0 && global_timer_ns() - t0 > limit_ns) {
            atomicOr(err, kErrTimeoutChain);
            return false;
        }
    }
}

struct Ring {
    uint8_t* smem;
    uint64_t* full;   // the slot's bytes have landed
    uint64_t* empty;  // consumers and reducer are done with the slot
    uint64_t* part;   // the consumers' partials of the slot's rows are stored
    float* red;       // per-lane partial sums, red_slot_floats per slot
    int S, slot_bytes, red_slot_floats;
};

// Consume this CTA's stages of one job.  k counts stages across jobs (the
// producer walks the same sequence).  Returns false if a wait ran out.
template <int FMT>
__device__ __forceinline__ bool run_job(const ChainParams& p, const ChainJob& jb, int jidx, int& k, const Ring& rg,
                                        const int8_t* q, const float* d, const int32_t* s, const Team& tm,
                                        const int64_t* range, int lane) {
    using LaneT = Lane<FMT, QX_MODE_W4A8>;
    static_assert(LaneT::kRows == gemv_rows_per_call(FMT, QX_MODE_W4A8), "row count must match the host geometry");
    if (threadIdx.x == 0) stamp(jidx, 8);
    LaneT X;
    if (tm.active) X.load(q, d, s, tm.slice, FMT != QX_Q8_0);  // slices permuted in shared memory
    if (threadIdx.x == 0) stamp(jidx, 9);
    const uint32_t rb = static_cast<uint32_t>(jb.row_bytes);
    JobWalker wk{range[0], range[1], 0};
    if (threadIdx.x == 0) stamp(jidx, 10);
    int e, nrows;
    int64_t lrow;
    bool first = true;
    while (wk.next(jb, e, lrow, nrows)) {
        const int slot = k % rg.S;
        if (first && threadIdx.x == 0) stamp(jidx, 11);
        if (!mbar_wait_bounded(&rg.full[slot], (k / rg.S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) return false;
        if (first && threadIdx.x == 0) stamp(jidx, 4);
        first = false;
        const uint8_t* sbuf = rg.smem + size_t(slot) * rg.slot_bytes;
        consume_stage<FMT, QX_MODE_W4A8, false>(X, tm, sbuf, nrows, rb, rg.red + size_t(slot) * rg.red_slot_floats,
                                                jb.RS, nullptr, 0);
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&rg.part[slot]);
            mbar_arrive(&rg.empty[slot]);
        }
        ++k;
    }
    return true;
}

// One CTA per SM: the ring can take most of the SM's shared memory.  Twelve
// warps in all (10 consumers, producer, reducer) are three per SM partition,
// so each thread may use up to 168 registers.
__global__ void __launch_bounds__(kChainThreads, 1) gemv_chain_kernel(const __grid_constant__ ChainParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_flag;
    Ring rg;
    rg.smem = smem;
    rg.S = p.stages;
    rg.slot_bytes = p.slot_bytes;
    rg.red_slot_floats = p.red_slot_floats;
    rg.full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    rg.empty = rg.full + rg.S;
    rg.part = rg.empty + rg.S;
    rg.red = reinterpret_cast<float*>(smem + p.red_off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < rg.S; ++s) {
            mbar_init(&rg.full[s], 1);
            mbar_init(&rg.empty[s], NW + 1);
            mbar_init(&rg.part[s], NW);
        }
        abort_flag = 0;
        fence_barrier_init();
    }
    // The job descriptors, copied once from the launch parameters into shared
    // memory: read from the parameter space, every job's first use would miss
    // the constant cache on each boundary's critical path (a few dependent
    // round trips to L2 while the weight stream loads it).
    ChainJob* jobs = reinterpret_cast<ChainJob*>(smem + p.jobs_off);
    {
        const uint4* src = reinterpret_cast<const uint4*>(&p.job[0]);
        uint4* dst = reinterpret_cast<uint4*>(jobs);
        const int words = p.n_jobs * int(sizeof(ChainJob) / 16);
        for (int i = threadIdx.x; i < words; i += blockDim.x) dst[i] = src[i];
    }
    // This CTA's row range of every job, [ranges[2j], ranges[2j + 1]), also
    // once at kernel start: the 64-bit divisions behind it would otherwise
    // sit on every job boundary of every role.
    int64_t* ranges = reinterpret_cast<int64_t*>(smem + p.ranges_off);
    for (int j = threadIdx.x; j < p.n_jobs; j += blockDim.x) {
        const ChainJob& jb = p.job[j];
        ranges[2 * j] = job_row_begin(jb, p.n_cta, blockIdx.x);
        ranges[2 * j + 1] = job_row_begin(jb, p.n_cta, blockIdx.x + 1);
    }
    __syncthreads();

    if (warp == NW) {
        // ---------------- producer: every job's rows, back to back ----------
        if (lane != 0) return;
        const uint64_t policy = policy_evict_first();
        int k = 0, issued = 0;
        unsigned tail_slots = 0;
        bool ok = true;
        for (int j = 0; j < p.n_jobs && ok; ++j) {
            const ChainJob& jb = jobs[j];
            JobWalker wk{ranges[2 * j], ranges[2 * j + 1], 0};
            int e, nrows;
            int64_t lrow;
            bool first = true;
            while (wk.next(jb, e, lrow, nrows)) {
                const int slot = k % rg.S;
                if (k >= rg.S &&
                    !mbar_wait_bounded(&rg.empty[slot], ((k / rg.S) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty)) {
                    ok = false;
                    break;
                }
                // at most p.inflight stages issued and not landed (0: the ring's
                // depth); stage k - p.inflight's slot is not reused before stage
                // k, so the parity is that stage's
                if (p.inflight > 0 && p.inflight < rg.S && k >= p.inflight) {
                    const int q = k - p.inflight;
                    if (!mbar_wait_bounded(&rg.full[q % rg.S], (q / rg.S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) {
                        ok = false;
                        break;
                    }
                }
                if (first) stamp(j, 0);
                first = false;
                const uint8_t* src = jb.e[e].W + lrow * jb.row_bytes;
                const uint32_t bytes = static_cast<uint32_t>(int64_t(nrows) * jb.row_bytes);
                const uint32_t abytes = bytes & ~15u;
                uint8_t* dst = smem + size_t(slot) * rg.slot_bytes;
                if (bytes != abytes) {
                    for (uint32_t t = abytes; t < bytes; ++t) dst[t] = src[t];
                    tail_slots |= 1u << slot;
                } else if (tail_slots & (1u << slot)) {
                    fence_proxy_async_smem();
                    tail_slots &= ~(1u << slot);
                }
                mbar_arrive_expect_tx(&rg.full[slot], abytes);
                if (abytes) bulk_g2s_evict_first(dst, src, abytes, &rg.full[slot], policy);
                issued = ++k;
            }
            stamp(j, 1);
        }
        for (int kk = issued > rg.S ? issued - rg.S : 0; kk < issued; ++kk)
            mbar_wait_bounded(&rg.full[kk % rg.S], (kk / rg.S) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
        return;
    }

    if (warp == NW + 1) {
        // ---------------- reducer: row sums, then job completion -----------
        int k = 0;
        bool ok = true;
        for (int j = 0; j < p.n_jobs && ok; ++j) {
            const ChainJob& jb = jobs[j];
            JobWalker wk{ranges[2 * j], ranges[2 * j + 1], 0};
            int e, nrows;
            int64_t lrow;
            while (wk.next(jb, e, lrow, nrows)) {
                const int slot = k % rg.S;
                if (!mbar_wait_bounded(&rg.part[slot], (k / rg.S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) {
                    ok = false;
                    break;
                }
                reduce_stage(rg.red + size_t(slot) * rg.red_slot_floats, jb.RS, jb.L, nrows, jb.e[e].y + lrow, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(&rg.empty[slot]);
                ++k;
            }
            if (!ok) break;
            if (lane == 0) stamp(j, 6);
            // every y of job j from this CTA is written: count the CTA.  The
            // warp barrier orders every lane's y stores before lane 0's
            // release, which makes them visible at GPU scope before the count
            // (release is cumulative).
            __syncwarp();
            if (lane == 0) {
                arrive_release_gpu(&p.counters[j]);
                stamp(j, 7);
            }
        }
        if (ok && lane == 0) {
            // the last CTA to finish the chain resets the counters for the next
            // call; every arrival of every CTA precedes its final count here
            __threadfence();
            if (atomicAdd(&p.counters[p.n_jobs], 1u) == unsigned(p.n_cta) - 1u) {
                for (int j = 0; j <= p.n_jobs; ++j) atomicExch(&p.counters[j], 0u);
                __threadfence();
            }
        }
        return;
    }

    // ---------------- consumers ----------------------------------------------
    pdl_wait_prior_grid();
    int8_t* sq = reinterpret_cast<int8_t*>(smem + p.act_off);
    float* sd = reinterpret_cast<float*>(sq + p.max_cols);
    int32_t* ss = reinterpret_cast<int32_t*>(sd + p.max_cols / 32);
    int k = 0;
    // the team layout of the previous job, rebuilt only when a job's differs
    Team tm = make_team(warp, lane, jobs[0].team_lanes, jobs[0].team_warps, jobs[0].nteams, jobs[0].L);
    for (int j = 0; j < p.n_jobs; ++j) {
        const ChainJob& jb = jobs[j];
        if (j > 0) {
            // job j may read job j - 1's output: wait for every CTA to finish it
            if (threadIdx.x == 0 && !wait_count(&p.counters[j - 1], unsigned(p.n_cta), p.wait_ns, p.err))
                abort_flag = 1;
            if (threadIdx.x == 0) stamp(j, 2);
            consumer_barrier<NW>();
            if (abort_flag) break;
        } else if (threadIdx.x == 0) {
            stamp(j, 2);
        }
        const int nblk = static_cast<int>(jb.cols / 32);
        quantize_all<2>(jb.x, nblk, threadIdx.x, NW * 32, sq, sd, ss, jb.fmt != QX_Q8_0);
        consumer_barrier<NW>();
        if (threadIdx.x == 0) stamp(j, 3);
        if (jb.team_lanes != tm.team_lanes || jb.team_warps != tm.team_warps || jb.nteams != tm.nteams ||
            jb.L != tm.L)
            tm = make_team(warp, lane, jb.team_lanes, jb.team_warps, jb.nteams, jb.L);
        const int64_t* rj = ranges + 2 * j;
        bool jok;
        switch (jb.fmt) {
            case QX_Q4_K: jok = run_job<QX_Q4_K>(p, jb, j, k, rg, sq, sd, ss, tm, rj, lane); break;
            case QX_Q6_K: jok = run_job<QX_Q6_K>(p, jb, j, k, rg, sq, sd, ss, tm, rj, lane); break;
            default: jok = run_job<QX_Q8_0>(p, jb, j, k, rg, sq, sd, ss, tm, rj, lane); break;
        }
        if (!jok) abort_flag = 1;
        consumer_barrier<NW>();  // every consumer has loaded its slice: the activation area may be rewritten
        if (threadIdx.x == 0) stamp(j, 5);
        if (abort_flag) break;
    }
}

constexpr int kMaxDynamicSmem = 227 * 1024;

cudaError_t configure_chain_once() {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    cudaFuncAttributes fa;
    err = cudaFuncGetAttributes(&fa, gemv_chain_kernel);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(gemv_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMaxDynamicSmem - static_cast<int>(fa.sharedSizeBytes));
    if (err == cudaSuccess) done[dev] = true;
    return err;
}

}  // namespace

cudaError_t chain_max_ctas_per_sm(size_t smem, int* out) {
    cudaError_t err = configure_chain_once();
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, gemv_chain_kernel, kChainThreads, smem);
}

cudaError_t chain_trace_read(void* host, size_t bytes) {
#ifdef QX_TRACE
    if (bytes > sizeof(g_trace)) bytes = sizeof(g_trace);
    return cudaMemcpyFromSymbol(host, g_trace, bytes);
#else
    (void)host;
    (void)bytes;
    return cudaErrorNotSupported;
#endif
}

cudaError_t launch_chain(const ChainParams& p, size_t smem, cudaStream_t s) {
    cudaError_t err = configure_chain_once();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_cta);
    cfg.blockDim = dim3(kChainThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_chain_kernel, p);
}

}  // namespace qx
