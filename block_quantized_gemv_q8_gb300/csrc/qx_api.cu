// qx_api.cu -- the C ABI declared in include/qx.h: argument validation,
// per-device set-up and launch geometry.  All arithmetic of the method runs
// in the kernels (qx_actq8.cu, qx_gemv.cu, qx_prefill.cu).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/qx.h"
#include "../../include/qx_debug.h"
#include "qx_internal.h"

namespace qx {

// Device error word: kernels OR a code in when a bounded wait runs out.
__device__ unsigned g_err_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s bound on every pipeline wait
// Build-time knobs for measurement sweeps (defaults are the shipped values).
// In-flight cap: with every SM streaming, the latency of every other load an
// SM makes (activation, parameters, the next kernel's first accesses) grows
// with the bytes queued in the memory system -- 0.2 us at 32 KB per SM, 0.3
// us at 64 KB, 0.85 us at 192 KB (GB300, L2-resident pointer chase beside a
// bulk-copy stream), while the stream itself needs only about 64 KB per SM to
// run at full rate.  A streaming GEMV CTA (two per SM) therefore keeps one
// stage in flight (Llama-3.1-8B decode step 1.167 -> 1.135 ms, same box;
// smaller stages were slower: the per-stage hand-offs cost more).
#ifndef QX_STAGE_KB
#define QX_STAGE_KB 48
#endif
#ifndef QX_INFLIGHT_KB
#define QX_INFLIGHT_KB 48
#endif
#ifndef QX_PREWAIT_KB
#define QX_PREWAIT_KB 0
#endif
constexpr size_t kStageTargetBytes = size_t(QX_STAGE_KB) * 1024;
// Most bytes a streaming CTA keeps in flight (0: no cap beyond the ring).
constexpr size_t kInflightBytes = size_t(QX_INFLIGHT_KB) * 1024;
#ifndef QX_CHAIN_INFLIGHT_KB
#define QX_CHAIN_INFLIGHT_KB 0
#endif
constexpr size_t kChainInflightBytes = size_t(QX_CHAIN_INFLIGHT_KB) * 1024;
// Bytes a large launch fetches before its dependency resolves (0: one stage).
constexpr size_t kPrewaitBytes = size_t(QX_PREWAIT_KB) * 1024;
// Shared memory of a CTA that leaves room for a second one on the SM.
constexpr size_t kHalfSmBytes = 110 * 1024;
// Automatic prefill path (measured on GB300, X [m, 4096] against Q4_K,
// Q6_K and Q8_0 weights of 4096, 14336 and 28672 rows): one GEMV for a single
// row of X (10.6 us on 14336 Q4_K rows); the small-batch GEMV up to
// prefill_batch_max_rows() rows; the tcgen05 GEMM above, which takes about
// 80 us for any M up to 256 (one tile row, every tile's K pipeline the same
// length) and 193 us at M = 512.  The small batch on the integer tensor path
// costs about 14.4 us per group of eight rows of X for 14336 x 4096 Q4_K
// (Q6_K 22-24, Q8_0 16-17): it beats tcgen05 up to 40 rows for Q4_K (71.9
// against 82.2 us), 32 for Q8_0 (67.9 against 80.1) and 24 for Q6_K (67.8
// against 89.6); on the lanes up to 16 (m = 16: 41 against 80 us).
constexpr int64_t kPrefillBatchMaxRows = 16;
// Shared memory of a chain CTA (one per SM): the ring, partial sums and
// activation within kChainSmBytes, and all of it with the job descriptors
// within kChainMaxSmem.
constexpr size_t kChainSmBytes = 200 * 1024;
constexpr size_t kChainMaxSmem = 227 * 1024;
constexpr int kMaxStageRows = 256;
// Launch bytes per SM up to which a PDL launch runs one CTA per SM.
constexpr int64_t kOneCtaPerSmBytes = 192 * 1024;
// Launches streaming at least this many bytes take the merged variant where
// one exists (gemv_has_merged).
constexpr int64_t kMergedMinBytes = int64_t(128) << 20;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int sm_count = 0;
    unsigned* err_word = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

// Text of the last CUDA failure on this thread (returned by qx_last_error).
thread_local char g_last_error[256] = "";

qx_status cuda_fail(cudaError_t e, const char* where) {
    std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e), int(e));
    cudaGetLastError();  // clear a non-sticky error so that it is not reported twice
    return QX_ERR_CUDA;
}
// Resident CTAs per SM, keyed by (device, format, mode, partials, merged, fused, smem bytes).
std::map<std::tuple<int, int, int, int, int, int, size_t>, int> g_occupancy;

qx_status ctas_per_sm(int fmt, int mode, bool partials, bool merged, bool fused, size_t smem, int* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    const auto key = std::make_tuple(dev, fmt, mode, partials ? 1 : 0, merged ? 1 : 0, fused ? 1 : 0, smem);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        auto it = g_occupancy.find(key);
        if (it != g_occupancy.end()) {
            *out = it->second;
            return QX_OK;
        }
    }
    int n = 0;
    if ((e = gemv_max_ctas_per_sm(fmt, mode, partials, merged, fused, smem, &n)) != cudaSuccess)
        return cuda_fail(e, "occupancy query");
    if (n < 1) return cuda_fail(cudaErrorInvalidConfiguration, "no CTA fits on an SM");
    std::lock_guard<std::mutex> lock(g_mu);
    g_occupancy[key] = n;
    *out = n;
    return QX_OK;
}

// Query the current device once: capability, SM count, error word address.
qx_status device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device ordinal");
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute");
        d.supported = (major == 10 && minor == 3);
        if (d.supported) {
            void* p = nullptr;
            if ((e = cudaGetSymbolAddress(&p, g_err_word)) != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
            d.err_word = static_cast<unsigned*>(p);
        }
        d.ready = true;
    }
    if (!d.supported) return QX_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return QX_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Outputs are written one 32-bit element at a time.
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int block_weights(int fmt) {
    switch (fmt) {
        case QX_Q8_0: return 32;
        case QX_Q4_K: return 256;
        case QX_Q6_K: return 256;
        case QX_Q6_K_SOA: return 256;
        default: return 0;
    }
}

int block_bytes(int fmt) {
    switch (fmt) {
        case QX_Q8_0: return 34;
        case QX_Q4_K: return 144;
        case QX_Q6_K: return 210;
        default: return 0;
    }
}

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// Bytes of one row (cols a positive multiple of the block width).  A
// QX_Q6_K_SOA row: 208 bytes per super-block, then the f16 d values padded to
// a 16-byte multiple.
int64_t row_bytes_of(int fmt, int64_t cols) {
    if (fmt == QX_Q6_K_SOA) {
        const int64_t nsb = cols / 256;
        return 208 * nsb + (2 * nsb + 15) / 16 * 16;
    }
    return cols / block_weights(fmt) * block_bytes(fmt);
}

qx_status check_shape(int fmt, int64_t rows, int64_t cols) {
    if (block_weights(fmt) == 0) return QX_ERR_FMT;
    if (rows < 1 || cols < 1 || cols % block_weights(fmt) != 0 || cols > QX_MAX_COLS) return QX_ERR_SHAPE;
    if (rows > (int64_t(1) << 40) / row_bytes_of(fmt, cols)) return QX_ERR_SHAPE;
    return QX_OK;
}

qx_status check_act(const qx_act_q8* a, int64_t m, int64_t cols) {
    if (!a || !a->q || !a->d || !a->sum) return QX_ERR_ARG;
    if (a->cols != cols || a->m < 1 || (m > 0 && a->m != m)) return QX_ERR_SHAPE;
    if (!aligned16(a->q) || !aligned16(a->d) || !aligned16(a->sum)) return QX_ERR_ALIGN;
    return QX_OK;
}

// Launch geometry of the streaming GEMV for one format/mode over a row space.
//   * A lane owns C columns, a team of lanes owns a row (several warps when
//     the row is wider than 32 lanes, several teams per warp when narrower).
//   * A stage is G whole rows (a multiple of the team count and of the rows
//     that make a 16-byte multiple), about kStageTargetBytes.
//   * W4A8 and Q8_0 launches keep each CTA within half an SM (registers and
//     shared memory) and run two CTAs per SM; under QX_FLAG_PDL the next
//     launch's CTAs take each SM's slots as this launch's CTAs leave them.
// Teams and stage rows for one format/mode/width (see gemv_geometry).
struct TeamGeom {
    int L, team_lanes, team_warps, nteams, quantum;
    int64_t rb, G, base;  // base: the smallest stage (rows) that keeps teams and copies whole
};

// batch_rows > 0: the small-batch lanes for that many rows of X.
qx_status team_geometry(int fmt, int kmode, bool partials, int64_t cols, int consumer_warps, TeamGeom& g,
                        int batch_rows = 0) {
    const bool batch = batch_rows > 0;
    const int C = batch ? batch_cols_per_lane(fmt, batch_rows) : gemv_cols_per_lane(fmt, kmode);
    if (cols % C) return QX_ERR_SHAPE;
    g.L = static_cast<int>(cols / C);
    if (g.L <= 32) {
        g.team_lanes = 1;
        while (g.team_lanes < g.L) g.team_lanes <<= 1;
        g.team_warps = 1;
        g.nteams = consumer_warps * (32 / g.team_lanes);
    } else {
        // teams of exactly L lanes, packed across warps
        g.team_warps = (g.L + 31) / 32;
        if (g.team_warps > consumer_warps) return QX_ERR_SHAPE;
        g.nteams = consumer_warps * 32 / g.L;
        g.team_lanes = g.L;
    }
    g.rb = row_bytes_of(fmt, cols);
    g.quantum = static_cast<int>(16 / gcd64(g.rb, 16));
    // every team gets the same number of whole row groups per stage
    const int64_t team_rows = int64_t(g.nteams) * ((partials || batch) ? 1 : gemv_rows_per_call(fmt, kmode));
    const int64_t base = team_rows / gcd64(team_rows, g.quantum) * g.quantum;  // lcm
    g.base = base;
    g.G = base;
    while (g.G + base <= kMaxStageRows && size_t((g.G + base) * g.rb) <= kStageTargetBytes) g.G += base;
    if (g.G > kMaxStageRows) g.G = base;  // very wide teams with tiny rows: keep one base group
    return QX_OK;
}

qx_status gemv_geometry(int fmt, int kmode, bool partials, bool fused, bool pdl, int64_t cols,
                        const DeviceInfo& dev, GemvParams& p, size_t& smem) {
    // The merged Q6_K W4A8 variant streams faster in steady state (lm_head
    // class launches: 5.95 TB/s against 5.40) but, packed next to the
    // following launches under PDL, costs the Llama-3.1-8B decode step more
    // than it saves on its 48 MB down projections: long launches only.
    const int64_t rb = row_bytes_of(fmt, cols);
    // f32 K-quants: the merged variant for small launches under programmatic
    // dependent launch (the launch then runs one CTA per SM, below, and the
    // next launch's CTA fits beside it)
    const bool small_bytes = p.total_rows * rb <= kOneCtaPerSmBytes * int64_t(dev.sm_count);
    bool merged = gemv_has_merged(fmt, kmode, partials) &&
                  (kmode == QX_MODE_F32 ? (pdl && small_bytes) : p.total_rows * rb >= kMergedMinBytes);
    TeamGeom g;
    // the merged variant's seven consumer warps cover rows of up to 28672
    // columns; wider rows take the standard kernel
    if (merged && team_geometry(fmt, kmode, partials, cols, gemv_consumer_warps(fmt, kmode, true), g) != QX_OK)
        merged = false;
    p.merged = merged ? 1 : 0;
    qx_status st = team_geometry(fmt, kmode, partials, cols, gemv_consumer_warps(fmt, kmode, merged), g);
    if (st != QX_OK) return st;
    const bool half_sm = (kmode == QX_MODE_W4A8 || fmt == QX_Q8_0 || merged);
    const size_t budget = half_sm ? kHalfSmBytes : 200 * 1024;
    const size_t act = fused ? (size_t(cols) + size_t(cols / 32) * 8 + 15) / 16 * 16 : 0;
    // per stage: the slot, three mbarriers and (for y outputs) the per-lane partial sums
    const int RS = partial_stride(g.L);
    const auto slot_of = [&](int64_t G) { return (size_t(G * g.rb) + kSlotPad + 127) / 128 * 128; };
    // The quantised activation (fused mode) is dead once every lane has its
    // slice in registers, before any partial sum is stored: the two share
    // one area.
    const auto bytes_for = [&](int64_t G, int st) {
        const size_t red = partials ? 0 : size_t(st) * size_t(G) * RS * 4;
        return size_t(st) * (slot_of(G) + 24) + 16 + (red > act ? red : act);
    };
    // Rows so wide that two stages exceed the budget: shrink the stage.
    while (g.G > g.base && bytes_for(g.G, 2) > budget) g.G -= g.base;
    const size_t slot = slot_of(g.G);
    const size_t red_stage = partials ? 0 : size_t(g.G) * RS * 4;
    int stages = 2;
    while (stages < 8 && bytes_for(g.G, stages + 1) <= budget) ++stages;
    p.bar_off = static_cast<int>(size_t(stages) * slot);
    p.red_off = static_cast<int>((size_t(p.bar_off) + 24 * size_t(stages) + 15) / 16 * 16);
    p.act_off = p.red_off;
    p.RS = RS;
    const size_t red_bytes = size_t(stages) * red_stage;
    smem = size_t(p.red_off) + (red_bytes > act ? red_bytes : act);
    if (smem > 227 * 1024) return QX_ERR_SHAPE;

    int per_sm = 0;
    st = ctas_per_sm(fmt, kmode, partials, merged, fused, smem, &per_sm);
    if (st != QX_OK) return st;
    // Under programmatic dependent launch, a launch that streams little per SM
    // runs one CTA per SM: the rest of each SM then holds the next launch's
    // CTA, which streams its weights during this launch's tail.  (GB300,
    // Llama-3.1-8B decode step: q/k/v and o launches at one CTA per SM,
    // gate/up and down at two, 1.38 ms per step; two everywhere, 1.47 ms.)
    const bool small = p.total_rows * g.rb <= kOneCtaPerSmBytes * int64_t(dev.sm_count);
    const int want = (pdl && small) ? 1 : 2;
    // A small launch fills its whole ring ahead of the preceding kernel's
    // completion; a large one only its first stage (measured on the same
    // step: 1.217 ms against 1.230 ms with one stage everywhere, 1.241 ms
    // with the whole ring everywhere).
    p.prewait = small ? stages : 1;
    if (!small && kPrewaitBytes > 0)
        p.prewait = std::max(1, std::min(stages, static_cast<int>(kPrewaitBytes / slot)));
    // the cap is per CTA at two CTAs per SM; a CTA alone on its SM keeps twice as much in flight
    const size_t inflight_cta = kInflightBytes * (want == 1 || per_sm < 2 ? 2 : 1);
    p.inflight = kInflightBytes > 0 ? std::max(1, static_cast<int>(inflight_cta / slot)) : 0;
    if (p.inflight >= stages) p.inflight = 0;
    const int64_t max_cta = int64_t(dev.sm_count) * (per_sm < want ? per_sm : want);
    const int64_t groups = (p.total_rows + g.quantum - 1) / g.quantum;
    p.cols = cols;
    p.row_bytes = g.rb;
    p.quantum = g.quantum;
    p.G = static_cast<int>(g.G);
    p.stages = stages;
    p.slot_bytes = static_cast<int>(slot);
    p.team_lanes = g.team_lanes;
    p.team_warps = g.team_warps;
    p.nteams = g.nteams;
    p.L = g.L;
    p.n_cta = static_cast<int>(groups < max_cta ? groups : max_cta);
    p.err = dev.err_word;
    p.wait_ns = kDefaultWaitNs;
    return QX_OK;
}

// Geometry of a chain: per-job teams and stage rows, one slot size and ring
// depth for all jobs, one CTA row split per job over the same grid.
qx_status chain_geometry(const DeviceInfo& dev, ChainParams& p, size_t& smem) {
    size_t max_stage = 0, red_slot = 4;
    int64_t max_cols = 0;
    for (int j = 0; j < p.n_jobs; ++j) {
        ChainJob& jb = p.job[j];
        TeamGeom g;
        const qx_status st = team_geometry(jb.fmt, QX_MODE_W4A8, false, jb.cols, kChainConsumerWarps, g);
        if (st != QX_OK) return st;
        jb.row_bytes = g.rb;
        jb.quantum = g.quantum;
        jb.G = static_cast<int>(g.G);
        jb.team_lanes = g.team_lanes;
        jb.team_warps = g.team_warps;
        jb.nteams = g.nteams;
        jb.L = g.L;
        jb.RS = partial_stride(g.L);
        max_stage = std::max(max_stage, size_t(g.G * g.rb));
        max_cols = std::max(max_cols, jb.cols);
        red_slot = std::max(red_slot, size_t(g.G) * jb.RS);
    }
    const size_t slot = (max_stage + kSlotPad + 127) / 128 * 128;
    const size_t act = (size_t(max_cols) + size_t(max_cols / 32) * 8 + 15) / 16 * 16;
    const size_t jobs_bytes = size_t(p.n_jobs) * (sizeof(ChainJob) + 2 * sizeof(int64_t));
    const auto bytes_for = [&](int st) { return size_t(st) * (slot + 24 + red_slot * 4) + 16 + act; };
    // the ring takes what the job descriptors leave of the budget
    const size_t ring_budget = std::min(kChainSmBytes, size_t(kChainMaxSmem) - jobs_bytes - 64);
    int stages = 2;
    while (stages < 8 && bytes_for(stages + 1) <= ring_budget) ++stages;
    p.stages = stages;
    p.slot_bytes = static_cast<int>(slot);
    p.red_slot_floats = static_cast<int>(red_slot);
    p.max_cols = max_cols;
    p.bar_off = static_cast<int>(size_t(stages) * slot);
    p.red_off = static_cast<int>((size_t(p.bar_off) + 24 * size_t(stages) + 15) / 16 * 16);
    p.act_off = static_cast<int>((size_t(p.red_off) + size_t(stages) * red_slot * 4 + 15) / 16 * 16);
    p.jobs_off = static_cast<int>((size_t(p.act_off) + act + 15) / 16 * 16);
    p.ranges_off = static_cast<int>(size_t(p.jobs_off) + size_t(p.n_jobs) * sizeof(ChainJob));
    smem = size_t(p.jobs_off) + jobs_bytes;
    if (smem > 227 * 1024) return QX_ERR_SHAPE;
    int per_sm = 0;
    const cudaError_t e = chain_max_ctas_per_sm(smem, &per_sm);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (per_sm < 1) return cuda_fail(cudaErrorInvalidConfiguration, "no CTA fits on an SM");
    p.n_cta = dev.sm_count;  // one CTA per SM (the kernel is built for one)
    p.inflight = kChainInflightBytes > 0 ? std::max(1, static_cast<int>(kChainInflightBytes / slot)) : 0;
    if (p.inflight >= stages) p.inflight = 0;
    p.err = dev.err_word;
    p.wait_ns = kDefaultWaitNs;
    return QX_OK;
}

// One streaming-GEMV launch over `n` matrices of the same format.  `mode` is
// the public mode (flags already removed).
// Whether the f32-mode tensor-pipe kernel (gemv_f32_mma_kernel) serves the
// shape: Q6_K rows (either layout) of 2048 or 4096 columns, where both
// layouts are served alike (GGUF rows are then a 16-byte multiple), so their
// outputs stay bit-identical; Q4_K rows of 256 to 4096 columns, except small
// launches under programmatic dependent launch, which take the merged f32
// lanes (half an SM, so the next launch's CTA fits beside them).
bool f32_mma_serves(int fmt, int64_t cols, bool pdl_small) {
    if (fmt == QX_Q6_K || fmt == QX_Q6_K_SOA) return cols == 2048 || cols == 4096;
    if (fmt == QX_Q4_K) return !pdl_small && cols % 256 == 0 && cols / 256 >= 1 && cols / 256 <= 16;
    return false;
}

// f32 mode on the tensor pipe: stages of 16 P gq rows (P = 16 / units per
// row warps per unit, each taking gq 16-row groups a stage) at a padded
// stride of row_bytes + 16, per stage the consumers' partials [P gq][units][16]
// floats.  One group a warp and stage: four stages of 16 rows of 4096
// columns ran the lm_head faster than two stages of 32 rows (80.5 against
// 88.8 us, repacked layout), which halve the per-stage overhead per output.
qx_status run_gemv_f32_mma(int fmt, GemvParams& p, int64_t cols, const DeviceInfo& dev, bool pdl, cudaStream_t s) {
    const int nsb = static_cast<int>(cols / 256), P = 16 / nsb, gq = 1;
    const int64_t rb = row_bytes_of(fmt, cols);
    const size_t slot = (size_t(16 * P * gq) * size_t(rb + 16) + 127) / 128 * 128;
    const size_t red_stage = size_t(P * gq) * nsb * 16 * 4;
    const size_t budget = 224 * 1024;
    int stages = 2;
    while (stages < 8 && size_t(stages + 1) * (slot + red_stage + 24) + 32 <= budget) ++stages;
    p.red_off = static_cast<int>(size_t(stages) * slot);
    p.bar_off = static_cast<int>(size_t(p.red_off) + size_t(stages) * red_stage);
    const size_t smem = size_t(p.bar_off) + 24 * size_t(stages);
    if (smem > 227 * 1024) return QX_ERR_SHAPE;
    p.cols = cols;
    p.row_bytes = rb;
    p.quantum = 16;
    p.G = 16 * P * gq;
    p.gq = gq;
    p.stages = stages;
    p.slot_bytes = static_cast<int>(slot);
    int64_t groups = 0;  // 16-row groups over the entries
    for (int k = 0; k < p.n_entries; ++k) groups += (p.e[k].rows + 15) / 16;
    p.n_cta = static_cast<int>(groups < dev.sm_count ? groups : dev.sm_count);
    p.err = dev.err_word;
    p.wait_ns = kDefaultWaitNs;
    const cudaError_t e = launch_gemv_f32_mma(fmt, p, smem, s, pdl);
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "gemv (f32, tensor) launch");
}

qx_status run_gemv(int fmt, int n, const void* const* W, const int64_t* rows, int64_t cols, const void* x,
                   float* const* y, int32_t* P, int mode, bool pdl, cudaStream_t s) {
    DeviceInfo* dev = nullptr;
    qx_status st = device_info(&dev);
    if (st != QX_OK) return st;
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.n_entries = n;
    int64_t total = 0;
    for (int k = 0; k < n; ++k) {
        p.e[k].W = static_cast<const uint8_t*>(W[k]);
        p.e[k].y = y ? y[k] : nullptr;
        p.e[k].P = P;
        p.e[k].rows = rows[k];
        p.e[k].row0 = total;
        total += rows[k];
    }
    p.total_rows = total;
    int kmode = QX_MODE_W4A8;
    if (mode == QX_MODE_F32) {
        p.x = static_cast<const float*>(x);
        kmode = QX_MODE_F32;
        const bool pdl_small = pdl && total * row_bytes_of(fmt, cols) <= kOneCtaPerSmBytes * int64_t(dev->sm_count);
        if (P == nullptr && y != nullptr && f32_mma_serves(fmt, cols, pdl_small))
            return run_gemv_f32_mma(fmt, p, cols, *dev, pdl, s);
    } else if (mode == QX_MODE_W4A8_FUSED) {
        p.xf = static_cast<const float*>(x);
    } else {
        const qx_act_q8* a = static_cast<const qx_act_q8*>(x);
        p.xq = a->q;
        p.xd = a->d;
        p.xs = a->sum;
    }
    size_t smem = 0;
    st = gemv_geometry(fmt, kmode, P != nullptr, p.xf != nullptr, pdl, cols, *dev, p, smem);
    if (st != QX_OK) return st;
    const cudaError_t e = launch_gemv(fmt, kmode, P != nullptr, p, smem, s, pdl);
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "gemv launch");
}

// One small-batch launch (gemv_batch_kernel): rows m0 .. m0 + mvalid - 1 of
// X (mvalid <= mb, mb = kBatchRows or kBatchRowsWide) against W [rows,
// cols], into Y [X->m, rows].
// Whether the integer-tensor small-batch kernel serves the shape: rows of
// 256 to 4096 columns in whole 256-column units (a Q4_K or Q6_K super-block,
// eight Q8_0 blocks), each row a 16-byte multiple (copied row by row; Q6_K
// rows of 2048 or 4096 columns).
bool batch_mma_serves(int fmt, int64_t cols) {
    if (fmt != QX_Q4_K && fmt != QX_Q6_K && fmt != QX_Q8_0) return false;
    if (cols % 256 != 0 || cols / 256 < 1 || cols / 256 > kMmaBatchMaxSuperBlocks) return false;
    return row_bytes_of(fmt, cols) % 16 == 0;
}

// The most rows of X the automatic prefill path gives the small-batch GEMV.
int64_t prefill_batch_max_rows(int fmt, int64_t cols) {
    if (!batch_mma_serves(fmt, cols)) return kPrefillBatchMaxRows;
    return fmt == QX_Q4_K ? 40 : (fmt == QX_Q8_0 ? 32 : 24);
}

// Up to eight rows of X (from row m0) on the integer tensor path
// (gemv_batch_mma_kernel).  Stage: 16 P rows (P = 16 / units per row) at a
// padded stride of row_bytes + 16; per stage the consumers' partials
// [P][units][16 x 8] floats; one table of the activation scales (one float4
// per 32-column block and pair of rows of X; Q6_K: per 16-column group).
qx_status run_gemv_batch_mma(int fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* X, int64_t m0,
                             int mvalid, float* Y, cudaStream_t s) {
    DeviceInfo* dev = nullptr;
    qx_status st = device_info(&dev);
    if (st != QX_OK) return st;
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.n_entries = 1;
    p.e[0].W = static_cast<const uint8_t*>(W);
    p.e[0].y = Y + m0 * rows;
    p.e[0].rows = rows;
    p.e[0].row0 = 0;
    p.total_rows = rows;
    p.xq = X->q + m0 * cols;
    p.xd = X->d + m0 * (cols / 32);
    p.xs = X->sum + m0 * (cols / 32);
    p.mb = kMmaBatchRows;
    p.m_valid = mvalid;
    p.y_stride = rows;
    const int nsb = static_cast<int>(cols / 256), P = 16 / nsb;
    const int64_t rb = row_bytes_of(fmt, cols);
    const size_t slot = (size_t(16 * P) * size_t(rb + 16) + 127) / 128 * 128;
    const size_t red_stage = size_t(P) * nsb * 128 * 4;
    const size_t act = size_t(cols / 32) * 64 * (fmt == QX_Q6_K ? 2 : 1);  // four float4 per block (group)
    const size_t budget = 200 * 1024;
    int stages = 2;
    while (stages < 8 && size_t(stages + 1) * (slot + red_stage + 24) + act + 32 <= budget) ++stages;
    p.red_off = static_cast<int>(size_t(stages) * slot);
    p.act_off = static_cast<int>(size_t(p.red_off) + size_t(stages) * red_stage);
    p.bar_off = static_cast<int>(size_t(p.act_off) + act);
    const size_t smem = size_t(p.bar_off) + 24 * size_t(stages);
    if (smem > 227 * 1024) return QX_ERR_SHAPE;
    p.cols = cols;
    p.row_bytes = rb;
    p.quantum = 16;
    p.G = 16 * P;
    p.stages = stages;
    p.slot_bytes = static_cast<int>(slot);
    const int64_t groups = (rows + 15) / 16;
    p.n_cta = static_cast<int>(groups < dev->sm_count ? groups : dev->sm_count);
    p.err = dev->err_word;
    p.wait_ns = kDefaultWaitNs;
    const cudaError_t e = launch_gemv_batch_mma(fmt, p, smem, s);
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "batched gemv (tensor) launch");
}

qx_status run_gemv_batch(int fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* X, int64_t m0,
                         int mvalid, int mb, float* Y, cudaStream_t s) {
    DeviceInfo* dev = nullptr;
    qx_status st = device_info(&dev);
    if (st != QX_OK) return st;
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.n_entries = 1;
    p.e[0].W = static_cast<const uint8_t*>(W);
    p.e[0].y = Y + m0 * rows;
    p.e[0].rows = rows;
    p.e[0].row0 = 0;
    p.total_rows = rows;
    p.xq = X->q + m0 * cols;
    p.xd = X->d + m0 * (cols / 32);
    p.xs = X->sum + m0 * (cols / 32);
    p.mb = mb;
    p.m_valid = mvalid;
    p.y_stride = rows;
    TeamGeom g;
    if ((st = team_geometry(fmt, QX_MODE_W4A8, false, cols, kBatchConsumerWarps, g, mb)) != QX_OK) return st;
    const int RS = partial_stride(g.L);
    const auto slot_of = [&](int64_t G) { return (size_t(G * g.rb) + kSlotPad + 127) / 128 * 128; };
    const auto bytes_for = [&](int64_t G, int stg) {
        return size_t(stg) * (slot_of(G) + 24 + size_t(G) * mb * RS * 4) + 32;
    };
    const size_t budget = 200 * 1024;
    while (g.G > g.base && bytes_for(g.G, 2) > budget) g.G -= g.base;
    int stages = 2;
    while (stages < 8 && bytes_for(g.G, stages + 1) <= budget) ++stages;
    const size_t slot = slot_of(g.G);
    p.bar_off = static_cast<int>(size_t(stages) * slot);
    p.red_off = static_cast<int>((size_t(p.bar_off) + 24 * size_t(stages) + 15) / 16 * 16);
    p.act_off = p.red_off;
    const size_t smem = size_t(p.red_off) + size_t(stages) * size_t(g.G) * mb * RS * 4;
    if (smem > 227 * 1024) return QX_ERR_SHAPE;
    p.RS = RS;
    p.cols = cols;
    p.row_bytes = g.rb;
    p.quantum = g.quantum;
    p.G = static_cast<int>(g.G);
    p.stages = stages;
    p.slot_bytes = static_cast<int>(slot);
    p.team_lanes = g.team_lanes;
    p.team_warps = g.team_warps;
    p.nteams = g.nteams;
    p.L = g.L;
    const int64_t groups = (rows + g.quantum - 1) / g.quantum;
    p.n_cta = static_cast<int>(groups < dev->sm_count ? groups : dev->sm_count);
    p.prewait = stages;
    p.err = dev->err_word;
    p.wait_ns = kDefaultWaitNs;
    const cudaError_t e = launch_gemv_batch(fmt, p, smem, s);
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "batched gemv launch");
}

// Split a public mode argument into the mode and the PDL flag.
qx_status parse_mode(int mode_arg, int* mode, bool* pdl) {
    if (mode_arg & ~(0xFF | QX_FLAG_PDL)) return QX_ERR_MODE;
    *mode = mode_arg & 0xFF;
    *pdl = (mode_arg & QX_FLAG_PDL) != 0;
    if (*mode != QX_MODE_F32 && *mode != QX_MODE_W4A8 && *mode != QX_MODE_W4A8_FUSED) return QX_ERR_MODE;
    return QX_OK;
}

qx_status check_x(int mode, const void* x, int64_t cols) {
    if (!x) return QX_ERR_ARG;
    if (mode == QX_MODE_F32 || mode == QX_MODE_W4A8_FUSED) return aligned16(x) ? QX_OK : QX_ERR_ALIGN;
    if (mode == QX_MODE_W4A8) return check_act(static_cast<const qx_act_q8*>(x), 1, cols);
    return QX_ERR_MODE;
}

}  // namespace
}  // namespace qx

using namespace qx;

namespace {

qx_status prefill_dispatch(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* X, float* Y,
                           int path, qx_stream_t s) {
    qx_status st = check_shape(fmt, rows, cols);
    if (st != QX_OK) return st;
    if (!W || !Y) return QX_ERR_ARG;
    if (!aligned16(W) || !aligned4(Y)) return QX_ERR_ALIGN;
    if ((st = check_act(X, 0, cols)) != QX_OK) return st;
    if (path < 0 || path > 4) return QX_ERR_ARG;
    if (fmt == QX_Q6_K_SOA) {
        if (path != 0 && path != 1) return QX_ERR_FMT;  // the GEMM paths read the GGUF layouts
        path = 1;
    }
    const int64_t rb = row_bytes_of(fmt, cols);
    if (path == 0) {
        path = X->m == 1 ? 1 : (X->m <= prefill_batch_max_rows(fmt, cols) ? 4 : 3);
        // shapes beyond the tensor-core kernel's 32-bit copy coordinates take one GEMV per row
        if (path == 3 && !prefill_tc_serves(fmt, rows, cols, X->m, rb)) path = 1;
        // rows wider than the small-batch lanes cover (eight-row lanes: 14336
        // columns, four-row K-quant lanes: 28672) take one GEMV per row
        if (path == 4) {
            TeamGeom g;
            const int mb = X->m > kBatchRows ? kBatchRowsWide : kBatchRows;
            if (team_geometry(fmt, QX_MODE_W4A8, false, cols, kBatchConsumerWarps, g, mb) != QX_OK ||
                team_geometry(fmt, QX_MODE_W4A8, false, cols, kBatchConsumerWarps, g, kBatchRows) != QX_OK)
                path = 1;
        }
    }
    if (path == 4) {
        // While more than four rows of X remain, eight of them per weight
        // stream: on the integer tensor path for rows of up to 4096 columns in
        // whole 256-column units, else on the eight-row lanes.  Then up to four
        // on the four-row lanes (faster than the tensor path at four rows or
        // fewer: 14.4 against 16.4 us for Q4_K, 20.5 against 22.8-24.1 for
        // Q6_K, equal for Q8_0, on 14336 x 4096).
        const bool mma_shape = batch_mma_serves(fmt, cols);
        for (int64_t m0 = 0; m0 < X->m;) {
            const int64_t left = X->m - m0;
            const bool mma = mma_shape && left > kBatchRows;
            const int mb = mma ? kMmaBatchRows : (left > kBatchRows ? kBatchRowsWide : kBatchRows);
            const int mv = static_cast<int>(left < mb ? left : mb);
            if (!aligned16(X->q + m0 * cols) || !aligned16(X->d + m0 * (cols / 32)) ||
                !aligned16(X->sum + m0 * (cols / 32)))
                return QX_ERR_ALIGN;
            st = mma ? run_gemv_batch_mma(fmt, W, rows, cols, X, m0, mv, Y, reinterpret_cast<cudaStream_t>(s))
                     : run_gemv_batch(fmt, W, rows, cols, X, m0, mv, mb, Y, reinterpret_cast<cudaStream_t>(s));
            if (st != QX_OK) return st;
            m0 += mv;
        }
        return QX_OK;
    }
    if (path == 3) {
        if (!prefill_tc_serves(fmt, rows, cols, X->m, rb)) return QX_ERR_SHAPE;
        DeviceInfo* dev = nullptr;
        if ((st = device_info(&dev)) != QX_OK) return st;
        const cudaError_t e = launch_prefill_tc(fmt, static_cast<const uint8_t*>(W), rows, cols, rb, X->q, X->d, X->m,
                                                Y, dev->err_word, dev->sm_count, reinterpret_cast<cudaStream_t>(s));
        return e == cudaSuccess ? QX_OK : cuda_fail(e, "tcgen05 prefill launch");
    }
    const bool tensor = path == 2;
    if (tensor) {
        if (fmt != QX_Q4_K) return QX_ERR_FMT;  // the tensor-core path serves Q4_K
        DeviceInfo* dev = nullptr;
        if ((st = device_info(&dev)) != QX_OK) return st;
        const cudaError_t e = launch_prefill_q4k(static_cast<const uint8_t*>(W), rows, cols, X->q, X->d, X->sum,
                                                 X->m, Y, reinterpret_cast<cudaStream_t>(s));
        return e == cudaSuccess ? QX_OK : cuda_fail(e, "prefill launch");
    }
    // Row-by-row: each row of X is an independent W4A8 GEMV.
    for (int64_t m = 0; m < X->m; ++m) {
        qx_act_q8 row{X->q + m * cols, X->d + m * (cols / 32), X->sum + m * (cols / 32), 1, cols};
        if (!aligned16(row.q) || !aligned16(row.d) || !aligned16(row.sum)) return QX_ERR_ALIGN;
        float* ym = Y + m * rows;
        if ((st = run_gemv(fmt, 1, &W, &rows, cols, &row, &ym, nullptr, QX_MODE_W4A8, false,
                           reinterpret_cast<cudaStream_t>(s))) != QX_OK)
            return st;
    }
    return QX_OK;
}

// Validate a chain's jobs and copy them into the launch descriptor (shared by
// qx_gemv_chain and qx_gemv_chain_noalloc); every check runs before any
// device work.  p.n_jobs is set; the geometry is left to chain_geometry.
qx_status marshal_chain(int n_jobs, const qx_gemv_job* jobs, ChainParams& p) {
    if (n_jobs < 1 || n_jobs > QX_CHAIN_MAX_JOBS || !jobs) return QX_ERR_ARG;
    std::memset(&p, 0, sizeof(p));
    p.n_jobs = n_jobs;
    qx_status st;
    for (int j = 0; j < n_jobs; ++j) {
        const qx_gemv_job& in = jobs[j];
        if (in.n < 1 || in.n > QX_CHAIN_MAX_ENTRIES) return QX_ERR_ARG;
        if (!in.x) return QX_ERR_ARG;
        if (!aligned16(in.x)) return QX_ERR_ALIGN;
        if (in.fmt == QX_Q6_K_SOA) return QX_ERR_FMT;  // the chain kernel reads the GGUF layouts
        ChainJob& jb = p.job[j];
        jb.fmt = in.fmt;
        jb.n_entries = in.n;
        jb.cols = in.cols;
        jb.x = in.x;
        int64_t total = 0;
        for (int k = 0; k < in.n; ++k) {
            if ((st = check_shape(in.fmt, in.rows[k], in.cols)) != QX_OK) return st;
            if (!in.W[k] || !in.y[k]) return QX_ERR_ARG;
            if (!aligned16(in.W[k]) || !aligned4(in.y[k])) return QX_ERR_ALIGN;
            jb.e[k].W = static_cast<const uint8_t*>(in.W[k]);
            jb.e[k].y = in.y[k];
            jb.e[k].rows = in.rows[k];
            jb.e[k].row0 = total;
            total += in.rows[k];
        }
        jb.total_rows = total;
    }
    return QX_OK;
}

}  // namespace

extern "C" {

size_t qx_row_bytes(qx_fmt fmt, int64_t cols) {
    const int bw = block_weights(fmt);
    if (bw == 0 || cols < 1 || cols % bw) return 0;
    return size_t(row_bytes_of(fmt, cols));
}

qx_status qx_repack(qx_fmt from, qx_fmt to, const void* src, int64_t rows, int64_t cols, void* dst,
                    qx_stream_t s) {
    const bool to_soa = from == QX_Q6_K && to == QX_Q6_K_SOA;
    if (!to_soa && !(from == QX_Q6_K_SOA && to == QX_Q6_K)) return QX_ERR_FMT;
    qx_status st = check_shape(from, rows, cols);
    if (st != QX_OK) return st;
    if ((st = check_shape(to, rows, cols)) != QX_OK) return st;
    if (!src || !dst) return QX_ERR_ARG;
    if (!aligned16(src) || !aligned16(dst)) return QX_ERR_ALIGN;
    const int64_t sb = row_bytes_of(from, cols), db = row_bytes_of(to, cols);
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src), d0 = reinterpret_cast<uintptr_t>(dst);
    if (s0 < d0 + uintptr_t(rows * db) && d0 < s0 + uintptr_t(rows * sb)) return QX_ERR_ARG;  // overlap
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != QX_OK) return st;
    const cudaError_t e = launch_repack_q6k(to_soa, static_cast<const uint8_t*>(src), rows, cols / 256, sb,
                                            static_cast<uint8_t*>(dst), db, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "repack launch");
}

qx_status qx_quantize_act_q8(const float* x, int64_t m, int64_t cols, qx_act_q8* out, qx_stream_t s) {
    if (!x || !out || !out->q || !out->d || !out->sum) return QX_ERR_ARG;
    if (m < 1 || cols < 32 || cols % 32 || cols > (int64_t(1) << 30) || m > (int64_t(1) << 40) / cols)
        return QX_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(out->q) || !aligned16(out->d) || !aligned16(out->sum)) return QX_ERR_ALIGN;
    DeviceInfo* dev = nullptr;
    const qx_status st = device_info(&dev);
    if (st != QX_OK) return st;
    const cudaError_t e =
        launch_actq8(x, m * cols / 32, out->q, out->d, out->sum, dev->sm_count, reinterpret_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return cuda_fail(e, "actq8 launch");
    out->m = m;
    out->cols = cols;
    return QX_OK;
}

qx_status qx_gemv(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const void* x, float* y, qx_mode mode_arg,
                  qx_stream_t s) {
    int mode;
    bool pdl;
    qx_status st = parse_mode(mode_arg, &mode, &pdl);
    if (st != QX_OK) return st;
    if ((st = check_shape(fmt, rows, cols)) != QX_OK) return st;
    if (!W || !y) return QX_ERR_ARG;
    if (!aligned16(W) || !aligned4(y)) return QX_ERR_ALIGN;
    if ((st = check_x(mode, x, cols)) != QX_OK) return st;
    return run_gemv(fmt, 1, &W, &rows, cols, x, &y, nullptr, mode, pdl, reinterpret_cast<cudaStream_t>(s));
}

qx_status qx_gemv_multi(int n, const qx_fmt* fmt, const void* const* W, const int64_t* rows, int64_t cols,
                        const void* x, float* const* y, qx_mode mode_arg, qx_stream_t s) {
    if (n < 1 || n > QX_MAX_MULTI || !fmt || !W || !rows || !y) return QX_ERR_ARG;
    int mode;
    bool pdl;
    qx_status st = parse_mode(mode_arg, &mode, &pdl);
    if (st != QX_OK) return st;
    for (int k = 0; k < n; ++k) {
        if ((st = check_shape(fmt[k], rows[k], cols)) != QX_OK) return st;
        if (!W[k] || !y[k]) return QX_ERR_ARG;
        if (!aligned16(W[k]) || !aligned4(y[k])) return QX_ERR_ALIGN;
    }
    if ((st = check_x(mode, x, cols)) != QX_OK) return st;
    // One launch per distinct format (in order of first appearance), entries
    // kept in call order; every entry's format passed check_shape above.
    int fmts[QX_MAX_MULTI];
    int nfmt = 0;
    for (int k = 0; k < n; ++k) {
        bool seen = false;
        for (int i = 0; i < nfmt; ++i) seen |= fmts[i] == fmt[k];
        if (!seen) fmts[nfmt++] = fmt[k];
    }
    for (int i = 0; i < nfmt; ++i) {
        const int f = fmts[i];
        const void* Wf[QX_MAX_MULTI];
        int64_t rf[QX_MAX_MULTI];
        float* yf[QX_MAX_MULTI];
        int nf = 0;
        for (int k = 0; k < n; ++k)
            if (fmt[k] == f) {
                Wf[nf] = W[k];
                rf[nf] = rows[k];
                yf[nf] = y[k];
                ++nf;
            }
        if (nf == 0) continue;
        if ((st = run_gemv(f, nf, Wf, rf, cols, x, yf, nullptr, mode, pdl, reinterpret_cast<cudaStream_t>(s))) !=
            QX_OK)
            return st;
    }
    return QX_OK;
}

qx_status qx_gemv_partials(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* x, int32_t* P,
                           qx_stream_t s) {
    qx_status st = check_shape(fmt, rows, cols);
    if (st != QX_OK) return st;
    if (!W || !P) return QX_ERR_ARG;
    if (!aligned16(W) || !aligned4(P)) return QX_ERR_ALIGN;
    if ((st = check_act(x, 1, cols)) != QX_OK) return st;
    return run_gemv(fmt, 1, &W, &rows, cols, x, nullptr, P, QX_MODE_W4A8, false, reinterpret_cast<cudaStream_t>(s));
}

qx_status qx_gemm_prefill_ex(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* X, float* Y,
                             int path, qx_stream_t s) {
    return prefill_dispatch(fmt, W, rows, cols, X, Y, path, s);
}

qx_status qx_gemm_prefill(qx_fmt fmt, const void* W, int64_t rows, int64_t cols, const qx_act_q8* X, float* Y,
                          qx_stream_t s) {
    return prefill_dispatch(fmt, W, rows, cols, X, Y, 0, s);
}

size_t qx_gemv_chain_scratch_bytes(int n_jobs) {
    if (n_jobs < 1 || n_jobs > QX_CHAIN_MAX_JOBS) return 0;
    return size_t(n_jobs + 1) * sizeof(unsigned);
}

qx_status qx_gemv_chain(int n_jobs, const qx_gemv_job* jobs, void* scratch, qx_stream_t s) {
    if (n_jobs < 1 || n_jobs > QX_CHAIN_MAX_JOBS || !jobs || !scratch) return QX_ERR_ARG;
    if (!aligned4(scratch)) return QX_ERR_ALIGN;
    static thread_local ChainParams p;  // large (tens of KB): not on the stack
    qx_status st = marshal_chain(n_jobs, jobs, p);
    if (st != QX_OK) return st;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != QX_OK) return st;
    size_t smem = 0;
    if ((st = chain_geometry(*dev, p, smem)) != QX_OK) return st;
    p.counters = static_cast<unsigned*>(scratch);
    const cudaError_t e = launch_chain(p, smem, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "chain launch");
}

qx_status qx_device_check(qx_stream_t s) {
    DeviceInfo* dev = nullptr;
    const qx_status st = device_info(&dev);
    if (st != QX_OK) return st;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned word = 0;
    if ((e = cudaMemcpyFromSymbol(&word, g_err_word, sizeof(word))) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpyFromSymbol");
    if (word) {
        const unsigned zero = 0;
        if ((e = cudaMemcpyToSymbol(g_err_word, &zero, sizeof(zero))) != cudaSuccess)
            return cuda_fail(e, "cudaMemcpyToSymbol");
        return QX_ERR_DEVICE_TIMEOUT;
    }
    return QX_OK;
}

qx_status qx_debug_timeout_probe(uint64_t limit_ns, qx_stream_t s) {
    if (limit_ns < 1000000ull || limit_ns > 10000000000ull) return QX_ERR_ARG;
    DeviceInfo* dev = nullptr;
    const qx_status st = device_info(&dev);
    if (st != QX_OK) return st;
    const cudaError_t e = launch_timeout_probe(dev->err_word, limit_ns, reinterpret_cast<cudaStream_t>(s));
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "probe launch");
}

const char* qx_status_string(qx_status st) {
    switch (st) {
        case QX_OK: return "QX_OK";
        case QX_ERR_ARG: return "QX_ERR_ARG: null pointer or invalid argument";
        case QX_ERR_FMT: return "QX_ERR_FMT: unknown block format";
        case QX_ERR_SHAPE: return "QX_ERR_SHAPE: shape not served (cols must be whole blocks, within limits)";
        case QX_ERR_ALIGN: return "QX_ERR_ALIGN: a pointer is not 16-byte aligned";
        case QX_ERR_MODE: return "QX_ERR_MODE: unknown mode";
        case QX_ERR_CUDA: return "QX_ERR_CUDA: a CUDA call or kernel launch failed";
        case QX_ERR_DEVICE_TIMEOUT: return "QX_ERR_DEVICE_TIMEOUT: a kernel's bounded wait ran out";
        case QX_ERR_UNSUPPORTED_DEVICE:
            return "QX_ERR_UNSUPPORTED_DEVICE: the current device is not compute capability 10.3 (GB300)";
        default: return "unknown qx status";
    }
}

const char* qx_last_error(void) { return g_last_error; }

const char* qx_version(void) {
    return "qx 0.2 sm_103a: actq8; gemv {q4_k,q6_k,q6_k_soa,q8_0} x {f32,w4a8,w4a8 fused} (bulk-copy stream, "
           "pdl); multi; chain; partials; prefill {gemv per row, mma.sync, tcgen05, small batch}; repack";
}

// ----------------------------------------------------------------------------
// qx_gemv_chain_noalloc: qx_gemv_chain with library-owned scratch.
//
// qx_gemv_chain needs a few hundred bytes of device scratch for its per-job
// arrival counters, which its caller allocates.  Some callers cannot
// allocate device memory at the point where they run a chain: code that
// executes while a CUDA graph is being captured (cudaMalloc is not allowed
// there), runtimes that hand out device memory only from a fixed pool set up
// at start, or plug-ins that may not touch the process's allocator.  For
// them the counters live in the array below, which every GPU that loads the
// library holds until the process exits.
// ----------------------------------------------------------------------------

// Largest chain the array serves (one counter per job plus one exit counter).
constexpr int kNoallocMaxJobs = QX_CHAIN_MAX_JOBS;
static __device__ __align__(256) unsigned g_noalloc_counters[kNoallocMaxJobs + 1];

namespace {
std::mutex g_noalloc_mu;
unsigned* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the counter array on the current device, looked up once
// per device (with that device current) and cached.
qx_status noalloc_counters(unsigned** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice, "device ordinal");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        unsigned* ptr = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_noalloc_counters);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return QX_OK;
}
}  // namespace

qx_status qx_gemv_chain_noalloc(int n_jobs, const qx_gemv_job* jobs, qx_stream_t s) {
    if (n_jobs > kNoallocMaxJobs) return QX_ERR_ARG;  // the array's capacity
    static thread_local ChainParams p;  // large (tens of KB): not on the stack
    qx_status st = marshal_chain(n_jobs, jobs, p);
    if (st != QX_OK) return st;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != QX_OK) return st;
    size_t smem = 0;
    if ((st = chain_geometry(*dev, p, smem)) != QX_OK) return st;
    unsigned* counters = nullptr;
    if ((st = noalloc_counters(&counters)) != QX_OK) return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    // The array keeps whatever the previous call left; the counters must
    // start at zero.
    cudaError_t e = cudaMemsetAsync(counters, 0, size_t(n_jobs + 1) * sizeof(unsigned), cs);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    p.counters = counters;
    e = launch_chain(p, smem, cs);
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "chain launch");
}

qx_status qx_debug_noalloc_fill(uint32_t value, qx_stream_t s) {
    DeviceInfo* dev = nullptr;
    qx_status st = device_info(&dev);
    if (st != QX_OK) return st;
    unsigned* counters = nullptr;
    if ((st = noalloc_counters(&counters)) != QX_OK) return st;
    const unsigned n = kNoallocMaxJobs + 1;
    // a copy from host memory, then a synchronisation: a test hook, not a hot path
    static thread_local unsigned host[kNoallocMaxJobs + 1];
    for (unsigned i = 0; i < n; ++i) host[i] = value;
    const cudaError_t e = cudaMemcpyAsync(counters, host, sizeof(host), cudaMemcpyHostToDevice,
                                          reinterpret_cast<cudaStream_t>(s));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
    const cudaError_t e2 = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s));
    return e2 == cudaSuccess ? QX_OK : cuda_fail(e2, "cudaStreamSynchronize");
}

qx_status qx_debug_trace_read(void* host, size_t bytes) {
    if (!host) return QX_ERR_ARG;
    const cudaError_t e = chain_trace_read(host, bytes);
    return e == cudaSuccess ? QX_OK : cuda_fail(e, "trace read (library built without QX_TRACE?)");
}

}  // extern "C"
