// qx_stage.cuh -- how the GEMV kernels split rows over CTAs and stages
// (shared by the batch-1, small-batch and f32 tensor-pipe kernels), and the
// producer of the row-group kernels: one bulk copy per row, to a padded
// stride (the f32 tensor-pipe kernel calls it; the small-batch kernel keeps
// the same loop inline, where ptxas then spills less at its 96-register
// cap).  sm_103a only.
#pragma once

#include "qx_device.cuh"
#include "qx_internal.h"

namespace qx {

// First row (in the concatenated row space) of CTA i: an even split of the
// rows, rounded down within its entry to a multiple of the alignment quantum.
__device__ __forceinline__ int64_t cta_row_begin(const GemvParams& p, int i) {
    if (i >= p.n_cta) return p.total_rows;
    const int64_t raw = p.total_rows * int64_t(i) / p.n_cta;
    int e = 0;
    while (e + 1 < p.n_entries && raw >= p.e[e + 1].row0) ++e;
    const int64_t local = raw - p.e[e].row0;
    return p.e[e].row0 + (local - local % p.quantum);
}

// Walks one CTA's rows as a sequence of stages: at most G rows, never
// crossing an entry boundary.
struct StageWalker {
    int64_t g, gend;
    int e;
    __device__ __forceinline__ bool next(const GemvParams& p, int& entry, int64_t& lrow, int& nrows) {
        if (g >= gend) return false;
        while (g >= p.e[e].row0 + p.e[e].rows) ++e;
        const int64_t entry_end = p.e[e].row0 + p.e[e].rows;
        const int64_t stop = gend < entry_end ? gend : entry_end;
        const int64_t n = stop - g < p.G ? stop - g : p.G;
        entry = e;
        lrow = g - p.e[e].row0;
        nrows = static_cast<int>(n);
        g += n;
        return true;
    }
};

// Every lane waits on the barrier itself; the outcome is made warp-uniform.
__device__ __forceinline__ bool warp_wait_all(uint64_t* bar, uint32_t parity, uint64_t ns, unsigned* err,
                                              unsigned code) {
    return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, ns, err, code));
}

// The producer warp of the row-group kernels: the CTA's rows [r0, r1) in
// stages of p.G rows, each row copied by one bulk copy (lanes in parallel) to
// slot `k % p.stages` at a stride of row_bytes + 16 bytes, so that the eight
// row groups of an MMA fragment load fall on different banks.  A slot is
// refilled once its `empty` barrier completes (consumers and reducer done).
// Waits are bounded; before returning the warp waits (bounded) for every copy
// it issued, so that no copy lands after the CTA has exited.
__device__ __forceinline__ void produce_padded_rows(const GemvParams& p, int64_t r0, int64_t r1, uint64_t* full,
                                                    uint64_t* empty, uint8_t* smem, int lane) {
    const int S = p.stages;
    const uint64_t policy = policy_evict_first();
    const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
    const int rstride = static_cast<int>(p.row_bytes) + 16;
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
}

}  // namespace qx
