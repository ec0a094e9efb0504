// qx_actq8.cu -- activation quantisation to int8 per block of 32.
//
// llamay docs, "Backends and hardware", section "CPU": in the W4A8 fused dot
// product the activation is quantised to int8 once per matmul.  Per block of
// 32 values: d = amax / 127, q = round-half-even(x / d) clamped to
// [-127, 127] (q = 0 when d == 0), and the block sum of q, which the Q4_K
// min term needs.  Division and rounding are IEEE round-to-nearest-even in
// f32, so the quants are reproducible bit for bit.
#include "qx_device.cuh"
#include "qx_internal.h"

namespace qx {

constexpr int kActq8Threads = 256;

// One warp per block of 32 values, one value per lane.
__global__ void __launch_bounds__(kActq8Threads) actq8_kernel(const float* __restrict__ x, int64_t nblocks,
                                                               int8_t* __restrict__ q, float* __restrict__ d,
                                                               int32_t* __restrict__ sum) {
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (kActq8Threads / 32);
    for (int64_t b = int64_t(blockIdx.x) * (kActq8Threads / 32) + (threadIdx.x >> 5); b < nblocks; b += warps) {
        const float v = x[b * 32 + lane];
        float amax = fabsf(v);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float db = __fdiv_rn(amax, 127.0f);
        int qi = 0;
        if (db != 0.0f) {
            const float r = rintf(__fdiv_rn(v, db));
            qi = static_cast<int>(fminf(fmaxf(r, -127.0f), 127.0f));
        }
        q[b * 32 + lane] = static_cast<int8_t>(qi);
        const int s = __reduce_add_sync(0xffffffffu, qi);
        if (lane == 0) {
            d[b] = db;
            sum[b] = s;
        }
    }
}

cudaError_t launch_actq8(const float* x, int64_t nblocks, int8_t* q, float* d, int32_t* sum, int sm_count,
                         cudaStream_t s) {
    const int64_t want = (nblocks + (kActq8Threads / 32) - 1) / (kActq8Threads / 32);
    const int grid = static_cast<int>(want < int64_t(sm_count) * 8 ? want : int64_t(sm_count) * 8);
    actq8_kernel<<<grid, kActq8Threads, 0, s>>>(x, nblocks, q, d, sum);
    return cudaGetLastError();
}

}  // namespace qx
