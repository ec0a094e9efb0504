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

constexpr int kActq8Threads = 128;

// Two adjacent lanes per block of 32 values.
__global__ void __launch_bounds__(kActq8Threads) actq8_kernel(const float* __restrict__ x, int64_t nblocks,
                                                               int8_t* __restrict__ q, float* __restrict__ d,
                                                               int32_t* __restrict__ sum) {
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    const int64_t stride = int64_t(gridDim.x) * kActq8Threads;
    for (int64_t base = 0; base < 2 * nblocks; base += stride)
        quantize_task(x, nblocks, base + int64_t(blockIdx.x) * kActq8Threads + threadIdx.x, q, d, sum);
}

cudaError_t launch_actq8(const float* x, int64_t nblocks, int8_t* q, float* d, int32_t* sum, int sm_count,
                         cudaStream_t s) {
    int64_t grid = (2 * nblocks + kActq8Threads - 1) / kActq8Threads;
    if (grid > int64_t(sm_count) * 8) grid = int64_t(sm_count) * 8;
    // Launched with programmatic stream serialisation: the CTAs may become
    // resident while the previous kernel in the stream drains, and the wait at
    // the top of the kernel keeps every read of x and write of q, d, sum after
    // that kernel has completed, so the order is the plain stream order.  A
    // following W4A8 GEMV launched with QX_FLAG_PDL then starts streaming its
    // weights during this launch.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kActq8Threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, actq8_kernel, x, nblocks, q, d, sum);
}

}  // namespace qx
