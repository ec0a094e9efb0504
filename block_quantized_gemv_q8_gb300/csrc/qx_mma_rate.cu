// qx_mma_rate.cu -- measured warp-level tensor-core rates on this device, the
// context for the prefill numbers: sm_103a has no int8 tcgen05 MMA
// (kind::i8), so the int8 rate available to a prefill is the legacy
// mma.sync one.  Each warp runs eight independent accumulators through a
// fixed number of mma.sync steps on register operands (no memory traffic in
// the loop); the rate is the multiply-adds x 2 over the CUDA-event time of
// the launch.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/qx.h"
#include "../../include/qx_debug.h"

namespace qx {

namespace {

constexpr int kRateWarps = 8;
constexpr int kRateIters = 4096;

template <int KIND>
__global__ void __launch_bounds__(kRateWarps * 32) mma_rate_kernel(uint32_t seed, int* out) {
    uint32_t A[4], B[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) A[i] = seed * (threadIdx.x + 7 * i + 1);
#pragma unroll
    for (int i = 0; i < 2; ++i) B[i] = seed ^ (threadIdx.x * 13 + i);
    int C[8][4] = {};
    float F[8][4] = {};
    for (int it = 0; it < kRateIters; ++it) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (KIND == 0)
                asm volatile(
                    "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+r"(C[j][0]), "+r"(C[j][1]), "+r"(C[j][2]), "+r"(C[j][3])
                    : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(B[0]), "r"(B[1]));
            else
                asm volatile(
                    "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
                    "{%0,%1,%2,%3};"
                    : "+f"(F[j][0]), "+f"(F[j][1]), "+f"(F[j][2]), "+f"(F[j][3])
                    : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(B[0]), "r"(B[1]));
        }
    }
    int s = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) s += C[j][i] + static_cast<int>(F[j][i]);
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;  // keeps the results live
}

}  // namespace
}  // namespace qx

using namespace qx;

extern "C" qx_status qx_debug_mma_rate(int kind, double* ops_per_s, qx_stream_t s) {
    if (!ops_per_s || (kind != 0 && kind != 1)) return QX_ERR_ARG;
    int dev = 0, sms = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return QX_ERR_CUDA;
    if (major != 10 || minor != 3) return QX_ERR_UNSUPPORTED_DEVICE;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(s);
    int* out = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    qx_status rc = QX_ERR_CUDA;
    float ms = 0.0f;
    if (cudaMalloc(&out, size_t(sms) * kRateWarps * 32 * sizeof(int)) != cudaSuccess) return QX_ERR_CUDA;
    if (cudaEventCreate(&e0) == cudaSuccess && cudaEventCreate(&e1) == cudaSuccess) {
        bool ok = true;
        for (int rep = 0; rep < 2 && ok; ++rep) {  // the first launch warms up
            ok = cudaEventRecord(e0, st) == cudaSuccess;
            if (kind == 0) mma_rate_kernel<0><<<sms, kRateWarps * 32, 0, st>>>(0x01020304u, out);
            else mma_rate_kernel<1><<<sms, kRateWarps * 32, 0, st>>>(0x3c003c00u, out);
            ok = ok && cudaGetLastError() == cudaSuccess && cudaEventRecord(e1, st) == cudaSuccess &&
                 cudaEventSynchronize(e1) == cudaSuccess && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess;
        }
        if (ok && ms > 0.0f) {
            const double macs_per_mma = kind == 0 ? 16.0 * 8 * 32 : 16.0 * 8 * 16;
            const double macs = double(sms) * kRateWarps * kRateIters * 8 * macs_per_mma;
            *ops_per_s = 2.0 * macs / (double(ms) * 1e-3);
            rc = QX_OK;
        }
    }
    if (e0) cudaEventDestroy(e0);
    if (e1) cudaEventDestroy(e1);
    cudaFree(out);
    return rc;
}
