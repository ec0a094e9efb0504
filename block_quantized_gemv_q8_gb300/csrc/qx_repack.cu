// qx_repack.cu -- load-time repack between the GGUF Q6_K block layout and
// QX_Q6_K_SOA (llamay docs, "Backends and hardware", section "Repacking is a
// per-device decision now": weights are rewritten once, at load, into the
// layout the device's kernels read best).
//
// A GGUF Q6_K super-block is 210 bytes: ql[128], qh[64], scales[16], then d
// (f16).  210-byte blocks put every other super-block on a 2-byte boundary,
// so the GEMV lanes assemble their words with funnel shifts.  QX_Q6_K_SOA
// keeps each super-block's first 208 bytes at 16-byte-aligned offsets 208 j
// of the row and gathers the row's d values after them (at 208 nsb, padded
// with zero bytes to a 16-byte multiple).  Pure data movement: one thread per
// super-block, 2-byte loads and stores (the GGUF side is 2-byte aligned).
#include <cuda_runtime.h>

#include <cstdint>

#include "qx_internal.h"

namespace qx {

namespace {

constexpr int kRepackThreads = 256;

__global__ void __launch_bounds__(kRepackThreads) repack_q6k_kernel(bool to_soa, const uint8_t* __restrict__ src,
                                                                    int64_t rows, int64_t nsb, int64_t src_rb,
                                                                    uint8_t* __restrict__ dst, int64_t dst_rb) {
    const int64_t i = int64_t(blockIdx.x) * kRepackThreads + threadIdx.x;
    if (i >= rows * nsb) return;
    const int64_t r = i / nsb, j = i % nsb;
    const int64_t soa_rb = to_soa ? dst_rb : src_rb;
    // the block's 208 bytes of quants and scales, then d
    const int64_t gguf_off = 210 * j, soa_off = 208 * j, soa_d = 208 * nsb + 2 * j;
    const uint16_t* in = reinterpret_cast<const uint16_t*>(src + r * src_rb + (to_soa ? gguf_off : soa_off));
    uint16_t* out = reinterpret_cast<uint16_t*>(dst + r * dst_rb + (to_soa ? soa_off : gguf_off));
    for (int k = 0; k < 104; ++k) out[k] = in[k];
    const uint16_t d = to_soa ? in[104] : *reinterpret_cast<const uint16_t*>(src + r * src_rb + soa_d);
    if (to_soa) {
        *reinterpret_cast<uint16_t*>(dst + r * dst_rb + soa_d) = d;
        // the padding after the last super-block's d: zero, written by the row's last thread
        if (j == nsb - 1)
            for (int64_t b = 208 * nsb + 2 * nsb; b < soa_rb; ++b) dst[r * dst_rb + b] = 0;
    } else {
        out[104] = d;
    }
}

}  // namespace

cudaError_t launch_repack_q6k(bool to_soa, const uint8_t* src, int64_t rows, int64_t nsb, int64_t src_row_bytes,
                              uint8_t* dst, int64_t dst_row_bytes, cudaStream_t s) {
    const int64_t n = rows * nsb;
    const int64_t grid = (n + kRepackThreads - 1) / kRepackThreads;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    repack_q6k_kernel<<<static_cast<unsigned>(grid), kRepackThreads, 0, s>>>(to_soa, src, rows, nsb, src_row_bytes,
                                                                               dst, dst_row_bytes);
    return cudaGetLastError();
}

}  // namespace qx
