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
// 2-byte word (the GGUF side is 2-byte aligned), consecutive threads on
// consecutive words.
#include <cuda_runtime.h>

#include <cstdint>

#include "qx_internal.h"

namespace qx {

namespace {

constexpr int kRepackThreads = 256;

__global__ void __launch_bounds__(kRepackThreads) repack_q6k_kernel(bool to_soa, const uint8_t* __restrict__ src,
                                                                    int64_t rows, int64_t nsb, int64_t src_rb,
                                                                    uint8_t* __restrict__ dst, int64_t dst_rb) {
    // one thread per 2-byte word of a super-block: words 0..103 are ql, qh and
    // scales, word 104 is d; consecutive threads move consecutive words
    const int64_t i = int64_t(blockIdx.x) * kRepackThreads + threadIdx.x;
    if (i >= rows * nsb * 105) return;
    const int64_t k = i % 105, blk = i / 105;
    const int64_t r = blk / nsb, j = blk % nsb;
    const int64_t gguf = 210 * j + 2 * k;                            // the word in the GGUF row
    const int64_t soa = k < 104 ? 208 * j + 2 * k : 208 * nsb + 2 * j;  // and in the repacked row
    const uint8_t* from = src + r * src_rb + (to_soa ? gguf : soa);
    uint8_t* to = dst + r * dst_rb + (to_soa ? soa : gguf);
    *reinterpret_cast<uint16_t*>(to) = *reinterpret_cast<const uint16_t*>(from);
    if (to_soa && k == 104 && j == nsb - 1)  // the zero padding after the row's d values
        for (int64_t b = 208 * nsb + 2 * nsb; b < dst_rb; ++b) dst[r * dst_rb + b] = 0;
}

}  // namespace

cudaError_t launch_repack_q6k(bool to_soa, const uint8_t* src, int64_t rows, int64_t nsb, int64_t src_row_bytes,
                              uint8_t* dst, int64_t dst_row_bytes, cudaStream_t s) {
    const int64_t n = rows * nsb * 105;
    const int64_t grid = (n + kRepackThreads - 1) / kRepackThreads;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    repack_q6k_kernel<<<static_cast<unsigned>(grid), kRepackThreads, 0, s>>>(to_soa, src, rows, nsb, src_row_bytes,
                                                                               dst, dst_row_bytes);
    return cudaGetLastError();
}

}  // namespace qx
