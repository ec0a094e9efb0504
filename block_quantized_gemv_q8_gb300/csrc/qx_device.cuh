// qx_device.cuh -- device-side building blocks shared by the qx kernels:
// mbarriers, 1-D bulk (TMA) copies, bounded waits, programmatic dependent
// launch, and small integer / float helpers.  sm_103a only.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

namespace qx {

// Error bits written to the device error word.
constexpr unsigned kErrTimeoutFull = 1u;   // consumer waited too long for data
constexpr unsigned kErrTimeoutEmpty = 2u;  // producer waited too long for a free slot
constexpr unsigned kErrTimeoutDrain = 4u;  // copies still in flight at exit
constexpr unsigned kErrTimeoutProbe = 8u;  // the test probe's wait ran out
constexpr unsigned kErrTimeoutMma = 16u;   // tensor-core pipeline wait ran out
constexpr unsigned kErrTimeoutChain = 32u; // a chain job waited too long for the previous job

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, for at most
// limit_ns nanoseconds.  On expiry, OR `code` into *err and return false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                                  unsigned* err, unsigned code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) {
            atomicOr(err, code);
            return false;
        }
    }
}

// 1-D bulk copy global -> shared, completion counted on `bar` in bytes.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Same, with an L2 eviction-first hint: streamed weights are read once.
__device__ __forceinline__ void bulk_g2s_evict_first(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                                     uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Programmatic dependent launch: wait until the preceding grid in the stream
// has completed and its memory is visible; let the next grid start launching.
__device__ __forceinline__ void pdl_wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// dp4a with the bytes of `a` unsigned (0..255) and the bytes of `b` signed.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Quantisation of an activation to int8 per block of 32 (llamay docs,
// "Backends and hardware", section "CPU": the activation is quantised to int8
// once per matmul):
//   d = amax / 127 (IEEE round-to-nearest f32 division),
//   q = round-half-even(fl(x / d)) with fl(x / d) the correctly rounded f32
//       quotient, clamped to [-127, 127]; q = 0 when d == 0;
//   sum = sum of the 32 quants.
// Every kernel that quantises an activation goes through the functions
// below, so their codes are identical.
//
// Rounding fl(x / d) without dividing: t = fl(x * fl(1 / d)) differs from
// fl(x / d) by at most 3 * 2^-24 * |x / d| (three roundings of relative size
// <= 2^-24), below 2.3e-5 when |t| <= 128.  When t lies farther than 2^-14
// from every half-integer, fl(x / d) rounds to the same integer as t does.
// Values that fail this test (about one in 10^4, and all values when 1 / d
// overflows) take the correctly rounded quotient from __fdiv_rn instead.
__device__ __forceinline__ bool quotient_rounding_is_safe(float t, float k) {
    return fabsf(t) <= 128.0f && 0.5f - fabsf(t - k) > 6.103515625e-05f;
}

// Quantise N consecutive values of one block (N = 32 / threads per block);
// amax over the block and the block's quant sum are combined across the
// THREADS adjacent lanes that share the block (THREADS a power of two <= 32,
// all lanes of the warp taking part).  A lane with live == false takes part in
// the shuffles only and stores nothing; the lane holding the block's first
// values (first == true) stores d and sum.
template <int N>
__device__ __forceinline__ void load_block_part(const float* __restrict__ x, float (&v)[N]) {
    const float4* src = reinterpret_cast<const float4*>(x);
#pragma unroll
    for (int k = 0; k < N / 4; ++k) {
        const float4 f = src[k];
        v[4 * k + 0] = f.x;
        v[4 * k + 1] = f.y;
        v[4 * k + 2] = f.z;
        v[4 * k + 3] = f.w;
    }
}

template <int N, int THREADS>
__device__ __forceinline__ void quantize_block_values(const float (&v)[N], int8_t* __restrict__ q, float* d,
                                                      int32_t* sum, bool live, bool first) {
    static_assert(N * THREADS == 32 && N % 4 == 0, "a block is 32 values, stored in 4-byte groups");
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int o = 1; o < THREADS; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float db = __fdiv_rn(amax, 127.0f);
    float r[N];
    if (db != 0.0f) {
        const float rcp = __frcp_rn(db);
        bool safe = true;
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float t = v[i] * rcp;
            r[i] = rintf(t);
            safe &= quotient_rounding_is_safe(t, r[i]);
        }
        if (!safe) {  // rare: some quotient lies too close to a rounding boundary
#pragma unroll
            for (int i = 0; i < N; ++i) r[i] = rintf(__fdiv_rn(v[i], db));
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) r[i] = 0.0f;
    }
    // |x / d| <= 127 (1 + 2^-23) for every x of the block, so every code is
    // already within [-127, 127]: the clamp of the definition never binds.
    uint32_t packed[N / 4];
    int s = 0;
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
        const int q0 = static_cast<int>(r[4 * j]), q1 = static_cast<int>(r[4 * j + 1]);
        const int q2 = static_cast<int>(r[4 * j + 2]), q3 = static_cast<int>(r[4 * j + 3]);
        const uint32_t lo = __byte_perm(uint32_t(q0), uint32_t(q1), 0x0040u);  // bytes q0, q1
        const uint32_t hi = __byte_perm(uint32_t(q2), uint32_t(q3), 0x0040u);  // bytes q2, q3
        packed[j] = __byte_perm(lo, hi, 0x5410u);
        s = __dp4a(static_cast<int>(packed[j]), 0x01010101, s);  // + q0 + q1 + q2 + q3 (signed bytes)
    }
#pragma unroll
    for (int o = 1; o < THREADS; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (live) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(q);
#pragma unroll
        for (int j = 0; j < N / 4; ++j) dst[j] = packed[j];
        if (first) {
            *d = db;
            *sum = s;
        }
    }
}

template <int N, int THREADS>
__device__ __forceinline__ void quantize_block_part(const float* __restrict__ x, int8_t* __restrict__ q,
                                                    float* d, int32_t* sum, bool live, bool first) {
    float v[N];
    load_block_part<N>(x, v);
    quantize_block_values<N, THREADS>(v, q, d, sum, live, first);
}

// Quantise blocks [0, nblocks) with two adjacent lanes per block, 16 values
// each: `task` runs over 2 * nblocks in rounds of `stride` (a multiple of 32),
// and every lane calls this the same number of times.  x, q: 16-byte aligned.
// With `swz`, the 16-byte chunk G of q is stored at chunk G ^ ((G / 8) % 8):
// the chunks of each 128-byte slice are permuted by the slice's index, so
// that 32 lanes reading their slices chunk by chunk hit distinct banks
// (act_chunk_swizzle gives the inverse for the reader).
__device__ __forceinline__ int64_t act_chunk_swizzle(int64_t chunk) { return chunk ^ ((chunk >> 3) & 7); }

__device__ __forceinline__ void quantize_task(const float* __restrict__ x, int64_t nblocks, int64_t task,
                                              int8_t* __restrict__ q, float* d, int32_t* sum, bool swz = false) {
    const bool live = task < 2 * nblocks;
    const int64_t b = live ? task >> 1 : nblocks - 1;
    const int half = static_cast<int>(task & 1);
    const int64_t chunk = 2 * b + half;
    quantize_block_part<16, 2>(x + b * 32 + half * 16, q + 16 * (swz ? act_chunk_swizzle(chunk) : chunk), d + b,
                               sum + b, live, half == 0);
}

// fp16 bit pattern -> f32 (exact; subnormals kept).
__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// 32-bit word at byte address p (p 2-byte aligned) in shared memory, built from
// the two aligned words around it.
__device__ __forceinline__ uint32_t lds_u32_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    return __funnelshift_r(w[0], w[1], sh);
}

}  // namespace qx
