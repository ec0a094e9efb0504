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

// Packed pairs of f32 (two lanes of one 64-bit register) and the sm_103a
// two-wide f32 add and fused multiply-add on them (each element rounded as
// its scalar counterpart).
__device__ __forceinline__ uint64_t f32x2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float2 f32x2_unpack(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
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
//
// The integer itself comes from the magic-number form of round-half-even:
// for |t| < 2^22, fl(t + 1.5 * 2^23) = 1.5 * 2^23 + rne(t) exactly (the sum
// lies in [2^23, 2^24), where the spacing of floats is 1), so subtracting
// 1.5 * 2^23 again gives rne(t) and t - rne(t) exactly, and the low byte of
// the sum's bit pattern is rne(t) as a two's-complement byte (the pattern of
// 1.5 * 2^23 has a zero low byte).  |x| <= amax for every x of the block, so
// the largest |t| is fl(amax * fl(1 / d)): one range check per block.
//
// The clamp binds only when d is an f32 subnormal: then d = fl(amax / 127)
// may carry a relative error far above 2^-24 (d = 2^-149 for amax = 178 *
// 2^-149 gives x / d = 178).  The fast path is taken only when
// fl(amax * fl(1 / d)) < 127.5, so all of its codes lie in [-127, 127]
// already; every other block (all blocks with 1 / d overflowing among them)
// takes the exact quotient and clamps it.
constexpr float kMagicRne = 12582912.0f;            // 1.5 * 2^23
constexpr float kTieMargin = 0.49993896484375f;     // 0.5 - 2^-14

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
    float m[N];
#pragma unroll
    for (int i = 0; i < N; ++i) m[i] = fabsf(v[i]);
#pragma unroll
    for (int w = N / 2; w >= 1; w >>= 1)  // max is exact: a tree gives the same amax
#pragma unroll
        for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    float amax = m[0];
#pragma unroll
    for (int o = 1; o < THREADS; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float db = __fdiv_rn(amax, 127.0f);
    uint32_t bits[N];  // low byte: the code
    if (db != 0.0f) {
        const float rcp = __frcp_rn(db);
        bool safe = amax * rcp < 127.5f;
        const uint64_t rcp2 = f32x2_pack(rcp, rcp);
        const uint64_t magic2 = f32x2_pack(kMagicRne, kMagicRne), unmagic2 = f32x2_pack(-kMagicRne, -kMagicRne);
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const uint64_t t2 = f32x2_mul(f32x2_pack(v[i], v[i + 1]), rcp2);
            const uint64_t m2 = f32x2_add(t2, magic2);           // 1.5 * 2^23 + rne(t)
            const float2 e = f32x2_unpack(f32x2_sub(t2, f32x2_add(m2, unmagic2)));  // t - rne(t)
            safe &= fabsf(e.x) < kTieMargin && fabsf(e.y) < kTieMargin;
            const float2 mm = f32x2_unpack(m2);
            bits[i] = __float_as_uint(mm.x);
            bits[i + 1] = __float_as_uint(mm.y);
        }
        if (!safe) {  // rare: a quotient near a rounding boundary, or a subnormal d
#pragma unroll
            for (int i = 0; i < N; ++i)
                bits[i] = __float_as_uint(fminf(fmaxf(rintf(__fdiv_rn(v[i], db)), -127.0f), 127.0f) + kMagicRne);
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) bits[i] = 0u;
    }
    uint32_t packed[N / 4];
    int s = 0;
#pragma unroll
    for (int j = 0; j < N / 4; ++j) {
        const uint32_t lo = __byte_perm(bits[4 * j], bits[4 * j + 1], 0x0040u);      // codes 0, 1
        const uint32_t hi = __byte_perm(bits[4 * j + 2], bits[4 * j + 3], 0x0040u);  // codes 2, 3
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

// Tasks task0 + r * stride (r < R) with every load issued before any
// arithmetic, so that R rounds cost one memory round trip.  Same codes as
// quantize_task.
template <int R>
__device__ __forceinline__ void quantize_tasks(const float* __restrict__ x, int64_t nblocks, int64_t task0,
                                               int64_t stride, int8_t* __restrict__ q, float* d, int32_t* sum,
                                               bool swz) {
    float v[R][16];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t task = task0 + r * stride;
        const int64_t b = task < 2 * nblocks ? task >> 1 : nblocks - 1;
        load_block_part<16>(x + b * 32 + (task & 1) * 16, v[r]);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int64_t task = task0 + r * stride;
        const bool live = task < 2 * nblocks;
        const int64_t b = live ? task >> 1 : nblocks - 1;
        const int half = static_cast<int>(task & 1);
        const int64_t chunk = 2 * b + half;
        quantize_block_values<16, 2>(v[r], q + 16 * (swz ? act_chunk_swizzle(chunk) : chunk), d + b, sum + b, live,
                                     half == 0);
    }
}

// Every task of an activation of `nblocks` blocks over `threads` threads
// (thread t takes tasks t, t + threads, ...; every thread of the group calls
// this), the loads of up to RMAX rounds in flight at once (RMAX <= 4: each
// round holds 16 values in registers).
template <int RMAX>
__device__ __forceinline__ void quantize_all(const float* __restrict__ x, int64_t nblocks, int t, int threads,
                                             int8_t* __restrict__ q, float* d, int32_t* sum, bool swz) {
    static_assert(RMAX >= 1 && RMAX <= 4, "one to four rounds per batch");
    int rounds = static_cast<int>((2 * nblocks + threads - 1) / threads);
    int64_t base = t;
    while (rounds > 0) {
        const int r = rounds < RMAX ? rounds : RMAX;
        if (RMAX >= 4 && r == 4) quantize_tasks<(RMAX >= 4 ? 4 : 1)>(x, nblocks, base, threads, q, d, sum, swz);
        else if (RMAX >= 3 && r == 3) quantize_tasks<(RMAX >= 3 ? 3 : 1)>(x, nblocks, base, threads, q, d, sum, swz);
        else if (RMAX >= 2 && r == 2) quantize_tasks<(RMAX >= 2 ? 2 : 1)>(x, nblocks, base, threads, q, d, sum, swz);
        else quantize_tasks<1>(x, nblocks, base, threads, q, d, sum, swz);
        base += int64_t(r) * threads;
        rounds -= r;
    }
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
