// qx_tc.cu -- the prefill contraction on the fifth-generation tensor cores
// (tcgen05 MMA, accumulator in tensor memory, operands staged by TMA).
//
// The W4A8 prefill product (llamay docs, "Backends and hardware", sections
// "CPU" and "CUDA") is Y[m, n] = sum_k xhat[m, k] * what[n, k] with
// xhat = dx * q_x (the dequantised int8 activation) and what the dequantised
// weight (Q4_K: d*sc*q - dmin*m, Q6_K: d*sc*(q - 32), Q8_0: d*q).  sm_103a has
// no integer tensor-core MMA, and the per-sub-block scales differ along K, so
// the integer partial sums cannot be scaled inside the MMA accumulation.
// Instead each operand is written once as two bf16 terms whose sum carries 16
// significant bits (hi = bf16(v), lo = bf16(v - hi)), and
//     Y = Xh Wh^T + Xh Wl^T + Xl Wh^T
// is one bf16 GEMM over three passes of K, accumulated in f32 in tensor
// memory.  The dropped Xl Wl^T term and the split truncation bound the error
// of every product by about 2^-15 of |xhat * what|, well inside the tolerance
// of 1e-4 * sum |w * x| per output.
//
// Kernels:
//   * Q4_K: the activation is split by a small pass; the weight terms are
//     formed inside the GEMM (tc_q4k_fused_kernel): TMA brings the raw
//     super-blocks of 128 weight rows into shared memory, 16 converter warps
//     dequantise each 64-wide K slice and write Wh / Wl directly in the
//     128-byte-swizzled K-major layout the tensor cores read, and one thread
//     issues the three split products per slice (M = 128, N = 128, K = 16).
//   * Q6_K, Q8_0: a dequantise-and-split pass per operand (memory-bound),
//     then tc_gemm_kernel: 128 x 256 tiles over three passes of K.
// In both, warp 0 issues the TMA loads, warp 1 owns the tensor memory and
// issues tcgen05.mma from one thread, and four warps drain the accumulator
// with tcgen05.ld.  Every wait is bounded and reports through the device
// error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "qx_device.cuh"
#include "qx_internal.h"

namespace qx {

namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kTcThreads = 192;
constexpr size_t kTcSmem = size_t(STAGES) * STAGE_BYTES + 1024 + 256;

struct TcParams {
    CUtensorMap a_map[2];  // Xh, Xl: [M, K] bf16
    CUtensorMap b_map[2];  // Wh, Wl: [N, K] bf16
    int M, N, K;
    float* Y;  // [M, N] f32
    unsigned* err;
    unsigned long long wait_ns;
};

// ---------------------------------------------------------------------------
// dequantise and split
// ---------------------------------------------------------------------------

__device__ __forceinline__ void split_store(const float (&w)[32], uint16_t* hi, uint16_t* lo) {
    uint32_t h[16], l[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(w[2 * i]), h1 = __float2bfloat16_rn(w[2 * i + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(w[2 * i] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(w[2 * i + 1] - __bfloat162float(h1));
        h[i] = uint32_t(__bfloat16_as_ushort(h0)) | (uint32_t(__bfloat16_as_ushort(h1)) << 16);
        l[i] = uint32_t(__bfloat16_as_ushort(l0)) | (uint32_t(__bfloat16_as_ushort(l1)) << 16);
    }
    uint4* hp = reinterpret_cast<uint4*>(hi);
    uint4* lp = reinterpret_cast<uint4*>(lo);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        hp[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
        lp[i] = make_uint4(l[4 * i], l[4 * i + 1], l[4 * i + 2], l[4 * i + 3]);
    }
}

__device__ __forceinline__ float f16_at(const uint8_t* p) {
    return __half2float(__ushort_as_half(uint16_t(p[0] | (uint16_t(p[1]) << 8))));
}

// One thread per (row, group of 32 weights).  Q4_K (GGUF layout): d, dmin,
// 12 bytes of 6-bit scales and mins, 128 bytes of nibbles; group j of a super-
// block is sub-block j.  Q6_K: group = quarter t of half h; Q8_0: group = block.
template <int FMT>
__global__ void __launch_bounds__(256) dequant_w_kernel(const uint8_t* __restrict__ W, int64_t N, int64_t K,
                                                        int64_t row_bytes, uint16_t* __restrict__ Wh,
                                                        uint16_t* __restrict__ Wl) {
    const int64_t groups = K / 32;
    const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= N * groups) return;
    const int64_t n = t / groups, g = t % groups;
    const uint8_t* row = W + n * row_bytes;
    float w[32];
    if constexpr (FMT == QX_Q4_K) {
        const uint8_t* b = row + (g / 8) * 144;
        const int j = int(g % 8);
        const float d = f16_at(b), dmin = f16_at(b + 2);
        const uint8_t* s = b + 4;
        int sc, m;
        if (j < 4) {
            sc = s[j] & 63;
            m = s[j + 4] & 63;
        } else {
            sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
        const float a = d * float(sc), c = dmin * float(m);  // exact products
        const uint8_t* qs = b + 16 + 32 * (j / 2);
        const int sh = 4 * (j & 1);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = fmaf(a, float((qs[i] >> sh) & 15), -c);
    } else if constexpr (FMT == QX_Q6_K) {
        const uint8_t* b = row + (g / 8) * 210;
        const int q8 = int(g % 8), h = q8 / 4, tq = q8 % 4;
        const float d = f16_at(b + 208);
        const uint8_t* ql = b + 64 * h + 32 * (tq & 1);
        const uint8_t* qh = b + 128 + 32 * h;
        const int8_t* sc = reinterpret_cast<const int8_t*>(b + 192 + 8 * h);
        const int nsh = (tq >= 2) ? 4 : 0;
        const float s0 = d * float(sc[2 * tq]), s1 = d * float(sc[2 * tq + 1]);  // l < 16, l >= 16
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int q = ((ql[i] >> nsh) & 15) | (((qh[i] >> (2 * tq)) & 3) << 4);
            w[i] = (i < 16 ? s0 : s1) * float(q - 32);
        }
    } else {
        const uint8_t* b = row + g * 34;
        const float d = f16_at(b);
        const int8_t* q = reinterpret_cast<const int8_t*>(b + 2);
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = d * float(q[i]);
    }
    split_store(w, Wh + n * K + 32 * g, Wl + n * K + 32 * g);
}

// xhat = dx * q_x per block of 32, split into two bf16 terms.
__global__ void __launch_bounds__(256) dequant_x_kernel(const int8_t* __restrict__ q, const float* __restrict__ d,
                                                        int64_t M, int64_t K, uint16_t* __restrict__ Xh,
                                                        uint16_t* __restrict__ Xl) {
    const int64_t groups = K / 32;
    const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= M * groups) return;
    const float dx = d[t];
    const int8_t* qp = q + 32 * t;
    float w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = dx * float(qp[i]);
    split_store(w, Xh + 32 * t, Xl + 32 * t);
}

// ---------------------------------------------------------------------------
// tcgen05 GEMM
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor of a K-major tile with the 128-byte swizzle
// written by TMA: rows of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFF) >> 4);  // start address
    d |= uint64_t(1) << 16;                  // leading byte offset (unused for swizzled K-major)
    d |= uint64_t(1024 >> 4) << 32;          // stride byte offset: one 8-row atom
    d |= uint64_t(1) << 46;                  // descriptor version
    d |= uint64_t(2) << 61;                  // 128-byte swizzle
    return d;
}
// Instruction descriptor, kind::f16: f32 accumulator, bf16 A and B, both
// K-major, M = 128, N = 256.
constexpr uint32_t kIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}
// Every lane of the warp waits on the barrier itself (so each observes the
// completed phase), and the outcome is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned long long ns, unsigned* err,
                                          unsigned code) {
    const bool ok = mbar_wait_bounded(bar, parity, ns, err, code);
    return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// blockIdx.x: M tile (fastest, so the CTAs that share a weight tile run
// together and read it from DRAM once), blockIdx.y: N tile.
__global__ void __launch_bounds__(kTcThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw & 1023)) & 1023);  // 1024-byte aligned stages
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int kt_per_pass = (p.K + BK - 1) / BK, n_iters = 3 * kt_per_pass;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: pass 0 = (Xh, Wh), 1 = (Xh, Wl), 2 = (Xl, Wh)
        int issued = 0;
        for (int it = 0; it < n_iters; ++it) {
            const int s = it % STAGES;
            if (it >= STAGES &&
                !mbar_wait_bounded(&empty[s], ((it / STAGES) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                break;
            const int pass = it / kt_per_pass, kt = it % kt_per_pass;
            uint8_t* a_s = smem + s * STAGE_BYTES;
            mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
            tma_load_2d(a_s, &p.a_map[pass == 2 ? 1 : 0], kt * BK, m0, &full[s]);
            tma_load_2d(a_s + A_BYTES, &p.b_map[pass == 1 ? 1 : 0], kt * BK, n0, &full[s]);
            issued = it + 1;
        }
        // keep the CTA alive until every copy it issued has landed
        for (int it = issued > STAGES ? issued - STAGES : 0; it < issued; ++it)
            mbar_wait_bounded(&full[it % STAGES], (it / STAGES) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer
        for (int it = 0; it < n_iters; ++it) {
            const int s = it % STAGES;
            if (!mbar_wait_bounded(&full[s], (it / STAGES) & 1, p.wait_ns, p.err, kErrTimeoutMma)) break;
            tc_fence_after();
            const uint32_t a_s = smem_addr(smem + s * STAGE_BYTES);
            const uint64_t ad = sw128_desc(a_s), bd = sw128_desc(a_s + A_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)  // K = 16 per MMA: 32 bytes further along the swizzled row
                tc_mma(tmem, ad + uint64_t(2 * k), bd + uint64_t(2 * k), kIdesc, (it | k) != 0 ? 1u : 0u);
            tc_commit(&empty[s]);
        }
        tc_commit(acc_full);  // also after a failed wait: arrives once the issued MMAs are done
    } else if (warp >= 2) {
        // ---- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        if (warp_wait(acc_full, 0, p.wait_ns, p.err, kErrTimeoutMma)) {
            tc_fence_after();
            const int q = warp & 3;
            const int row = m0 + 32 * q + lane;
            const bool row_ok = row < p.M;
            const bool vec = (n0 + BN <= p.N) && (p.N % 4 == 0);
            float* yrow = p.Y + size_t(row_ok ? row : 0) * p.N + n0;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t v[32];
                tc_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(32 * c), v);
                if (!row_ok) continue;
                if (vec) {
                    float4* dst = reinterpret_cast<float4*>(yrow + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (n0 + 32 * c + i < p.N) yrow[32 * c + i] = __uint_as_float(v[i]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(BN) : "memory");
}

// ---------------------------------------------------------------------------
// fused Q4_K GEMM: the weight operand is dequantised and split inside the
// kernel, from the raw super-blocks, straight into the swizzled tiles
// ---------------------------------------------------------------------------

constexpr int FBM = 128, FBN = 128, FBK = 64;
constexpr int X_STAGES = 3, W_STAGES = 2, RAW_SLOTS = 3;
constexpr int F_TILE = FBM * FBK * 2;                 // one 128 x 64 bf16 tile: 16 KB
constexpr int F_PAIR = 2 * F_TILE;                    // hi and lo tiles of one operand
constexpr int F_RAW_BYTES = FBN * 144;                // 128 rows of one Q4_K super-block
constexpr int kConvWarps = 16;                        // converter warps; the first four drain the accumulator
constexpr int kFusedThreads = 32 * (2 + kConvWarps);
constexpr size_t kFusedSmem =
    size_t(X_STAGES + W_STAGES) * F_PAIR + size_t(RAW_SLOTS) * F_RAW_BYTES + 1024 + 256;
static_assert(F_RAW_BYTES % 1024 == 0, "raw slots keep the 1024-byte alignment");
constexpr uint32_t kIdescF =
    (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(FBN >> 3) << 17) | (uint32_t(FBM >> 4) << 24);

struct FusedParams {
    CUtensorMap x_map[2];  // Xh, Xl: [M, K] bf16, boxes 64 x 128, 128-byte swizzle
    CUtensorMap w_map;     // Q4_K rows as bytes [N, row_bytes], boxes 144 x 128
    int M, N, K;
    float* Y;
    unsigned* err;
    unsigned long long wait_ns;
};

// One row's quarter of a 64-wide K slice (chunk c of the super-block): 16
// weights of sub-block 2c + half, the column groups 4 half + g0 and
// 4 half + g0 + 1 (g0 = 0 or 2), dequantised and split into hi and lo bf16.
// The sub-block's weights are the low nibbles (half 0) or high nibbles
// (half 1) of the chunk's 32 quant bytes.
__device__ __forceinline__ void q4k_convert_quarter(const uint8_t* rawrow, int c, int half, int g0, uint4 (&hi)[2],
                                                    uint4 (&lo)[2]) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(rawrow);
    const uint4 qv = *reinterpret_cast<const uint4*>(rawrow + 16 + 32 * c + 8 * g0);
    const float d = __half2float(__ushort_as_half(uint16_t(hdr.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(uint16_t(hdr.x >> 16)));
    const int sub = 2 * c + half;
    int sc, m;
    if (sub < 4) {
        sc = (hdr.y >> (8 * sub)) & 63;
        m = (hdr.z >> (8 * sub)) & 63;
    } else {
        const int u = sub - 4;
        sc = ((hdr.w >> (8 * u)) & 15) | (((hdr.y >> (8 * u + 6)) & 3) << 4);
        m = ((hdr.w >> (8 * u + 4)) & 15) | (((hdr.z >> (8 * u + 6)) & 3) << 4);
    }
    const float a = d * float(sc), cm = dmin * float(m);  // exact products
    const uint32_t sh = 4u * uint32_t(half);
    // the nibbles of this half, one per byte
    const uint32_t nb[4] = {(qv.x >> sh) & 0x0F0F0F0Fu, (qv.y >> sh) & 0x0F0F0F0Fu, (qv.z >> sh) & 0x0F0F0F0Fu,
                            (qv.w >> sh) & 0x0F0F0F0Fu};
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        uint32_t h[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t word = nb[2 * g + (i >> 1)];
            const int b0 = 2 * (i & 1);
            const float w0 = fmaf(a, float((word >> (8 * b0)) & 0xFFu), -cm);
            const float w1 = fmaf(a, float((word >> (8 * b0 + 8)) & 0xFFu), -cm);
            const __nv_bfloat162 hb = __floats2bfloat162_rn(w0, w1);
            const float2 hf = __bfloat1622float2(hb);
            const __nv_bfloat162 lb = __floats2bfloat162_rn(w0 - hf.x, w1 - hf.y);
            h[i] = *reinterpret_cast<const uint32_t*>(&hb);
            l[i] = *reinterpret_cast<const uint32_t*>(&lb);
        }
        hi[g] = make_uint4(h[0], h[1], h[2], h[3]);
        lo[g] = make_uint4(l[0], l[1], l[2], l[3]);
    }
}

// blockIdx.x: M tile (fastest), blockIdx.y: N tile.  Warp 0: TMA producer
// (activation tiles per K step, raw super-blocks two ahead); warp 1: tensor
// memory and the MMA issuer (three split products per K slice); warps 2-17:
// convert raw super-blocks into the Wh / Wl tiles; warps 2-5 then drain the
// accumulator (warp w reads tensor-memory lanes 32 (w % 4) .. + 31).
__global__ void __launch_bounds__(kFusedThreads, 1) tc_q4k_fused_kernel(const __grid_constant__ FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t rawaddr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (rawaddr & 1023)) & 1023);
    uint8_t* xst = smem;                                     // [X_STAGES][Xh, Xl]
    uint8_t* wst = xst + X_STAGES * F_PAIR;                  // [W_STAGES][Wh, Wl]
    uint8_t* raw = wst + W_STAGES * F_PAIR;                  // [RAW_SLOTS][128 rows x 144 bytes]
    uint64_t* full_x = reinterpret_cast<uint64_t*>(raw + RAW_SLOTS * F_RAW_BYTES);
    uint64_t* empty_x = full_x + X_STAGES;
    uint64_t* full_w = empty_x + X_STAGES;
    uint64_t* empty_w = full_w + W_STAGES;
    uint64_t* full_raw = empty_w + W_STAGES;
    uint64_t* empty_raw = full_raw + RAW_SLOTS;
    uint64_t* acc_full = empty_raw + RAW_SLOTS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * FBM, n0 = blockIdx.y * FBN;
    const int n_k = p.K / FBK, n_sb = p.K / 256;

    if (threadIdx.x == 0) {
        for (int s = 0; s < X_STAGES; ++s) {
            mbar_init(&full_x[s], 1);
            mbar_init(&empty_x[s], 1);
        }
        for (int s = 0; s < W_STAGES; ++s) {
            mbar_init(&full_w[s], kConvWarps);
            mbar_init(&empty_w[s], 1);
        }
        for (int r = 0; r < RAW_SLOTS; ++r) {
            mbar_init(&full_raw[r], 1);
            mbar_init(&empty_raw[r], kConvWarps);
        }
        mbar_init(acc_full, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(FBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ---- producer: activation tiles per K slice, raw super-blocks two ahead
        int x_issued = 0, raw_issued = 0;
        auto issue_raw = [&](int sb) {
            const int r = sb % RAW_SLOTS;
            if (sb >= RAW_SLOTS &&
                !mbar_wait_bounded(&empty_raw[r], ((sb / RAW_SLOTS) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                return false;
            mbar_arrive_expect_tx(&full_raw[r], F_RAW_BYTES);
            tma_load_2d(raw + r * F_RAW_BYTES, &p.w_map, sb * 144, n0, &full_raw[r]);
            raw_issued = sb + 1;
            return true;
        };
        bool ok = issue_raw(0);
        if (ok && n_sb > 1) ok = issue_raw(1);
        for (int t = 0; t < n_k && ok; ++t) {
            const int s = t % X_STAGES;
            if (t >= X_STAGES &&
                !mbar_wait_bounded(&empty_x[s], ((t / X_STAGES) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                break;
            uint8_t* st = xst + s * F_PAIR;
            mbar_arrive_expect_tx(&full_x[s], F_PAIR);
            tma_load_2d(st, &p.x_map[0], t * FBK, m0, &full_x[s]);
            tma_load_2d(st + F_TILE, &p.x_map[1], t * FBK, m0, &full_x[s]);
            x_issued = t + 1;
            if ((t & 3) == 0 && t / 4 + 2 < n_sb) ok = issue_raw(t / 4 + 2);
        }
        // keep the CTA alive until every copy it issued has landed
        for (int t = x_issued > X_STAGES ? x_issued - X_STAGES : 0; t < x_issued; ++t)
            mbar_wait_bounded(&full_x[t % X_STAGES], (t / X_STAGES) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
        for (int sb = raw_issued > RAW_SLOTS ? raw_issued - RAW_SLOTS : 0; sb < raw_issued; ++sb)
            mbar_wait_bounded(&full_raw[sb % RAW_SLOTS], (sb / RAW_SLOTS) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: Xh Wh + Xh Wl + Xl Wh per K slice of 64
        for (int t = 0; t < n_k; ++t) {
            const int sx = t % X_STAGES, sw = t % W_STAGES;
            if (!mbar_wait_bounded(&full_x[sx], (t / X_STAGES) & 1, p.wait_ns, p.err, kErrTimeoutMma)) break;
            if (!mbar_wait_bounded(&full_w[sw], (t / W_STAGES) & 1, p.wait_ns, p.err, kErrTimeoutMma)) break;
            tc_fence_after();
            const uint32_t xa = smem_addr(xst + sx * F_PAIR), wa = smem_addr(wst + sw * F_PAIR);
            const uint64_t xh = sw128_desc(xa), xl = sw128_desc(xa + F_TILE);
            const uint64_t wh = sw128_desc(wa), wl = sw128_desc(wa + F_TILE);
#pragma unroll
            for (int k = 0; k < FBK / 16; ++k) {
                const uint64_t o = uint64_t(2 * k);
                tc_mma(tmem, xh + o, wh + o, kIdescF, (t | k) != 0 ? 1u : 0u);
                tc_mma(tmem, xh + o, wl + o, kIdescF, 1u);
                tc_mma(tmem, xl + o, wh + o, kIdescF, 1u);
            }
            tc_commit(&empty_x[sx]);  // both arrive once these MMAs have read their operands
            tc_commit(&empty_w[sw]);
        }
        tc_commit(acc_full);  // also after a failed wait: arrives once the issued MMAs are done
    } else if (warp >= 2) {
        // ---- converters: thread ct takes row ct / 4, sub-block half (ct / 2) % 2,
        //      column groups 2 (ct % 2) and 2 (ct % 2) + 1 of that half
        const int ct = threadIdx.x - 64;
        const int row = ct >> 2, half = (ct >> 1) & 1, g0 = 2 * (ct & 1);
        bool ok = true;
        for (int t = 0; t < n_k && ok; ++t) {
            const int sb = t >> 2, c = t & 3, r = sb % RAW_SLOTS, s = t % W_STAGES;
            if ((c == 0 && !warp_wait(&full_raw[r], (sb / RAW_SLOTS) & 1, p.wait_ns, p.err, kErrTimeoutFull)) ||
                (t >= W_STAGES &&
                 !warp_wait(&empty_w[s], ((t / W_STAGES) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))) {
                ok = false;
                break;
            }
            uint8_t* whs = wst + s * F_PAIR + row * 128;
            uint4 hi[2], lo[2];
            q4k_convert_quarter(raw + r * F_RAW_BYTES + row * 144, c, half, g0, hi, lo);
#pragma unroll
            for (int g = 0; g < 2; ++g) {  // 128-byte swizzle: column group j of row r at (j ^ (r % 8)) * 16
                const uint32_t off = uint32_t(((4 * half + g0 + g) ^ (row & 7)) * 16);
                *reinterpret_cast<uint4*>(whs + off) = hi[g];
                *reinterpret_cast<uint4*>(whs + F_TILE + off) = lo[g];
            }
            fence_proxy_async_smem();  // generic-proxy stores, read by the tensor cores
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&full_w[s]);
                if (c == 3) mbar_arrive(&empty_raw[r]);
            }
        }
        // ---- epilogue: warps 2-5; warp w reads tensor-memory lanes 32 (w % 4) .. + 31
        if (warp < 6 && warp_wait(acc_full, 0, p.wait_ns, p.err, kErrTimeoutMma) && ok) {
            tc_fence_after();
            const int q = warp & 3;
            const int yr = m0 + 32 * q + lane;
            const bool row_ok = yr < p.M;
            const bool vec = (n0 + FBN <= p.N) && (p.N % 4 == 0);
            float* yrow = p.Y + size_t(row_ok ? yr : 0) * p.N + n0;
#pragma unroll 1
            for (int cc = 0; cc < FBN / 32; ++cc) {
                uint32_t v[32];
                tc_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(32 * cc), v);
                if (!row_ok) continue;
                if (vec) {
                    float4* dst = reinterpret_cast<float4*>(yrow + 32 * cc);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (n0 + 32 * cc + i < p.N) yrow[32 * cc + i] = __uint_as_float(v[i]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(FBN) : "memory");
}

// ---------------------------------------------------------------------------
// host
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// [rows, K] bf16 row-major, boxes of 64 K x box_rows rows, 128-byte swizzle.
bool encode_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t K, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(K) * 2};
    cuuint32_t box[2] = {cuuint32_t(BK), cuuint32_t(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q4_K rows as a byte matrix [rows, row_bytes], boxes of one super-block
// (144 bytes) x 128 rows, no swizzle.
bool encode_raw_map(CUtensorMap* m, const void* ptr, int64_t rows, int64_t row_bytes) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(row_bytes), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
    cuuint32_t box[2] = {144u, cuuint32_t(FBN)};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

cudaError_t configure_smem(const void* kernel, size_t bytes, bool* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

}  // namespace

size_t prefill_tc_workspace_bytes(int fmt, int64_t N, int64_t K, int64_t M) {
    const size_t x = 2 * round256(size_t(M) * K * 2);
    return fmt == QX_Q4_K ? x : x + 2 * round256(size_t(N) * K * 2);  // Q4_K: weights split in-kernel
}

cudaError_t launch_prefill_tc(int fmt, const uint8_t* W, int64_t N, int64_t K, int64_t row_bytes, const int8_t* xq,
                              const float* xd, int64_t M, float* Y, void* ws, unsigned* err, cudaStream_t s) {
    uint8_t* base = static_cast<uint8_t*>(ws);
    if (fmt == QX_Q4_K) {
        // activation split, then the fused kernel (weights split in shared memory)
        uint16_t* Xh = reinterpret_cast<uint16_t*>(base);
        uint16_t* Xl = reinterpret_cast<uint16_t*>(base + round256(size_t(M) * K * 2));
        const int64_t xthreads = M * (K / 32);
        dequant_x_kernel<<<unsigned((xthreads + 255) / 256), 256, 0, s>>>(xq, xd, M, K, Xh, Xl);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        FusedParams p;
        memset(&p, 0, sizeof(p));
        if (!encode_map(&p.x_map[0], Xh, M, K, FBM) || !encode_map(&p.x_map[1], Xl, M, K, FBM) ||
            !encode_raw_map(&p.w_map, W, N, row_bytes))
            return cudaErrorInvalidValue;
        p.M = int(M);
        p.N = int(N);
        p.K = int(K);
        p.Y = Y;
        p.err = err;
        p.wait_ns = 2000000000ull;
        static bool configured[64] = {false};
        if ((e = configure_smem(reinterpret_cast<const void*>(tc_q4k_fused_kernel), kFusedSmem, configured)) !=
            cudaSuccess)
            return e;
        const dim3 grid(unsigned((M + FBM - 1) / FBM), unsigned((N + FBN - 1) / FBN));
        tc_q4k_fused_kernel<<<grid, kFusedThreads, kFusedSmem, s>>>(p);
        return cudaGetLastError();
    }
    uint16_t* Wh = reinterpret_cast<uint16_t*>(base);
    uint16_t* Wl = reinterpret_cast<uint16_t*>(base + round256(size_t(N) * K * 2));
    uint16_t* Xh = reinterpret_cast<uint16_t*>(base + 2 * round256(size_t(N) * K * 2));
    uint16_t* Xl = reinterpret_cast<uint16_t*>(base + 2 * round256(size_t(N) * K * 2) + round256(size_t(M) * K * 2));

    const int64_t wthreads = N * (K / 32), xthreads = M * (K / 32);
    switch (fmt) {
        case QX_Q4_K:
            dequant_w_kernel<QX_Q4_K><<<unsigned((wthreads + 255) / 256), 256, 0, s>>>(W, N, K, row_bytes, Wh, Wl);
            break;
        case QX_Q6_K:
            dequant_w_kernel<QX_Q6_K><<<unsigned((wthreads + 255) / 256), 256, 0, s>>>(W, N, K, row_bytes, Wh, Wl);
            break;
        default:
            dequant_w_kernel<QX_Q8_0><<<unsigned((wthreads + 255) / 256), 256, 0, s>>>(W, N, K, row_bytes, Wh, Wl);
            break;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dequant_x_kernel<<<unsigned((xthreads + 255) / 256), 256, 0, s>>>(xq, xd, M, K, Xh, Xl);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    TcParams p;
    memset(&p, 0, sizeof(p));
    if (!encode_map(&p.a_map[0], Xh, M, K, BM) || !encode_map(&p.a_map[1], Xl, M, K, BM) ||
        !encode_map(&p.b_map[0], Wh, N, K, BN) || !encode_map(&p.b_map[1], Wl, N, K, BN))
        return cudaErrorInvalidValue;
    p.M = int(M);
    p.N = int(N);
    p.K = int(K);
    p.Y = Y;
    p.err = err;
    p.wait_ns = 2000000000ull;
    static bool configured[64] = {false};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTcSmem));
        if (e != cudaSuccess) return e;
        configured[dev] = true;
    }
    const dim3 grid(unsigned((M + BM - 1) / BM), unsigned((N + BN - 1) / BN));
    tc_gemm_kernel<<<grid, kTcThreads, kTcSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace qx
