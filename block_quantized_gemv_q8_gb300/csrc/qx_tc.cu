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
// Kernels: a dequantise-and-split pass per operand (memory-bound), then the
// GEMM: one CTA per 128 x 256 output tile (one per SM: 192 KB of stages),
// warp 0 issues the TMA loads of 128B-swizzled K-major tiles, warp 1 owns the
// tensor memory and issues tcgen05.mma (M = 128, N = 256, K = 16) from one
// thread, warps 2-5 drain the accumulator with tcgen05.ld and store Y.  Every
// wait is bounded and reports through the device error word.
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
        int ok = 0;
        if (lane == 0) ok = mbar_wait_bounded(acc_full, 0, p.wait_ns, p.err, kErrTimeoutMma) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (ok) {
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

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

}  // namespace

size_t prefill_tc_workspace_bytes(int64_t N, int64_t K, int64_t M) {
    return 2 * round256(size_t(N) * K * 2) + 2 * round256(size_t(M) * K * 2);
}

cudaError_t launch_prefill_tc(int fmt, const uint8_t* W, int64_t N, int64_t K, int64_t row_bytes, const int8_t* xq,
                              const float* xd, int64_t M, float* Y, void* ws, unsigned* err, cudaStream_t s) {
    uint8_t* base = static_cast<uint8_t*>(ws);
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
