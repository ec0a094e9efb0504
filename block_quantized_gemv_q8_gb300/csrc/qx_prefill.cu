// qx_prefill.cu -- the W4A8 contraction at prefill batch sizes on tensor cores.
//
// llamay docs, "Backends and hardware", section "CUDA": a tensor-core prefill
// kernel for the W4A8 contraction.  Y[m, n] = sum over the Q4_K sub-blocks j
// of dx[m, j] * (d[n] * sc_j[n] * P_j[m, n] - dmin[n] * m_j[n] * S[m, j]),
// with P_j the integer dot of the int8 activation codes and the 4-bit quants.
//
// The integer products run on the tensor cores as f16 MMAs whose operands
// are small integers, all exact in f16: activation codes in [-127, 127] and
// q * sc_j in [0, 945] (the 6-bit scale folded into the weight operand).  The
// f32 accumulation of one 32-wide sub-block stays below 2^24 in magnitude, so
// every D_j = sc_j * P_j is exact.  The per-(row, sub-block) activation scale
// then has to be applied outside the MMA, once per sub-block, in registers:
//   acc_sb += dx[m, j] * D_j;   mt += dx[m, j] * S[m, j] * m_j[n]
// and per super-block  acc += d[n] * acc_sb - dmin[n] * mt.
//
// CTA tile 64 x 128 (rows of X x weight rows), 8 warps of 32 x 32, K steps
// of half a super-block (128 columns = 4 sub-blocks).  Each K step the next
// tile's activation codes and Q4_K bytes are loaded to registers while the
// current one is multiplied, then converted to f16 into the other shared-
// memory buffer (XOR-swizzled 16-byte chunks, read with ldmatrix).
#include "qx_device.cuh"
#include "qx_internal.h"

namespace qx {

namespace {

constexpr int BM = 64;          // rows of X per CTA
constexpr int BN = 128;         // weight rows (output features) per CTA
constexpr int BK = 128;         // columns per K step (half a Q4_K super-block)
constexpr int kThreads = 256;   // 8 warps: 2 along M x 4 along N, 32 x 32 each
constexpr int kRowHalves = BK;  // f16 elements per smem row
// shared memory per buffer: A [BM][BK] f16, B [BN][BK] f16, per-row/col scales
constexpr int kAbytes = BM * BK * 2;
constexpr int kBbytes = BN * BK * 2;

struct PrefillParams {
    const uint8_t* W;   // Q4_K [N, K/256 * 144]
    const int8_t* xq;   // [M, K]
    const float* xd;    // [M, K/32]
    const int32_t* xs;  // [M, K/32]
    float* Y;           // [M, N]
    int64_t M, N, K;
    int64_t row_bytes;
};

// byte offset of 16-byte chunk c of row r in a swizzled [rows][BK] f16 tile
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return uint32_t(r) * (kRowHalves * 2) + uint32_t((c ^ (r & 7)) << 4);
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// two int8 codes -> packed f16x2, exactly (signed byte values)
__device__ __forceinline__ uint32_t s8x2_to_f16x2(uint32_t lo, uint32_t hi) {
    const __half2 h = __halves2half2(__short2half_rn(static_cast<short>(static_cast<int8_t>(lo))),
                                     __short2half_rn(static_cast<short>(static_cast<int8_t>(hi))));
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Registers holding one K step of raw inputs for this thread.
struct Raw {
    uint4 a[2];       // activation codes: 2 x 16 bytes
    uint4 q[2];       // Q4_K quants of this thread's (row, 32-byte chunk) pieces
    uint4 hdr;        // Q4_K header (d, dmin, packed scales) of the thread's first weight row
};

// A tile: BM rows x BK int8 = 8 KB; 256 threads x 2 x 16 bytes.
// B tile: BN rows x (64 quant bytes of the half super-block); 256 threads x 2
// x 16 bytes: thread t takes row t / 2, 16-byte chunks 2 * (t % 2) + {0, 1}.
__device__ __forceinline__ void load_raw(const PrefillParams& p, int64_t m0, int64_t n0, int ks, Raw& r) {
    const int t = threadIdx.x;
    const int64_t k0 = int64_t(ks) * BK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = t + i * kThreads;  // 0 .. 511: row idx / 8, chunk idx % 8
        const int64_t m = m0 + idx / 8;
        r.a[i] = m < p.M ? *reinterpret_cast<const uint4*>(p.xq + m * p.K + k0 + (idx % 8) * 16)
                         : make_uint4(0, 0, 0, 0);
    }
    const int64_t n = n0 + t / 2;
    const int sb = ks >> 1, h = ks & 1;
    if (n < p.N) {
        const uint8_t* bp = p.W + n * p.row_bytes + int64_t(sb) * 144;
        const uint4* qs = reinterpret_cast<const uint4*>(bp + 16 + 64 * h);
        r.q[0] = qs[2 * (t % 2)];
        r.q[1] = qs[2 * (t % 2) + 1];
        r.hdr = *reinterpret_cast<const uint4*>(bp);
    } else {
        r.q[0] = r.q[1] = r.hdr = make_uint4(0, 0, 0, 0);
    }
}

// Write one K step to shared memory as f16, plus the per-row activation
// terms (dx, dx*S) and per-weight-row terms (d, dmin*m_j as f32).
__device__ __forceinline__ void store_tile(const PrefillParams& p, int64_t m0, int64_t n0, int ks, const Raw& r,
                                           uint8_t* As, uint8_t* Bs, float* sdx, float* sT, float* sd, float* sdm) {
    const int t = threadIdx.x;
    // activation codes -> f16 (16 codes per 16-byte chunk -> two 16-byte f16 chunks)
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int idx = t + i * kThreads;
        const int row = idx / 8, c8 = idx % 8;  // c8: 16-code chunk = f16 chunks 2*c8, 2*c8 + 1
        const uint32_t w[4] = {r.a[i].x, r.a[i].y, r.a[i].z, r.a[i].w};
        uint32_t h[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            h[2 * k] = s8x2_to_f16x2(w[k] & 0xFF, (w[k] >> 8) & 0xFF);
            h[2 * k + 1] = s8x2_to_f16x2((w[k] >> 16) & 0xFF, w[k] >> 24);
        }
        *reinterpret_cast<uint4*>(As + swz(row, 2 * c8)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(As + swz(row, 2 * c8 + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
    // weights: thread t holds 32 quant bytes = chunk cc = t % 2 of the half
    // super-block's two 32-byte chunks; low nibbles are sub-block 2cc (k 0..31
    // of the chunk), high nibbles sub-block 2cc + 1 (k 32..63).
    {
        const int row = t / 2, cc = t % 2;
        const int h = ks & 1;
        const uint32_t s0 = r.hdr.y, s1 = r.hdr.z, s2 = r.hdr.w;
        const uint32_t sc_w = h ? ((s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u)) : (s0 & 0x3F3F3F3Fu);
        const uint32_t m_w = h ? (((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u)) : (s1 & 0x3F3F3F3Fu);
        const int jlo = 2 * cc, jhi = 2 * cc + 1;  // sub-blocks within the half (0..3)
        const __half2 sclo = __half2half2(__int2half_rn(int((sc_w >> (8 * jlo)) & 0xFF)));
        const __half2 schi = __half2half2(__int2half_rn(int((sc_w >> (8 * jhi)) & 0xFF)));
        const uint32_t q[8] = {r.q[0].x, r.q[0].y, r.q[0].z, r.q[0].w, r.q[1].x, r.q[1].y, r.q[1].z, r.q[1].w};
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            // nibbles -> f16 q exactly (0x6400 | q is 1024 + q), times the scale
            const uint32_t bias = 0x64006400u;
            const uint32_t l02 = (q[k] & 0x000F000Fu) | bias, l13 = ((q[k] >> 8) & 0x000F000Fu) | bias;
            const uint32_t h02 = ((q[k] >> 4) & 0x000F000Fu) | bias, h13 = ((q[k] >> 12) & 0x000F000Fu) | bias;
            const __half2 off = __half2half2(__ushort_as_half(0x6400));
            __half2 a = __hsub2(*reinterpret_cast<const __half2*>(&l02), off);  // bytes 0, 2
            __half2 b = __hsub2(*reinterpret_cast<const __half2*>(&l13), off);  // bytes 1, 3
            __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&h02), off);
            __half2 d = __hsub2(*reinterpret_cast<const __half2*>(&h13), off);
            a = __hmul2(a, sclo);
            b = __hmul2(b, sclo);
            c = __hmul2(c, schi);
            d = __hmul2(d, schi);
            // reorder to element order: (byte0, byte1), (byte2, byte3)
            const __half2 e01 = __halves2half2(__low2half(a), __low2half(b));
            const __half2 e23 = __halves2half2(__high2half(a), __high2half(b));
            const __half2 f01 = __halves2half2(__low2half(c), __low2half(d));
            const __half2 f23 = __halves2half2(__high2half(c), __high2half(d));
            lo[2 * k] = *reinterpret_cast<const uint32_t*>(&e01);
            lo[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&e23);
            hi[2 * k] = *reinterpret_cast<const uint32_t*>(&f01);
            hi[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&f23);
        }
        // k within the half: sub-block j occupies k = 32 j .. 32 j + 31, i.e.
        // f16 chunks 4 j .. 4 j + 3 (8 halves each)
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            *reinterpret_cast<uint4*>(Bs + swz(row, 4 * jlo + c4)) =
                make_uint4(lo[4 * c4], lo[4 * c4 + 1], lo[4 * c4 + 2], lo[4 * c4 + 3]);
            *reinterpret_cast<uint4*>(Bs + swz(row, 4 * jhi + c4)) =
                make_uint4(hi[4 * c4], hi[4 * c4 + 1], hi[4 * c4 + 2], hi[4 * c4 + 3]);
        }
        if (cc == 0) {
            const float d = f16_bits_to_f32(r.hdr.x), dmin = f16_bits_to_f32(r.hdr.x >> 16);
            sd[row] = d;
#pragma unroll
            for (int j = 0; j < 4; ++j) sdm[row * 4 + j] = dmin * float((m_w >> (8 * j)) & 0xFF);
        }
    }
    // activation scales of this K step: BM rows x 4 sub-blocks
    if (t < BM * 4) {
        const int row = t / 4, j = t % 4;
        const int64_t m = m0 + row;
        float dx = 0.0f, T = 0.0f;
        if (m < p.M) {
            const int64_t g = m * (p.K / 32) + int64_t(ks) * 4 + j;
            dx = p.xd[g];
            T = dx * float(p.xs[g]);
        }
        sdx[row * 4 + j] = dx;
        sT[row * 4 + j] = T;
    }
}

__global__ void __launch_bounds__(kThreads, 1) prefill_q4k_kernel(const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    // two buffers: [A f16][B f16][dx BM*4][T BM*4][d BN][dmin*m BN*4]
    constexpr int kScal = (BM * 4 * 2 + BN + BN * 4) * 4;
    constexpr int kBuf = kAbytes + kBbytes + kScal;
    const int64_t n0 = int64_t(blockIdx.x) * BN, m0 = int64_t(blockIdx.y) * BM;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wm = warp / 4, wn = warp % 4;  // warp tile: rows wm*32.., cols wn*32..
    const int g = lane >> 2, tg = lane & 3;

    auto buf = [&](int b) { return smem + b * kBuf; };
    auto As = [&](int b) { return buf(b); };
    auto Bs = [&](int b) { return buf(b) + kAbytes; };
    auto sdx = [&](int b) { return reinterpret_cast<float*>(buf(b) + kAbytes + kBbytes); };
    auto sT = [&](int b) { return sdx(b) + BM * 4; };
    auto sd = [&](int b) { return sT(b) + BM * 4; };
    auto sdm = [&](int b) { return sd(b) + BN; };

    float acc[2][4][4], acc_sb[2][4][4], mt[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int jn = 0; jn < 4; ++jn)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][jn][e] = acc_sb[i][jn][e] = mt[i][jn][e] = 0.0f;

    const int nks = static_cast<int>(p.K / BK);
    Raw raw;
    load_raw(p, m0, n0, 0, raw);
    store_tile(p, m0, n0, 0, raw, As(0), Bs(0), sdx(0), sT(0), sd(0), sdm(0));
    __syncthreads();

    for (int ks = 0; ks < nks; ++ks) {
        const int cur = ks & 1;
        if (ks + 1 < nks) load_raw(p, m0, n0, ks + 1, raw);  // overlaps the MMAs below
        const uint32_t a_base = smem_addr(As(cur)), b_base = smem_addr(Bs(cur));
        const float* cdx = sdx(cur);
        const float* cT = sT(cur);
        const float* cdm = sdm(cur);
#pragma unroll
        for (int j = 0; j < 4; ++j) {  // sub-blocks of this K step
            float D[2][4][4];
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {  // two k16 steps per sub-block
                const int kc = 4 * j + 2 * kk;  // 16-byte chunk index of this k16 step
                uint32_t a[2][4], b[4][2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int row = wm * 32 + i * 16 + (lane & 15);
                    ldmatrix_x4(a_base + swz(row, kc + (lane >> 4)), a[i]);
                }
#pragma unroll
                for (int jp = 0; jp < 2; ++jp) {  // two n8 tiles per ldmatrix.x4
                    const int row = wn * 32 + jp * 16 + (lane & 7) + ((lane >> 4) << 3);
                    uint32_t r4[4];
                    ldmatrix_x4(b_base + swz(row, kc + ((lane >> 3) & 1)), r4);
                    b[2 * jp][0] = r4[0];
                    b[2 * jp][1] = r4[1];
                    b[2 * jp + 1][0] = r4[2];
                    b[2 * jp + 1][1] = r4[3];
                }
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int jn = 0; jn < 4; ++jn) {
                        if (kk == 0) {
                            const float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                            mma_16816(D[i][jn], a[i], b[jn][0], b[jn][1], z);
                        } else {
                            mma_16816(D[i][jn], a[i], b[jn][0], b[jn][1], D[i][jn]);
                        }
                    }
            }
            // scale the exact sub-block sums: rows r0 = g, r1 = g + 8 of each m16 tile
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int r0 = wm * 32 + i * 16 + g;
                const float dx0 = cdx[r0 * 4 + j], dx1 = cdx[(r0 + 8) * 4 + j];
                const float T0 = cT[r0 * 4 + j], T1 = cT[(r0 + 8) * 4 + j];
#pragma unroll
                for (int jn = 0; jn < 4; ++jn) {
                    const int c0 = wn * 32 + jn * 8 + 2 * tg;
                    const float mj0 = cdm[c0 * 4 + j], mj1 = cdm[(c0 + 1) * 4 + j];
                    acc_sb[i][jn][0] = fmaf(dx0, D[i][jn][0], acc_sb[i][jn][0]);
                    acc_sb[i][jn][1] = fmaf(dx0, D[i][jn][1], acc_sb[i][jn][1]);
                    acc_sb[i][jn][2] = fmaf(dx1, D[i][jn][2], acc_sb[i][jn][2]);
                    acc_sb[i][jn][3] = fmaf(dx1, D[i][jn][3], acc_sb[i][jn][3]);
                    mt[i][jn][0] = fmaf(T0, mj0, mt[i][jn][0]);
                    mt[i][jn][1] = fmaf(T0, mj1, mt[i][jn][1]);
                    mt[i][jn][2] = fmaf(T1, mj0, mt[i][jn][2]);
                    mt[i][jn][3] = fmaf(T1, mj1, mt[i][jn][3]);
                }
            }
        }
        // half super-block done: fold in d and dmin of the weight rows
        {
            const float* cd = sd(cur);
#pragma unroll
            for (int jn = 0; jn < 4; ++jn) {
                const int c0 = wn * 32 + jn * 8 + 2 * tg;
                const float d0 = cd[c0], d1 = cd[c0 + 1];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    acc[i][jn][0] += d0 * acc_sb[i][jn][0] - mt[i][jn][0];
                    acc[i][jn][1] += d1 * acc_sb[i][jn][1] - mt[i][jn][1];
                    acc[i][jn][2] += d0 * acc_sb[i][jn][2] - mt[i][jn][2];
                    acc[i][jn][3] += d1 * acc_sb[i][jn][3] - mt[i][jn][3];
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc_sb[i][jn][e] = mt[i][jn][e] = 0.0f;
                }
            }
        }
        if (ks + 1 < nks) store_tile(p, m0, n0, ks + 1, raw, As(cur ^ 1), Bs(cur ^ 1), sdx(cur ^ 1), sT(cur ^ 1),
                                     sd(cur ^ 1), sdm(cur ^ 1));
        __syncthreads();
    }
    // write Y
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int64_t m = m0 + wm * 32 + i * 16 + g + 8 * half;
            if (m >= p.M) continue;
#pragma unroll
            for (int jn = 0; jn < 4; ++jn) {
                const int64_t n = n0 + wn * 32 + jn * 8 + 2 * tg;
                if (n < p.N) p.Y[m * p.N + n] = acc[i][jn][2 * half];
                if (n + 1 < p.N) p.Y[m * p.N + n + 1] = acc[i][jn][2 * half + 1];
            }
        }
    }
}

constexpr int kPrefillSmem = 2 * (kAbytes + kBbytes + (BM * 4 * 2 + BN + BN * 4) * 4);

}  // namespace

cudaError_t launch_prefill_q4k(const uint8_t* W, int64_t N, int64_t K, const int8_t* xq, const float* xd,
                               const int32_t* xs, int64_t M, float* Y, cudaStream_t s) {
    static bool configured[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        err = cudaFuncSetAttribute(prefill_q4k_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrefillSmem);
        if (err != cudaSuccess) return err;
        configured[dev] = true;
    }
    PrefillParams p;
    p.W = W;
    p.xq = xq;
    p.xd = xd;
    p.xs = xs;
    p.Y = Y;
    p.M = M;
    p.N = N;
    p.K = K;
    p.row_bytes = K / 256 * 144;
    const dim3 grid(static_cast<unsigned>((N + BN - 1) / BN), static_cast<unsigned>((M + BM - 1) / BM));
    prefill_q4k_kernel<<<grid, kThreads, kPrefillSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace qx
