// qx_f32mma.cu -- f32-mode GEMV of Q6_K rows (GGUF blocks or the repacked
// QX_Q6_K_SOA layout) and Q4_K rows with the products on the tensor pipe,
// sm_103a.  (Q6_K below; Q4_K differs in its unit, see q4k_f32_mma.)
//
// f32 mode is the dequantise-and-FMA GEMV (llambda.lisp README, "Features &
// Architecture"): y_r = sum_k w_rk x_k with the f32 activation and the Q6_K
// weights w = d sc (q - 32) (one int8 scale sc per 16 weights, one f16 d per
// 256).  The lanes of gemv_kernel spend about 4.5 instructions per weight on
// it, mostly converting quants to f32; here the multiplications run as
// mma.sync m16n8k16 with bf16 operands and f32 accumulation:
//
//   * A = 16 weight rows x 16 columns: the quants q - 32 (-32..31), which
//     are exact bf16 values -- a byte q becomes the bf16 128 + q by one byte
//     permute (0x43 above the byte), and one bf16x2 subtraction of 160 leaves
//     q - 32, two values per instruction;
//   * B = the activation of the warp's 256-column super-block, scaled by a
//     power of two 2^e that brings its largest magnitude into [1, 2), and
//     split into two bf16 terms: x 2^e = hi + lo + r, |r| <= 2^-18 |x 2^e|;
//   * the eight B columns are four pairs (hi, lo), one pair per 16-column
//     group and zero outside it, so one accumulator holds, per weight row,
//     the hi and lo sums of four groups; per group the f32 epilogue adds
//     sc (D_hi + D_lo), per super-block d 2^-e, and the reducer warp adds the
//     super-blocks of each row in a fixed order.
//
// Error: each product (q - 32) hi, (q - 32) lo is exact (6 x 8 significant
// bits); the split drops at most 2^-18 of each |x| (for every element within
// 2^-100 of its super-block's largest, whose terms stay normal); the f32 sums
// (the tensor pipe's, the epilogue's, the reduction's) add a few units of
// 2^-24 of the sum of |terms|.  So |y - y_exact| is below about 2^-17 of
// sum_k |w_rk x_k|, well inside the f32-mode tolerance of 1e-4 of that sum.
// Both layouts hold the same values and run the same arithmetic in the same
// order, so their outputs are bit-identical.
//
// Structure: the row-group kernel of the small-batch tensor path -- one CTA
// per SM, a producer warp copying each row of a stage of 16 P gq rows to a
// padded stride (qx_stage.cuh), 16 consumer warps (warp w owns super-block
// w % nsb of row groups w / nsb, w / nsb + P, ... of every stage, P = 16 /
// nsb, so its B fragments stay in registers), and a reducer warp.  Rows of
// 2048 or 4096 columns (GGUF Q6_K rows are then a 16-byte multiple).
#include <cuda_runtime.h>

#include "qx_device.cuh"
#include "qx_internal.h"
#include "qx_stage.cuh"

namespace qx {

namespace {

constexpr int kF32MmaWarps = 16;

// bf16x2 (hi half = b, lo half = a), rounded to nearest even.
__device__ __forceinline__ uint32_t bf16x2_rn(float a, float b) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}

__device__ __forceinline__ float bf16_rn_f32(float v) {
    return __uint_as_float(bf16x2_rn(v, 0.0f) << 16);
}

// The bf16 pair (q0 - 32, q1 - 32) of bytes k, k + 1 (k = 0 or 2) of a word
// of 6-bit quants: 0x43 above each byte is the bf16 128 + q; minus 160, exact.
template <int K>
__device__ __forceinline__ uint32_t q6_pair_bf16(uint32_t w) {
    const uint32_t biased = __byte_perm(w, 0x43u, K == 0 ? 0x4140u : 0x4342u);
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x43204320u));
    return r;
}

// Byte sel & 3 of w, sign-extended (prmt with the sign-replicate selectors).
__device__ __forceinline__ int sext_byte(uint32_t w, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(w), "r"(sel));
    return static_cast<int>(r);
}

// D += A B, m16n8k16, bf16 operands, f32 accumulators.
__device__ __forceinline__ void mma_bf16_k16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (w0 >> 16) | (w1 << 16) with two multiplies (the FMA pipe; the ALU pipe is
// this kernel's busiest): m = 65536, passed as a run-time value.
__device__ __forceinline__ uint32_t join16(uint32_t w0, uint32_t w1, uint32_t m) {
    return __umulhi(w0, m) + w1 * m;
}

// A Q6_K super-block as stored in a stage: ql[128] at 0, qh[64] at 128,
// scales[16] at 192; GGUF blocks are 210 bytes (d at 208), repacked ones
// 208 (every field 16-byte aligned, d gathered at the end of the row).  A
// GGUF super-block sb starts at byte 210 sb of a 16-byte-aligned row: on a
// 4-byte boundary for even sb (MIS = 0), 2 bytes past one for odd sb
// (MIS = 2), the same for every field a thread reads.
template <int FMT, int MIS = 0>
struct Q6Block {
    static constexpr bool kSoa = FMT == QX_Q6_K_SOA;
    static constexpr int kBytes = kSoa ? 208 : 210;
    __device__ __forceinline__ static uint2 ld8(const uint8_t* p, uint32_t m) {
        if constexpr (kSoa) {
            return *reinterpret_cast<const uint2*>(p);
        } else if constexpr (MIS == 0) {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
            return make_uint2(w[0], w[1]);
        } else {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(p - 2);
            const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
            return make_uint2(join16(w0, w1, m), join16(w1, w2, m));
        }
    }
    __device__ __forceinline__ static uint4 ld16(const uint8_t* p, uint32_t m) {
        if constexpr (kSoa) {
            return *reinterpret_cast<const uint4*>(p);
        } else if constexpr (MIS == 0) {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
            return make_uint4(w[0], w[1], w[2], w[3]);
        } else {
            const uint32_t* w = reinterpret_cast<const uint32_t*>(p - 2);
            const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
            return make_uint4(join16(w0, w1, m), join16(w1, w2, m), join16(w2, w3, m), join16(w3, w4, m));
        }
    }
    // d of super-block sb of the row at `row`
    __device__ __forceinline__ static float d(const uint8_t* row, int sb, int nsb) {
        const uint8_t* p = kSoa ? row + 208 * nsb + 2 * sb : row + 210 * sb + 208;
        return f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(p));
    }
};

// MMA index of (half h, quarter tq, step s) within a super-block; its B
// fragment is bx[2 i], bx[2 i + 1].
__device__ __forceinline__ constexpr int mma_index(int h, int tq, int s) { return 8 * h + 2 * tq + s; }

// The B fragments of the warp's super-block (its 256 values at xs, times
// `up`), in the order of mma_index.  MMA (h, tq, s) covers, for thread
// (gid, t), elements 128 h + 32 tq + 8 t + 4 s + {0, 1} (logical k = 2 t,
// 2 t + 1) and + {2, 3} (k = 2 t + 8, 2 t + 9); they lie in group (tq, u =
// t >> 1) of the 32-column quarter, whose (hi, lo) pair is column pair
// 2 (tq & 1) + u.  Column gid holds them iff gid >> 1 is that pair: hi for
// even gid, lo for odd; every other B entry is zero.
__device__ __forceinline__ void load_b_f32(const float* xs, float up, int gid, int t, bool live,
                                           uint32_t (&bx)[32]) {
    const bool odd = gid & 1;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int tq = 0; tq < 4; ++tq)
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int i = mma_index(h, tq, s);
                const bool mine = live && (gid >> 1) == 2 * (tq & 1) + (t >> 1);
                uint32_t b0 = 0u, b1 = 0u;
                if (mine) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(xs + 128 * h + 32 * tq + 8 * t + 4 * s));
                    float e[4] = {v.x * up, v.y * up, v.z * up, v.w * up};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float hi = bf16_rn_f32(e[j]);
                        // non-finite activations: the hi term alone carries them
                        e[j] = odd ? (isfinite(hi) ? e[j] - hi : 0.0f) : hi;
                    }
                    b0 = bf16x2_rn(e[0], e[1]);
                    b1 = bf16x2_rn(e[2], e[3]);
                }
                bx[2 * i] = b0;
                bx[2 * i + 1] = b1;
            }
}

// One super-block of rows gid (ra) and gid + 8 (rb) of a 16-row group:
// returns, for thread (gid, t), sum over its groups g = 8 h + 4 a + t of
// sc_g (D_hi + D_lo), rows gid and gid + 8.
template <int FMT, int MIS>
__device__ __forceinline__ void q6_f32_mma(const uint8_t* ra, const uint8_t* rb, int t, uint32_t scsel, uint32_t m,
                                           const uint32_t (&bx)[32], float& ya, float& yb) {
    using B = Q6Block<FMT, MIS>;
    const uint4 sca = B::ld16(ra + 192, m), scb = B::ld16(rb + 192, m);
    const uint32_t swa[4] = {sca.x, sca.y, sca.z, sca.w}, swb[4] = {scb.x, scb.y, scb.z, scb.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        // thread t's 8 bytes of each 32-byte chunk: ql of quarters 0 / 2 and 1 / 3, qh
        const uint2 l0[2] = {B::ld8(ra + 64 * h + 8 * t, m), B::ld8(rb + 64 * h + 8 * t, m)};
        const uint2 l1[2] = {B::ld8(ra + 64 * h + 32 + 8 * t, m), B::ld8(rb + 64 * h + 32 + 8 * t, m)};
        const uint2 hh[2] = {B::ld8(ra + 128 + 32 * h + 8 * t, m), B::ld8(rb + 128 + 32 * h + 8 * t, m)};
        // qh fields 0, 2 (bits 0-1, 4-5 of each byte) and 1, 3 (bits 2-3, 6-7), each word
        // masked once: shifted so that the quarter's field lands on bits 4-5, bits 6-7 stay zero
        uint32_t he[2][2], ho[2][2];  // [row][s]
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            he[r][0] = hh[r].x & 0x33333333u;
            he[r][1] = hh[r].y & 0x33333333u;
            ho[r][0] = hh[r].x & 0xCCCCCCCCu;
            ho[r][1] = hh[r].y & 0xCCCCCCCCu;
        }
#pragma unroll
        for (int a = 0; a < 2; ++a) {  // quarters 2 a, 2 a + 1: low (a = 0) or high nibbles of ql
            float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int tp = 0; tp < 2; ++tp) {
                const int tq = 2 * a + tp;
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    uint32_t w[2];  // rows gid, gid + 8: the 6-bit quants of 4 consecutive elements
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const uint2 lq = tp ? l1[r] : l0[r];
                        const uint32_t lw = s ? lq.y : lq.x;
                        const uint32_t lo4 = a ? (lw >> 4) : lw;
                        const uint32_t hm = tp ? ho[r][s] : he[r][s];
                        const uint32_t hi2 = tq == 0 ? (hm << 4) : tq == 1 ? (hm << 2) : tq == 2 ? hm : (hm >> 2);
                        // bits 0-3 from the nibble, 4-7 from the field (bits 6-7 zero): one lop3
                        w[r] = (lo4 & 0x0F0F0F0Fu) | (hi2 & 0xF0F0F0F0u);
                    }
                    const uint32_t A[4] = {q6_pair_bf16<0>(w[0]), q6_pair_bf16<0>(w[1]), q6_pair_bf16<2>(w[0]),
                                           q6_pair_bf16<2>(w[1])};
                    const int i = mma_index(h, tq, s);
                    mma_bf16_k16(d, A, bx[2 * i], bx[2 * i + 1]);
                }
            }
            // column pair t = group 8 h + 4 a + t: its scale is byte t of scale word 2 h + a
            const float sa = static_cast<float>(sext_byte(swa[2 * h + a], scsel));
            const float sb = static_cast<float>(sext_byte(swb[2 * h + a], scsel));
            ya = fmaf(sa, d[0] + d[1], ya);
            yb = fmaf(sb, d[2] + d[3], yb);
        }
    }
}

// ---------------------------------------------------------------------------
// Q4_K (d, dmin f16; twelve bytes of 6-bit scales sc and mins m; 128 bytes of
// nibbles: chunk j = bytes 16 + 32 j .. + 31 holds sub-block 2 j in its low
// nibbles and 2 j + 1 in its high ones).  w = d sc_s q - dmin m_s, so a
// sub-block s adds d sc_s sum q x - dmin m_s sum x: the first on the tensor
// pipe (q exact in bf16: the nibble under the exponent pattern 0x43 is the
// bf16 128 + q, one lop3 for two of them, minus 128 exactly), the second from
// the sub-block's sum of x.  MMA (s, f), f = 0, 1, covers sub-block s alone:
// thread (gid, t) holds elements 32 s + 8 t + 4 f + {0, 2} (logical k = 2 t,
// 2 t + 1) and + {1, 3} (k = 2 t + 8, 2 t + 9), so that a word's bytes 0, 2 and
// 1, 3 are its pairs; column pair s & 3 holds the sub-block's (hi, lo), and
// an accumulator holds the four sub-blocks 4 a .. 4 a + 3 (a = 0, 1).
// ---------------------------------------------------------------------------

__device__ __forceinline__ void load_b_q4k(const float* xs, float up, int gid, int t, bool live,
                                           uint32_t (&bx)[32]) {
    const bool odd = gid & 1;
#pragma unroll
    for (int sbk = 0; sbk < 8; ++sbk)
#pragma unroll
        for (int f = 0; f < 2; ++f) {
            const int i = 2 * sbk + f;
            const bool mine = live && (gid >> 1) == (sbk & 3);
            uint32_t b0 = 0u, b1 = 0u;
            if (mine) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(xs + 32 * sbk + 8 * t + 4 * f));
                float e[4] = {v.x * up, v.y * up, v.z * up, v.w * up};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float hi = bf16_rn_f32(e[j]);
                    e[j] = odd ? (isfinite(hi) ? e[j] - hi : 0.0f) : hi;
                }
                b0 = bf16x2_rn(e[0], e[2]);
                b1 = bf16x2_rn(e[1], e[3]);
            }
            bx[2 * i] = b0;
            bx[2 * i + 1] = b1;
        }
}

// The bf16 pair (q0, q2) of the nibbles at bits 0-3 and 16-19 of w: 0x43 over
// each nibble is the bf16 128 + q; one subtraction of 128 gives q, exactly.
// (w & mask) | 0x43004300 is one lop3 with the mask in a register (`mask` =
// 0x000F000F, passed in: with both constants as immediates the compiler
// emits two instructions).
__device__ __forceinline__ uint32_t q4_pair_bf16(uint32_t w, uint32_t mask) {
    uint32_t biased, r;
    asm("lop3.b32 %0, %1, %2, 0x43004300, 0xEA;" : "=r"(biased) : "r"(w), "r"(mask));
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x43004300u));
    return r;
}

// One super-block of rows gid (ra) and gid + 8 (rb): returns, for thread
// (gid, t), the sum over its sub-blocks s = t, t + 4 of d sc_s (D_hi + D_lo) -
// dmin m_s S_s (S_s: the sub-block's sum of the scaled activation), rows gid
// and gid + 8.  bsel = 0x7650 + t selects byte t of a scale word as 2^23 + byte.
__device__ __forceinline__ void q4k_f32_mma(const uint8_t* ra, const uint8_t* rb, uint32_t bsel, uint32_t nmask,
                                            float s_lo, float s_hi, const uint32_t (&bx)[32], int t, float& ya,
                                            float& yb) {
    const uint8_t* rows[2] = {ra, rb};
    float dd[2], ndd[2], dm[2], ndm[2];
    uint32_t scw[2][2], mw[2][2];
    uint2 qw[2][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const uint4 h = *reinterpret_cast<const uint4*>(rows[r]);
        dd[r] = f16_bits_to_f32(h.x & 0xFFFFu);
        dm[r] = f16_bits_to_f32(h.x >> 16);
        ndd[r] = dd[r] * -8388608.0f;
        ndm[r] = dm[r] * -8388608.0f;
        scw[r][0] = h.y & 0x3F3F3F3Fu;
        mw[r][0] = h.z & 0x3F3F3F3Fu;
        scw[r][1] = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
        mw[r][1] = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
#pragma unroll
        for (int j = 0; j < 4; ++j) qw[r][j] = *reinterpret_cast<const uint2*>(rows[r] + 16 + 32 * j + 8 * t);
    }
#pragma unroll
    for (int a = 0; a < 2; ++a) {
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int sbk = 4 * a + k, j = sbk >> 1;
#pragma unroll
            for (int f = 0; f < 2; ++f) {
                uint32_t w[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint32_t word = f ? qw[r][j].y : qw[r][j].x;
                    w[r] = (sbk & 1) ? (word >> 4) : word;
                }
                const uint32_t A[4] = {q4_pair_bf16(w[0], nmask), q4_pair_bf16(w[1], nmask),
                                       q4_pair_bf16(w[0] >> 8, nmask), q4_pair_bf16(w[1] >> 8, nmask)};
                const int i = 2 * sbk + f;
                mma_bf16_k16(d, A, bx[2 * i], bx[2 * i + 1]);
            }
        }
        // column pair t = sub-block 4 a + t: d sc and dmin m exactly (an f16 times a 6-bit integer)
        const float sx = a ? s_hi : s_lo;
        const float sca = fmaf(dd[0], __int_as_float(__byte_perm(scw[0][a], 0x4B000000u, bsel)), ndd[0]);
        const float ma = fmaf(dm[0], __int_as_float(__byte_perm(mw[0][a], 0x4B000000u, bsel)), ndm[0]);
        const float scb = fmaf(dd[1], __int_as_float(__byte_perm(scw[1][a], 0x4B000000u, bsel)), ndd[1]);
        const float mb = fmaf(dm[1], __int_as_float(__byte_perm(mw[1][a], 0x4B000000u, bsel)), ndm[1]);
        ya = fmaf(-ma, sx, fmaf(sca, d[0] + d[1], ya));
        yb = fmaf(-mb, sx, fmaf(scb, d[2] + d[3], yb));
    }
}

template <int FMT>
__global__ void __launch_bounds__(kF32MmaThreads, 1) gemv_f32_mma_kernel(const __grid_constant__ GemvParams p) {
    constexpr int NW = kF32MmaWarps;
    constexpr bool kQ4 = FMT == QX_Q4_K;
    using B = Q6Block<kQ4 ? QX_Q6_K : FMT>;  // Q6_K layouts only
    constexpr int kBytes = kQ4 ? 144 : B::kBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + S;
    uint64_t* part = empty + S;
    const int nsb = static_cast<int>(p.cols / 256), P = NW / nsb;  // warps per super-block
    const int GS = P * p.gq;                                          // 16-row groups per stage
    float* red = reinterpret_cast<float*>(smem + p.red_off);          // [S][GS][nsb][16]
    const int red_stage = GS * nsb * 16;
    const int rstride = static_cast<int>(p.row_bytes) + 16;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = cta_row_begin(p, blockIdx.x), r1 = cta_row_begin(p, blockIdx.x + 1);
    if (threadIdx.x == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(&full[k], 1);
            mbar_init(&empty[k], NW + 1);
            mbar_init(&part[k], NW);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == NW) {
        produce_padded_rows(p, r0, r1, full, empty, smem, lane);
        return;
    }
    if (warp == NW + 1) {
        // ---------------- reducer: y[row] = the nsb partials in a fixed order --
        pdl_wait_prior_grid();  // y may be read by the previous kernel
        StageWalker wk{r0, r1, 0};
        int e, nrows;
        int64_t lrow;
        const int row = lane & 15, half = lane >> 4;
        int slot = 0, lap = 0;
        for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
            if (!warp_wait_all(&part[slot], lap & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
            const float* rs = red + size_t(slot) * red_stage;
            for (int gi = 0; gi < GS && 16 * gi < nrows; ++gi) {
                float acc = 0.0f;  // super-blocks half, half + 2, ...; then the two halves
                for (int sb = half; sb < nsb; sb += 2) acc += rs[(gi * nsb + sb) * 16 + row];
                acc += __shfl_xor_sync(0xffffffffu, acc, 16);
                if (half == 0 && 16 * gi + row < nrows) p.e[e].y[lrow + 16 * gi + row] = acc;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            if (++slot == S) {
                slot = 0;
                ++lap;
            }
        }
        return;
    }

    // ---------------- consumers ----------------------------------------------
    pdl_wait_prior_grid();  // x may come from the previous kernel
    const int sb = warp % nsb, gsub = warp / nsb;
    const bool active = gsub < P;
    const int gid = lane >> 2, t = lane & 3;
    // 2^e from the largest magnitude of the super-block's activation (every lane reads 8 values)
    const float* xs = p.x + 256 * sb;
    uint32_t amax = 0u;
    {
        const float4 v0 = __ldg(reinterpret_cast<const float4*>(xs + 8 * lane));
        const float4 v1 = __ldg(reinterpret_cast<const float4*>(xs + 8 * lane + 4));
        const float m = fmaxf(fmaxf(fmaxf(fabsf(v0.x), fabsf(v0.y)), fmaxf(fabsf(v0.z), fabsf(v0.w))),
                              fmaxf(fmaxf(fabsf(v1.x), fabsf(v1.y)), fmaxf(fabsf(v1.z), fabsf(v1.w))));
        amax = __float_as_uint(m);
        // a NaN anywhere: the exponent field 255, like inf (fmaxf drops NaN operands)
        if (isnan(v0.x) || isnan(v0.y) || isnan(v0.z) || isnan(v0.w) || isnan(v1.x) || isnan(v1.y) ||
            isnan(v1.z) || isnan(v1.w))
            amax = 0x7F800000u;
    }
    amax = __reduce_max_sync(0xffffffffu, amax);
    int ex = static_cast<int>(amax >> 23);  // biased exponent of the largest magnitude (0: zero or subnormal)
    if (ex == 255) ex = 127;                // inf or NaN: unscaled
    const float up = ldexpf(1.0f, 127 - ex), down = ldexpf(1.0f, ex - 127);
    uint32_t bx[32];
    float s_lo = 0.0f, s_hi = 0.0f;  // Q4_K: sums of the scaled activation over sub-blocks t and t + 4
    if constexpr (kQ4) {
        load_b_q4k(xs, up, gid, t, active, bx);
        // lane L holds x[8 L .. 8 L + 7] of the super-block: sub-block L / 4
        const float4 v0 = __ldg(reinterpret_cast<const float4*>(xs + 8 * lane));
        const float4 v1 = __ldg(reinterpret_cast<const float4*>(xs + 8 * lane + 4));
        float sum = ((v0.x * up + v0.y * up) + (v0.z * up + v0.w * up)) +
                    ((v1.x * up + v1.y * up) + (v1.z * up + v1.w * up));
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        s_lo = __shfl_sync(0xffffffffu, sum, 4 * t);
        s_hi = __shfl_sync(0xffffffffu, sum, 4 * t + 16);
    } else {
        load_b_f32(xs, up, gid, t, active, bx);
    }
    const uint32_t bsel = 0x7650u + static_cast<uint32_t>(t);
    const uint32_t nmask = 0x000F000Fu * static_cast<uint32_t>(p.stages > 0);  // a register, not an immediate
    // byte t of a scale word, sign-extended
    const uint32_t tt = static_cast<uint32_t>(t);
    const uint32_t scsel = tt | ((tt | 8u) << 4) | ((tt | 8u) << 8) | ((tt | 8u) << 12);
    // 65536 for the GGUF layout's 2-byte joins, from a value the compiler cannot fold
    const uint32_t jm = 65536u * static_cast<uint32_t>(p.stages > 0);

    // The consumers need only each stage's row count: for one matrix, the
    // CTA's rows in stages of p.G (32-bit); otherwise the full stage walk.
    StageWalker wk{r0, r1, 0};
    int e, nrows;
    int64_t lrow;
    const bool one = p.n_entries == 1;
    int left = static_cast<int>(r1 - r0);
    int slot = 0, lap = 0;  // ring position of stage k: k % S, k / S
    for (;;) {
        if (one) {
            if (left <= 0) break;
            nrows = left < p.G ? left : p.G;
            left -= nrows;
        } else if (!wk.next(p, e, lrow, nrows)) {
            break;
        }
        if (!warp_wait_all(&full[slot], lap & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
        const uint8_t* stage = smem + size_t(slot) * p.slot_bytes;
        float* rs = red + size_t(slot) * red_stage + sb * 16;
        if (active) {
            for (int gi = gsub; gi < GS && 16 * gi < nrows; gi += P) {  // warp-uniform
                const uint8_t* rowa = stage + (16 * gi + gid) * rstride;
                const uint8_t* rowb = rowa + 8 * rstride;
                float ya = 0.0f, yb = 0.0f;
                if constexpr (kQ4) {
                    q4k_f32_mma(rowa + kBytes * sb, rowb + kBytes * sb, bsel, nmask, s_lo, s_hi, bx, t, ya, yb);
                } else {
                    if (FMT == QX_Q6_K && (sb & 1))  // warp-uniform
                        q6_f32_mma<FMT, 2>(rowa + kBytes * sb, rowb + kBytes * sb, t, scsel, jm, bx, ya, yb);
                    else
                        q6_f32_mma<FMT, 0>(rowa + kBytes * sb, rowb + kBytes * sb, t, scsel, jm, bx, ya, yb);
                }
                ya += __shfl_xor_sync(0xffffffffu, ya, 1);
                yb += __shfl_xor_sync(0xffffffffu, yb, 1);
                ya += __shfl_xor_sync(0xffffffffu, ya, 2);
                yb += __shfl_xor_sync(0xffffffffu, yb, 2);
                if (t == 0) {
                    if constexpr (kQ4) {  // d and dmin are inside
                        rs[gi * nsb * 16 + gid] = ya * down;
                        rs[gi * nsb * 16 + gid + 8] = yb * down;
                    } else {
                        rs[gi * nsb * 16 + gid] = (ya * B::d(rowa, sb, nsb)) * down;
                        rs[gi * nsb * 16 + gid + 8] = (yb * B::d(rowb, sb, nsb)) * down;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&part[slot]);
            mbar_arrive(&empty[slot]);
        }
        if (++slot == S) {
            slot = 0;
            ++lap;
        }
    }
}

// Largest shared memory (static + dynamic) a CTA may use on sm_103a.
constexpr int kMaxDynamicSmem = 227 * 1024;

template <int FMT>
cudaError_t launch_f32_mma_one(const GemvParams& p, size_t smem, cudaStream_t s, bool pdl) {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!done[dev]) {
        cudaFuncAttributes fa;
        if ((err = cudaFuncGetAttributes(&fa, gemv_f32_mma_kernel<FMT>)) != cudaSuccess) return err;
        err = cudaFuncSetAttribute(gemv_f32_mma_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kMaxDynamicSmem - static_cast<int>(fa.sharedSizeBytes));
        if (err != cudaSuccess) return err;
        done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_cta);
    cfg.blockDim = dim3(kF32MmaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_f32_mma_kernel<FMT>, p);
}

}  // namespace

cudaError_t launch_gemv_f32_mma(int fmt, const GemvParams& p, size_t smem, cudaStream_t s, bool pdl) {
    switch (fmt) {
        case QX_Q6_K: return launch_f32_mma_one<QX_Q6_K>(p, smem, s, pdl);
        case QX_Q6_K_SOA: return launch_f32_mma_one<QX_Q6_K_SOA>(p, smem, s, pdl);
        case QX_Q4_K: return launch_f32_mma_one<QX_Q4_K>(p, smem, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qx
