// qx_lanes.cuh -- per-format lane arithmetic of the streaming GEMV and the
// processing of one pipeline stage of rows, shared by the single-launch
// kernel (qx_gemv.cu) and the chained kernel (qx_chain.cu).
//
// A consumer lane owns a fixed slice of C columns for the whole launch (its
// activation slice lives in registers); a team of lanes covers one weight
// row.  Lane<FMT, MODE> holds the per-format unpacking and dot products:
//   * W4A8 (llamay docs, "Backends and hardware", sections "CPU" and
//     "CUDA"): per 32-weight sub-block (16 for Q6_K) the int8 x int4/int6/int8
//     products are summed exactly with dp4a, and only then scaled; the weight
//     rows are never materialised.
//   * f32 mode (llambda.lisp README, "Features & Architecture"): every quant
//     is converted exactly to f32 and fused-multiply-added with the f32
//     activation; the per-sub-block scale d*sc (and the Q4_K min term
//     dmin*m*sum(x)) is applied once per sub-block, which is the same sum
//     reassociated.
#pragma once

#include "qx_device.cuh"
#include "qx_internal.h"

namespace qx {
namespace lanes {

// Exact f32 value of a small non-negative integer n < 2^23, via the exponent
// trick: the float with bits 0x4B000000 | n is 2^23 + n.
__device__ __forceinline__ float small_uint_to_f32(uint32_t n) {
    return __int_as_float(0x4B000000u | n) - 8388608.0f;
}

// Byte k of w as the float 2^23 + byte (bits 0x4B0000bb), one byte-permute:
// the caller subtracts 2^23 (plus any offset of the code) exactly.
__device__ __forceinline__ float byte_biased_f32(uint32_t w, int k) {
    return __int_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + uint32_t(k)));
}

// N consecutive (possibly 2-byte aligned) little-endian words from shared
// memory, read as N + 1 aligned words and funnel-shifted.
template <int N>
__device__ __forceinline__ void load_words(const uint8_t* p, uint32_t (&out)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3u) * 8u;
    uint32_t prev = w[0];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const uint32_t next = w[i + 1];
        out[i] = __funnelshift_r(prev, next, sh);
        prev = next;
    }
}

__device__ __forceinline__ uint32_t byte_of(uint32_t w, int k) { return (w >> (8 * k)) & 0xFFu; }

// Q4_K: the eight 6-bit scales and mins of a super-block, four per word.
//   sc_lo / m_lo: sub-blocks 0..3,  sc_hi / m_hi: sub-blocks 4..7.
struct Q4KScales {
    uint32_t sc_lo, m_lo, sc_hi, m_hi;
};

__device__ __forceinline__ Q4KScales q4k_unpack_scales(uint32_t s0, uint32_t s1, uint32_t s2) {
    Q4KScales r;
    r.sc_lo = s0 & 0x3F3F3F3Fu;
    r.m_lo = s1 & 0x3F3F3F3Fu;
    r.sc_hi = (s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u);
    r.m_hi = ((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u);
    return r;
}

// ----------------------------------------------------------------------------
// Per-(format, mode) lane work.  Each specialisation owns C columns per lane:
//   load(): the activation slice into registers (once per kernel)
//   row():  this lane's contribution to one row (or its integer partials)
// ----------------------------------------------------------------------------
template <int FMT, int MODE>
struct Lane;

// Q4_K, W4A8: 128 columns = half a super-block = sub-blocks 4h..4h+3.
// Integer partials of the lane's four sub-blocks; the high-nibble ones are
// formed as dot(16 * q, x) with the unsigned x signed dp4a and are exactly 16
// times the partial.
__device__ __forceinline__ void q4k_half_dots(const uint8_t* bp, int h, const uint32_t (&xq)[32], int (&P)[4]) {
    const uint4* qsp = reinterpret_cast<const uint4*>(bp + 16 + 64 * h);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const uint4 a = qsp[2 * cc], b = qsp[2 * cc + 1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        int plo = 0, phi16 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            plo = dp4a(w[i] & 0x0F0F0F0Fu, xq[16 * cc + i], plo);
            phi16 = dp4a_us(w[i] & 0xF0F0F0F0u, xq[16 * cc + 8 + i], phi16);
        }
        P[2 * cc] = plo;
        P[2 * cc + 1] = phi16;
    }
}

template <>
struct Lane<QX_Q4_K, QX_MODE_W4A8> {
    static constexpr int C = 128;
    static constexpr int kGroups = 4;  // partials per lane
    static constexpr int kRows = 1;    // rows per call
    uint32_t xq[32];
    float dxs[4];  // dx of sub-block u; the odd (high-nibble) ones divided by 16
    float t[4];    // dx * (sum of q_x) of sub-block u: weight of the min term
    // swz: the slice's 16-byte chunks are stored permuted (act_chunk_swizzle)
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t* s, int l, bool swz) {
        const uint4* src = reinterpret_cast<const uint4*>(q + int64_t(l) * C);
        const int sw = swz ? (l & 7) : 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = src[k ^ sw];
            xq[4 * k + 0] = v.x;
            xq[4 * k + 1] = v.y;
            xq[4 * k + 2] = v.z;
            xq[4 * k + 3] = v.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float dx = d[l * 4 + u];
            dxs[u] = (u & 1) ? dx * 0.0625f : dx;
            t[u] = dx * float(s[l * 4 + u]);
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 1, h = l & 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 144;
            const uint4 hdr = *reinterpret_cast<const uint4*>(bp);
            int P[4];
            q4k_half_dots(bp, h, xq, P);
            const Q4KScales S = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
            const uint32_t scw = h ? S.sc_hi : S.sc_lo;
            const uint32_t mw = h ? S.m_hi : S.m_lo;
            float accd = 0.0f, accm = 0.0f;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                accd = fmaf(float(P[u] * int(byte_of(scw, u))), dxs[u], accd);
                accm = fmaf(float(int(byte_of(mw, u))), t[u], accm);
            }
            out[r] = f16_bits_to_f32(hdr.x) * accd - f16_bits_to_f32(hdr.x >> 16) * accm;
        }
    }
    __device__ __forceinline__ void partials(const uint8_t* rowp, int l, int (&P)[kGroups]) const {
        const int sb = l >> 1, h = l & 1;
        q4k_half_dots(rowp + sb * 144, h, xq, P);
        P[1] >>= 4;  // exact: the high-nibble dots are 16 x the partial
        P[3] >>= 4;
    }
    __device__ __forceinline__ static int64_t part_index(int l, int g) { return int64_t(l) * 4 + g; }
};

// Q4_K, f32: 64 columns = one 32-byte chunk c of quants = sub-blocks 2c, 2c+1.
template <>
struct Lane<QX_Q4_K, QX_MODE_F32> {
    static constexpr int C = 64;
    static constexpr int kGroups = 1;
    static constexpr int kRows = 1;
    uint64_t x2[32];  // the 64 activation values as 32 packed pairs (x[2j], x[2j + 1])
    float xsum[2];
    __device__ __forceinline__ void load(const float* xp, int l) {
        const float4* src = reinterpret_cast<const float4*>(xp + int64_t(l) * C);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float s = 0.0f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 v = src[8 * u + k];
                x2[16 * u + 2 * k + 0] = f32x2_pack(v.x, v.y);
                x2[16 * u + 2 * k + 1] = f32x2_pack(v.z, v.w);
                s += v.x;
                s += v.y;
                s += v.z;
                s += v.w;
            }
            xsum[u] = s;
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 2, c = l & 3;
        // 2^23 + q minus 2^23 = q, exactly, two at a time
        const uint64_t bias = f32x2_pack(-8388608.0f, -8388608.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 144;
            const uint4 hdr = *reinterpret_cast<const uint4*>(bp);
            const uint4* qsp = reinterpret_cast<const uint4*>(bp + 16 + 32 * c);
            const uint4 a = qsp[0], b = qsp[1];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            uint64_t s2[4] = {0, 0, 0, 0};  // low nibbles (two sums), high nibbles (two sums)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // the low and the high nibbles, one per byte; each byte becomes an exact float
                const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
                for (int kp = 0; kp < 2; ++kp) {
                    const uint64_t flo =
                        f32x2_add(f32x2_pack(byte_biased_f32(lo, 2 * kp), byte_biased_f32(lo, 2 * kp + 1)), bias);
                    const uint64_t fhi =
                        f32x2_add(f32x2_pack(byte_biased_f32(hi, 2 * kp), byte_biased_f32(hi, 2 * kp + 1)), bias);
                    s2[i & 1] = f32x2_fma(flo, x2[2 * i + kp], s2[i & 1]);
                    s2[2 + (i & 1)] = f32x2_fma(fhi, x2[16 + 2 * i + kp], s2[2 + (i & 1)]);
                }
            }
            float slo, shi;
            {
                const float2 a0 = f32x2_unpack(s2[0]), a1 = f32x2_unpack(s2[1]);
                const float2 b0 = f32x2_unpack(s2[2]), b1 = f32x2_unpack(s2[3]);
                slo = (a0.x + a0.y) + (a1.x + a1.y);
                shi = (b0.x + b0.y) + (b1.x + b1.y);
            }
            const Q4KScales S = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
            const uint32_t scw = c < 2 ? S.sc_lo : S.sc_hi;
            const uint32_t mw = c < 2 ? S.m_lo : S.m_hi;
            const int k0 = 2 * (c & 1);
            const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
            float acc = d * float(byte_of(scw, k0)) * slo;
            acc = fmaf(-dmin * float(byte_of(mw, k0)), xsum[0], acc);
            acc = fmaf(d * float(byte_of(scw, k0 + 1)), shi, acc);
            acc = fmaf(-dmin * float(byte_of(mw, k0 + 1)), xsum[1], acc);
            out[r] = acc;
        }
    }
};

// Q6_K, W4A8: 128 columns = half h of a super-block = quarters t = 0..3 of
// 32 columns, each made of two 16-weight scale groups.  The quants q are
// dotted unsigned (0..63) and the -32 offset is applied as -32 * sum(q_x)
// per group, which is the same integer.
__device__ __forceinline__ void q6k_half_dots(const uint8_t* bp, int h, const uint32_t (&xq)[32],
                                              const int (&s16)[8], int (&P)[8]) {
    uint32_t qh[8];
    load_words<8>(bp + 128 + 32 * h, qh);
    // quarters t and t + 2 share the same 32 ql bytes (low and high nibbles):
    // keep only those 8 words live at a time
#pragma unroll
    for (int tl = 0; tl < 2; ++tl) {
        uint32_t ql[8];
        load_words<8>(bp + 64 * h + 32 * tl, ql);
#pragma unroll
        for (int th = 0; th < 2; ++th) {
            const int t = tl + 2 * th;
            int pu[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo4 = (th ? (ql[i] >> 4) : ql[i]) & 0x0F0F0F0Fu;
                // bits 2t, 2t+1 of each qh byte moved to bits 4, 5
                const uint32_t hsh = t < 2 ? (qh[i] << (4 - 2 * t)) : (qh[i] >> (2 * t - 4));
                pu[i >> 2] = dp4a_us(lo4 | (hsh & 0x30303030u), xq[8 * t + i], pu[i >> 2]);
            }
            P[2 * t] = pu[0] - 32 * s16[2 * t];
            P[2 * t + 1] = pu[1] - 32 * s16[2 * t + 1];
        }
    }
}

template <>
struct Lane<QX_Q6_K, QX_MODE_W4A8> {
    static constexpr int C = 128;
    static constexpr int kGroups = 8;
    static constexpr int kRows = 1;
    uint32_t xq[32];
    float dx[4];
    int s16[8];  // sum of q_x over each 16-group
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int l, bool swz) {
        const uint4* src = reinterpret_cast<const uint4*>(q + int64_t(l) * C);
        const int sw = swz ? (l & 7) : 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = src[k ^ sw];
            xq[4 * k + 0] = v.x;
            xq[4 * k + 1] = v.y;
            xq[4 * k + 2] = v.z;
            xq[4 * k + 3] = v.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) dx[u] = d[l * 4 + u];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            int s = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) s = dp4a(xq[4 * g + i], 0x01010101u, s);
            s16[g] = s;
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 1, h = l & 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 210;
            int P[8];
            q6k_half_dots(bp, h, xq, s16, P);
            uint32_t scw[2];
            load_words<2>(bp + 192 + 8 * h, scw);
            float acc = 0.0f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int sc0 = int(int8_t(byte_of(scw[t >> 1], 2 * (t & 1))));
                const int sc1 = int(int8_t(byte_of(scw[t >> 1], 2 * (t & 1) + 1)));
                acc = fmaf(dx[t], float(sc0 * P[2 * t] + sc1 * P[2 * t + 1]), acc);
            }
            out[r] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp + 208)) * acc;
        }
    }
    __device__ __forceinline__ void partials(const uint8_t* rowp, int l, int (&P)[kGroups]) const {
        const int sb = l >> 1, h = l & 1;
        q6k_half_dots(rowp + sb * 210, h, xq, s16, P);
    }
    __device__ __forceinline__ static int64_t part_index(int l, int g) { return int64_t(l) * 8 + g; }
};

// Q6_K, f32: 64 columns = quarters t = tp and t = tp + 2 of half h (they
// share the same ql bytes, low and high nibbles).
template <>
struct Lane<QX_Q6_K, QX_MODE_F32> {
    static constexpr int C = 64;
    static constexpr int kGroups = 1;
    static constexpr int kRows = 1;
    uint64_t x2[32];  // the 64 activation values as 32 packed pairs (x[2j], x[2j + 1])
    __device__ __forceinline__ void load(const float* xp, int l) {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
        const int64_t c0 = int64_t(sb) * 256 + 128 * h + 32 * tp;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const float4* src = reinterpret_cast<const float4*>(xp + c0 + 64 * half);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 v = src[k];
                x2[16 * half + 2 * k + 0] = f32x2_pack(v.x, v.y);
                x2[16 * half + 2 * k + 1] = f32x2_pack(v.z, v.w);
            }
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
        // 2^23 + q minus (2^23 + 32) = q - 32, exactly, two at a time
        const uint64_t bias = f32x2_pack(-8388640.0f, -8388640.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 210;
            uint32_t ql[8], qh[8], scw[2];
            load_words<8>(bp + 64 * h + 32 * tp, ql);
            load_words<8>(bp + 128 + 32 * h, qh);
            load_words<2>(bp + 192 + 8 * h, scw);
            uint64_t sg2[4] = {0, 0, 0, 0};  // lo g0, lo g1, hi g0, hi g1; two running sums each
            // qh bits 2 tp, 2 tp + 1 (quarter tp) and 2 tp + 4, 2 tp + 5 (quarter tp + 2) to bits 4, 5
            const uint32_t sh_lo = 4u - 2u * uint32_t(tp), sh_hi = 2u * uint32_t(tp);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                // the 6-bit quants of both quarters, one per byte
                const uint32_t wlo = (ql[i] & 0x0F0F0F0Fu) | ((qh[i] << sh_lo) & 0x30303030u);
                const uint32_t whi = ((ql[i] >> 4) & 0x0F0F0F0Fu) | ((qh[i] >> sh_hi) & 0x30303030u);
#pragma unroll
                for (int kp = 0; kp < 2; ++kp) {
                    const uint64_t flo =
                        f32x2_add(f32x2_pack(byte_biased_f32(wlo, 2 * kp), byte_biased_f32(wlo, 2 * kp + 1)), bias);
                    const uint64_t fhi =
                        f32x2_add(f32x2_pack(byte_biased_f32(whi, 2 * kp), byte_biased_f32(whi, 2 * kp + 1)), bias);
                    sg2[i >> 2] = f32x2_fma(flo, x2[2 * i + kp], sg2[i >> 2]);
                    sg2[2 + (i >> 2)] = f32x2_fma(fhi, x2[16 + 2 * i + kp], sg2[2 + (i >> 2)]);
                }
            }
            float sg[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float2 v = f32x2_unpack(sg2[g]);
                sg[g] = v.x + v.y;
            }
            // scale bytes of this half: index 2t + g for t in {tp, tp + 2}
            const int lo0 = 2 * tp, hi0 = 2 * tp + 4;
            float acc = float(int(int8_t(byte_of(scw[lo0 >> 2], lo0 & 3)))) * sg[0];
            acc = fmaf(float(int(int8_t(byte_of(scw[(lo0 + 1) >> 2], (lo0 + 1) & 3)))), sg[1], acc);
            acc = fmaf(float(int(int8_t(byte_of(scw[hi0 >> 2], hi0 & 3)))), sg[2], acc);
            acc = fmaf(float(int(int8_t(byte_of(scw[(hi0 + 1) >> 2], (hi0 + 1) & 3)))), sg[3], acc);
            out[r] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp + 208)) * acc;
        }
    }
};

// Q6_K repacked at load time (QX_Q6_K_SOA, qx_repack): per super-block 208
// bytes -- ql[128], qh[64], scales[16], every field 16-byte aligned -- and
// the row's d values gathered after its super-blocks, at byte d_off =
// 208 * (super-blocks per row).  The same arithmetic as the Q6_K lanes above;
// the fields are read with aligned vector loads instead of funnel-shifted
// words.
__device__ __forceinline__ void load8_al(const uint8_t* p, uint32_t (&w)[8]) {
    const uint4* p4 = reinterpret_cast<const uint4*>(p);
    const uint4 a = p4[0], b = p4[1];
    w[0] = a.x;
    w[1] = a.y;
    w[2] = a.z;
    w[3] = a.w;
    w[4] = b.x;
    w[5] = b.y;
    w[6] = b.z;
    w[7] = b.w;
}

__device__ __forceinline__ void q6k_half_dots_al(const uint8_t* bp, int h, const uint32_t (&xq)[32],
                                                 const int (&s16)[8], int (&P)[8]) {
    uint32_t qh[8];
    load8_al(bp + 128 + 32 * h, qh);
#pragma unroll
    for (int tl = 0; tl < 2; ++tl) {
        uint32_t ql[8];
        load8_al(bp + 64 * h + 32 * tl, ql);
#pragma unroll
        for (int th = 0; th < 2; ++th) {
            const int t = tl + 2 * th;
            int pu[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t lo4 = (th ? (ql[i] >> 4) : ql[i]) & 0x0F0F0F0Fu;
                const uint32_t hsh = t < 2 ? (qh[i] << (4 - 2 * t)) : (qh[i] >> (2 * t - 4));
                pu[i >> 2] = dp4a_us(lo4 | (hsh & 0x30303030u), xq[8 * t + i], pu[i >> 2]);
            }
            P[2 * t] = pu[0] - 32 * s16[2 * t];
            P[2 * t + 1] = pu[1] - 32 * s16[2 * t + 1];
        }
    }
}

template <>
struct Lane<QX_Q6_K_SOA, QX_MODE_W4A8> {
    static constexpr int C = 128;
    static constexpr int kGroups = 8;
    static constexpr int kRows = 1;
    uint32_t xq[32];
    float dx[4];
    int s16[8];
    int d_off;
    __device__ __forceinline__ void geometry(int64_t cols) { d_off = static_cast<int>(cols / 256) * 208; }
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int l, bool swz) {
        const uint4* src = reinterpret_cast<const uint4*>(q + int64_t(l) * C);
        const int sw = swz ? (l & 7) : 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = src[k ^ sw];
            xq[4 * k + 0] = v.x;
            xq[4 * k + 1] = v.y;
            xq[4 * k + 2] = v.z;
            xq[4 * k + 3] = v.w;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) dx[u] = d[l * 4 + u];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            int s = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) s = dp4a(xq[4 * g + i], 0x01010101u, s);
            s16[g] = s;
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 1, h = l & 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 208;
            int P[8];
            q6k_half_dots_al(bp, h, xq, s16, P);
            const uint2 sc2 = *reinterpret_cast<const uint2*>(bp + 192 + 8 * h);
            const uint32_t scw[2] = {sc2.x, sc2.y};
            float acc = 0.0f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int sc0 = int(int8_t(byte_of(scw[t >> 1], 2 * (t & 1))));
                const int sc1 = int(int8_t(byte_of(scw[t >> 1], 2 * (t & 1) + 1)));
                acc = fmaf(dx[t], float(sc0 * P[2 * t] + sc1 * P[2 * t + 1]), acc);
            }
            out[r] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rp[r] + d_off + 2 * sb)) * acc;
        }
    }
    __device__ __forceinline__ void partials(const uint8_t* rowp, int l, int (&P)[kGroups]) const {
        const int sb = l >> 1, h = l & 1;
        q6k_half_dots_al(rowp + sb * 208, h, xq, s16, P);
    }
    __device__ __forceinline__ static int64_t part_index(int l, int g) { return int64_t(l) * 8 + g; }
};

template <>
struct Lane<QX_Q6_K_SOA, QX_MODE_F32> {
    static constexpr int C = 64;
    static constexpr int kGroups = 1;
    static constexpr int kRows = 1;
    uint64_t x2[32];  // the 64 activation values as 32 packed pairs (x[2j], x[2j + 1])
    int d_off;
    __device__ __forceinline__ void geometry(int64_t cols) { d_off = static_cast<int>(cols / 256) * 208; }
    __device__ __forceinline__ void load(const float* xp, int l) {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
        const int64_t c0 = int64_t(sb) * 256 + 128 * h + 32 * tp;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const float4* src = reinterpret_cast<const float4*>(xp + c0 + 64 * half);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 v = src[k];
                x2[16 * half + 2 * k + 0] = f32x2_pack(v.x, v.y);
                x2[16 * half + 2 * k + 1] = f32x2_pack(v.z, v.w);
            }
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
        // 2^23 + q minus (2^23 + 32) = q - 32, exactly, two at a time
        const uint64_t bias = f32x2_pack(-8388640.0f, -8388640.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 208;
            uint32_t ql[8], qh[8];
            load8_al(bp + 64 * h + 32 * tp, ql);
            load8_al(bp + 128 + 32 * h, qh);
            const uint2 sc2 = *reinterpret_cast<const uint2*>(bp + 192 + 8 * h);
            const uint32_t scw[2] = {sc2.x, sc2.y};
            uint64_t sg2[4] = {0, 0, 0, 0};  // lo g0, lo g1, hi g0, hi g1; two running sums each
            const uint32_t sh_lo = 4u - 2u * uint32_t(tp), sh_hi = 2u * uint32_t(tp);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t wlo = (ql[i] & 0x0F0F0F0Fu) | ((qh[i] << sh_lo) & 0x30303030u);
                const uint32_t whi = ((ql[i] >> 4) & 0x0F0F0F0Fu) | ((qh[i] >> sh_hi) & 0x30303030u);
#pragma unroll
                for (int kp = 0; kp < 2; ++kp) {
                    const uint64_t flo =
                        f32x2_add(f32x2_pack(byte_biased_f32(wlo, 2 * kp), byte_biased_f32(wlo, 2 * kp + 1)), bias);
                    const uint64_t fhi =
                        f32x2_add(f32x2_pack(byte_biased_f32(whi, 2 * kp), byte_biased_f32(whi, 2 * kp + 1)), bias);
                    sg2[i >> 2] = f32x2_fma(flo, x2[2 * i + kp], sg2[i >> 2]);
                    sg2[2 + (i >> 2)] = f32x2_fma(fhi, x2[16 + 2 * i + kp], sg2[2 + (i >> 2)]);
                }
            }
            float sg[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float2 v = f32x2_unpack(sg2[g]);
                sg[g] = v.x + v.y;
            }
            const int lo0 = 2 * tp, hi0 = 2 * tp + 4;
            float acc = float(int(int8_t(byte_of(scw[lo0 >> 2], lo0 & 3)))) * sg[0];
            acc = fmaf(float(int(int8_t(byte_of(scw[(lo0 + 1) >> 2], (lo0 + 1) & 3)))), sg[1], acc);
            acc = fmaf(float(int(int8_t(byte_of(scw[hi0 >> 2], hi0 & 3)))), sg[2], acc);
            acc = fmaf(float(int(int8_t(byte_of(scw[(hi0 + 1) >> 2], (hi0 + 1) & 3)))), sg[3], acc);
            out[r] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(rp[r] + d_off + 2 * sb)) * acc;
        }
    }
};

// Q8_0, W4A8: 32 columns = one block.
template <>
struct Lane<QX_Q8_0, QX_MODE_W4A8> {
    static constexpr int C = 32;
    static constexpr int kGroups = 1;
    static constexpr int kRows = 2;
    uint32_t xq[8];
    float dx;
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int l, bool) {
        const uint4* src = reinterpret_cast<const uint4*>(q + int64_t(l) * C);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint4 v = src[k];
            xq[4 * k + 0] = v.x;
            xq[4 * k + 1] = v.y;
            xq[4 * k + 2] = v.z;
            xq[4 * k + 3] = v.w;
        }
        dx = d[l];
    }
    __device__ __forceinline__ int dot(const uint8_t* bp) const {
        uint32_t qs[8];
        load_words<8>(bp + 2, qs);
        int acc = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = dp4a(qs[i], xq[i], acc);
        return acc;
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + l * 34;
            out[r] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp)) * dx * float(dot(bp));
        }
    }
    __device__ __forceinline__ void partials(const uint8_t* rowp, int l, int (&P)[kGroups]) const {
        P[0] = dot(rowp + l * 34);
    }
    __device__ __forceinline__ static int64_t part_index(int l, int) { return l; }
};

// Q8_0, f32: 32 columns = one block.
template <>
struct Lane<QX_Q8_0, QX_MODE_F32> {
    static constexpr int C = 32;
    static constexpr int kGroups = 1;
    static constexpr int kRows = 2;
    uint64_t x2[16];  // the 32 activation values as 16 packed pairs
    __device__ __forceinline__ void load(const float* xp, int l) {
        const float4* src = reinterpret_cast<const float4*>(xp + int64_t(l) * C);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = src[k];
            x2[2 * k + 0] = f32x2_pack(v.x, v.y);
            x2[2 * k + 1] = f32x2_pack(v.z, v.w);
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        // int8 -> f32 exactly: every byte biased by 128 into [0, 255], then 2^23 + 128 taken off
        const uint64_t bias = f32x2_pack(-8388736.0f, -8388736.0f);
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + l * 34;
            uint32_t qs[8];
            load_words<8>(bp + 2, qs);
            uint64_t s2[2] = {0, 0};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t u = qs[i] ^ 0x80808080u;
#pragma unroll
                for (int kp = 0; kp < 2; ++kp) {
                    const uint64_t f =
                        f32x2_add(f32x2_pack(byte_biased_f32(u, 2 * kp), byte_biased_f32(u, 2 * kp + 1)), bias);
                    s2[i & 1] = f32x2_fma(f, x2[2 * i + kp], s2[i & 1]);
                }
            }
            const float2 a0 = f32x2_unpack(s2[0]), a1 = f32x2_unpack(s2[1]);
            out[r] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp)) * ((a0.x + a0.y) + (a1.x + a1.y));
        }
    }
};

// ----------------------------------------------------------------------------
// Teams and one stage of rows
// ----------------------------------------------------------------------------

// Where a consumer lane sits among the row teams of a launch.
struct Team {
    int team;       // team index within the CTA
    int slice;      // this lane's column slice within the team
    bool in_team;   // the warp belongs to a team (a few warps may be spare)
    bool active;    // the slice holds columns
    int team_lanes, team_warps, nteams, L;
};

__device__ __forceinline__ Team make_team(int warp, int lane, int team_lanes, int team_warps, int nteams, int L) {
    Team t;
    if (team_warps == 1) {
        t.team = warp * (32 / team_lanes) + lane / team_lanes;
        t.slice = lane % team_lanes;
    } else {
        // teams of exactly L lanes packed across warp boundaries: the per-lane
        // partials meet only in shared memory, so a team need not be whole warps
        const int flat = warp * 32 + lane;
        t.team = flat / team_lanes;
        t.slice = flat % team_lanes;
    }
    t.in_team = t.team < nteams;
    t.active = t.in_team && t.slice < L;
    t.team_lanes = team_lanes;
    t.team_warps = team_warps;
    t.nteams = nteams;
    t.L = L;
    return t;
}

// All rows of one stage (rows [0, nrows) of `sbuf`, rb bytes each): team t
// takes rows t, t + nteams, ... in calls of R rows.  Every lane stores its
// partial sum of row i to red[i * RS + slice] (plain shared-memory stores, no
// waiting); the reducer warp adds the L partials of each row later
// (reduce_stage).  With PART, integer partials go to Pb + i * ng instead.
template <int FMT, int MODE, bool PART, class LaneT>
__device__ __forceinline__ void consume_stage(const LaneT& X, const Team& tm, const uint8_t* sbuf, int nrows,
                                              uint32_t rb, float* red, int RS, int32_t* Pb, int64_t ng) {
    if (!tm.active) return;
    constexpr int R = PART ? 1 : LaneT::kRows;
    for (int ib = tm.team; ib < nrows; ib += tm.nteams * R) {
        int ir[R];
        bool vr[R];
        const uint8_t* rp[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            ir[r] = ib + r * tm.nteams;
            vr[r] = ir[r] < nrows;
            rp[r] = sbuf + (vr[r] ? uint32_t(ir[r]) : 0u) * rb;
        }
        if constexpr (PART) {
            int P[LaneT::kGroups];
            X.partials(rp[0], tm.slice, P);
            int32_t* dst = Pb + int64_t(ir[0]) * ng;
#pragma unroll
            for (int g = 0; g < LaneT::kGroups; ++g) dst[LaneT::part_index(tm.slice, g)] = P[g];
        } else {
            float v[R];
            X.template rows<R>(rp, tm.slice, v);
#pragma unroll
            for (int r = 0; r < R; ++r)
                if (vr[r]) red[ir[r] * RS + tm.slice] = v[r];
        }
    }
}

// The reducer warp's share of one stage: y[i] = the L partials of row i
// (red[i * RS + 0 .. L)) added in a fixed order -- four running sums over
// slices s = 4k + c, then (c0 + c1) + (c2 + c3) -- one row per lane.
__device__ __forceinline__ void reduce_stage(const float* red, int RS, int L, int nrows, float* y, int lane) {
    for (int row = lane; row < nrows; row += 32) {
        const float* pr = red + row * RS;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        int s = 0;
        for (; s + 16 <= L; s += 16) {
            // four loads in flight, then the adds in slice order
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4*>(pr + s + 4 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a0 += v[u].x;
                a1 += v[u].y;
                a2 += v[u].z;
                a3 += v[u].w;
            }
        }
        for (; s + 4 <= L; s += 4) {
            const float4 v = *reinterpret_cast<const float4*>(pr + s);
            a0 += v.x;
            a1 += v.y;
            a2 += v.z;
            a3 += v.w;
        }
        if (s < L) a0 += pr[s];
        if (s + 1 < L) a1 += pr[s + 1];
        if (s + 2 < L) a2 += pr[s + 2];
        y[row] = (a0 + a1) + (a2 + a3);
    }
}

// ----------------------------------------------------------------------------
// Small-batch lanes (gemv_batch_kernel): kBatchRows rows of a quantised
// activation X share every weight row's bytes, so the weights stream once
// for all of them.  A lane owns batch_cols_per_lane(fmt) columns and holds
// the slices of every row of X in registers; the weight words are unpacked
// once and dotted with each row's codes.  Same arithmetic per (row of X,
// weight row) as the batch-1 W4A8 lanes.
// ----------------------------------------------------------------------------
template <int FMT, int MB>
struct BatchLane;

// Four rows of X.
// Q4_K: 64 columns = the 32-byte quant chunk c of super-block sb: sub-block
// 2c in the low nibbles, sub-block 2c + 1 in the high nibbles.
template <>
struct BatchLane<QX_Q4_K, 4> {
    static constexpr int C = 64;
    static constexpr int MB = 4;
    uint32_t xq[MB][16];
    float dxs[MB][2];  // dx of sub-blocks 2c and 2c + 1, the second divided by 16
    float t[MB][2];    // dx * (sum of q_x): weight of the min term
    // row m of X (rows >= mvalid repeat row mvalid - 1); qstride: bytes per row of X's codes
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t* s, int64_t qstride,
                                         int mvalid, int l) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int64_t mm = m < mvalid ? m : mvalid - 1;
            const uint4* src = reinterpret_cast<const uint4*>(q + mm * qstride + int64_t(l) * C);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = src[k];
                xq[m][4 * k + 0] = v.x;
                xq[m][4 * k + 1] = v.y;
                xq[m][4 * k + 2] = v.z;
                xq[m][4 * k + 3] = v.w;
            }
            const int64_t b = mm * (qstride / 32) + 2 * l;
            const float d0 = d[b], d1 = d[b + 1];
            dxs[m][0] = d0;
            dxs[m][1] = d1 * 0.0625f;
            t[m][0] = d0 * float(s[b]);
            t[m][1] = d1 * float(s[b + 1]);
        }
    }
    __device__ __forceinline__ void row(const uint8_t* rp, int l, float (&out)[MB]) const {
        const int sb = l >> 2, c = l & 3;
        const uint8_t* bp = rp + sb * 144;
        const uint4 hdr = *reinterpret_cast<const uint4*>(bp);
        const uint4* qsp = reinterpret_cast<const uint4*>(bp + 16 + 32 * c);
        const uint4 a = qsp[0], b = qsp[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        int plo[MB], phi16[MB];  // phi16: 16 x the high-nibble partial (unsigned x signed dp4a)
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            plo[m] = 0;
            phi16[m] = 0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = w[i] & 0xF0F0F0F0u;
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                plo[m] = dp4a(lo, xq[m][i], plo[m]);
                phi16[m] = dp4a_us(hi, xq[m][8 + i], phi16[m]);
            }
        }
        const Q4KScales S = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
        const uint32_t scw = c < 2 ? S.sc_lo : S.sc_hi;
        const uint32_t mw = c < 2 ? S.m_lo : S.m_hi;
        const int k0 = 2 * (c & 1);
        const int sc0 = int(byte_of(scw, k0)), sc1 = int(byte_of(scw, k0 + 1));
        const float m0 = float(int(byte_of(mw, k0))), m1 = float(int(byte_of(mw, k0 + 1)));
        const float dd = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const float accd = fmaf(float(phi16[m] * sc1), dxs[m][1], float(plo[m] * sc0) * dxs[m][0]);
            const float accm = fmaf(m1, t[m][1], m0 * t[m][0]);
            out[m] = dd * accd - dmin * accm;
        }
    }
};

// Q6_K: 64 columns = quarters tp and tp + 2 of half h of super-block sb
// (they share the same 32 ql bytes, low and high nibbles, and the same qh
// bytes); four scale groups of 16.  The quants are dotted unsigned (0..63)
// and the -32 offset is applied as -32 * sum(q_x) per group.
template <>
struct BatchLane<QX_Q6_K, 4> {
    static constexpr int C = 64;
    static constexpr int MB = 4;
    uint32_t xq[MB][16];  // quarter tp (words 0..7), quarter tp + 2 (words 8..15)
    float dx[MB][2];
    int s16[MB][4];
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int64_t qstride,
                                         int mvalid, int l) {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
        const int64_t c0 = int64_t(sb) * 256 + 128 * h + 32 * tp;
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int64_t mm = m < mvalid ? m : mvalid - 1;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint4* src = reinterpret_cast<const uint4*>(q + mm * qstride + c0 + 64 * half);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const uint4 v = src[k];
                    xq[m][8 * half + 4 * k + 0] = v.x;
                    xq[m][8 * half + 4 * k + 1] = v.y;
                    xq[m][8 * half + 4 * k + 2] = v.z;
                    xq[m][8 * half + 4 * k + 3] = v.w;
                }
                dx[m][half] = d[mm * (qstride / 32) + (c0 + 64 * half) / 32];
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                int sg = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) sg = dp4a(xq[m][4 * g + i], 0x01010101u, sg);
                s16[m][g] = sg;
            }
        }
    }
    __device__ __forceinline__ void row(const uint8_t* rp, int l, float (&out)[MB]) const {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
        const uint8_t* bp = rp + sb * 210;
        uint32_t ql[8], qh[8], scw[2];
        load_words<8>(bp + 64 * h + 32 * tp, ql);
        load_words<8>(bp + 128 + 32 * h, qh);
        load_words<2>(bp + 192 + 8 * h, scw);
        // qh bits 2 tp, 2 tp + 1 (quarter tp) and 2 tp + 4, 2 tp + 5 (quarter tp + 2) to bits 4, 5
        const uint32_t sh_lo = 4u - 2u * uint32_t(tp), sh_hi = 2u * uint32_t(tp);
        int P[MB][4];
#pragma unroll
        for (int m = 0; m < MB; ++m)
#pragma unroll
            for (int g = 0; g < 4; ++g) P[m][g] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t wlo = (ql[i] & 0x0F0F0F0Fu) | ((qh[i] << sh_lo) & 0x30303030u);
            const uint32_t whi = ((ql[i] >> 4) & 0x0F0F0F0Fu) | ((qh[i] >> sh_hi) & 0x30303030u);
#pragma unroll
            for (int m = 0; m < MB; ++m) {
                P[m][i >> 2] = dp4a_us(wlo, xq[m][i], P[m][i >> 2]);
                P[m][2 + (i >> 2)] = dp4a_us(whi, xq[m][8 + i], P[m][2 + (i >> 2)]);
            }
        }
        // scale bytes of this half: 2 tp, 2 tp + 1 (quarter tp), 2 tp + 4, 2 tp + 5 (quarter tp + 2)
        const int sa = int(int8_t(byte_of(scw[0], 2 * tp))), sbb = int(int8_t(byte_of(scw[0], 2 * tp + 1)));
        const int sc = int(int8_t(byte_of(scw[1], 2 * tp))), sd = int(int8_t(byte_of(scw[1], 2 * tp + 1)));
        const float dd = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp + 208));
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int lo = sa * (P[m][0] - 32 * s16[m][0]) + sbb * (P[m][1] - 32 * s16[m][1]);
            const int hi = sc * (P[m][2] - 32 * s16[m][2]) + sd * (P[m][3] - 32 * s16[m][3]);
            out[m] = dd * fmaf(dx[m][1], float(hi), dx[m][0] * float(lo));
        }
    }
};

// Eight rows of X: 32-column lanes, so that eight slices fit in registers.
// Q4_K: 32 columns = sub-block j = 2c + hb of super-block sb: the low (hb =
// 0) or high (hb = 1) nibbles of quant chunk c.  The high nibbles are dotted
// in place (16 x q, the unsigned x signed dp4a) and the factor folded into dx.
template <>
struct BatchLane<QX_Q4_K, 8> {
    static constexpr int C = 32;
    static constexpr int MB = 8;
    uint32_t xq[MB][8];
    float dxs[MB];  // dx, divided by 16 for a high-nibble sub-block
    float t[MB];    // dx * (sum of q_x)
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t* s, int64_t qstride,
                                         int mvalid, int l) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int64_t mm = m < mvalid ? m : mvalid - 1;
            const uint4* src = reinterpret_cast<const uint4*>(q + mm * qstride + int64_t(l) * C);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint4 v = src[k];
                xq[m][4 * k + 0] = v.x;
                xq[m][4 * k + 1] = v.y;
                xq[m][4 * k + 2] = v.z;
                xq[m][4 * k + 3] = v.w;
            }
            const int64_t b = mm * (qstride / 32) + l;
            const float dx = d[b];
            dxs[m] = (l & 1) ? dx * 0.0625f : dx;
            t[m] = dx * float(s[b]);
        }
    }
    __device__ __forceinline__ void row(const uint8_t* rp, int l, float (&out)[MB]) const {
        const int sb = l >> 3, j = l & 7;
        const uint8_t* bp = rp + sb * 144;
        const uint4 hdr = *reinterpret_cast<const uint4*>(bp);
        const uint4* qsp = reinterpret_cast<const uint4*>(bp + 16 + 32 * (j >> 1));
        const uint4 a = qsp[0], b = qsp[1];
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const uint32_t mask = (j & 1) ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
        int P[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) P[m] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t wq = w[i] & mask;
#pragma unroll
            for (int m = 0; m < MB; ++m) P[m] = dp4a_us(wq, xq[m][i], P[m]);
        }
        const Q4KScales S = q4k_unpack_scales(hdr.y, hdr.z, hdr.w);
        const int sc = int(byte_of(j < 4 ? S.sc_lo : S.sc_hi, j & 3));
        const float mn = float(int(byte_of(j < 4 ? S.m_lo : S.m_hi, j & 3)));
        const float dd = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
#pragma unroll
        for (int m = 0; m < MB; ++m) out[m] = dd * (float(P[m] * sc) * dxs[m]) - dmin * (mn * t[m]);
    }
};

// Q6_K: 32 columns = quarter t of half h of super-block sb (ql bytes
// 64h + 32 (t & 1), low nibbles for t < 2, high for t >= 2; qh bits 2t,
// 2t + 1); two scale groups of 16.
template <>
struct BatchLane<QX_Q6_K, 8> {
    static constexpr int C = 32;
    static constexpr int MB = 8;
    uint32_t xq[MB][8];
    float dx[MB];
    int s16[MB][2];
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int64_t qstride,
                                         int mvalid, int l) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int64_t mm = m < mvalid ? m : mvalid - 1;
            const uint4* src = reinterpret_cast<const uint4*>(q + mm * qstride + int64_t(l) * C);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint4 v = src[k];
                xq[m][4 * k + 0] = v.x;
                xq[m][4 * k + 1] = v.y;
                xq[m][4 * k + 2] = v.z;
                xq[m][4 * k + 3] = v.w;
            }
            dx[m] = d[mm * (qstride / 32) + l];
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                int sg = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) sg = dp4a(xq[m][4 * g + i], 0x01010101u, sg);
                s16[m][g] = sg;
            }
        }
    }
    __device__ __forceinline__ void row(const uint8_t* rp, int l, float (&out)[MB]) const {
        const int sb = l >> 3, h = (l >> 2) & 1, tq = l & 3;
        const uint8_t* bp = rp + sb * 210;
        uint32_t ql[8], qh[8], scw;
        load_words<8>(bp + 64 * h + 32 * (tq & 1), ql);
        load_words<8>(bp + 128 + 32 * h, qh);
        scw = lds_u32_a2(bp + 192 + 8 * h + 2 * tq);  // scale bytes 2t, 2t + 1 of this half
        const uint32_t nib = (tq >> 1) * 4u, hsh = 2u * uint32_t(tq);
        int P[MB][2];
#pragma unroll
        for (int m = 0; m < MB; ++m) P[m][0] = P[m][1] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // the 6-bit quants of quarter t, one per byte
            const uint32_t wq = ((ql[i] >> nib) & 0x0F0F0F0Fu) | (((qh[i] >> hsh) & 0x03030303u) << 4);
#pragma unroll
            for (int m = 0; m < MB; ++m) P[m][i >> 2] = dp4a_us(wq, xq[m][i], P[m][i >> 2]);
        }
        const int s0 = int(int8_t(byte_of(scw, 0))), s1 = int(int8_t(byte_of(scw, 1)));
        const float dd = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp + 208));
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int acc = s0 * (P[m][0] - 32 * s16[m][0]) + s1 * (P[m][1] - 32 * s16[m][1]);
            out[m] = dd * (dx[m] * float(acc));
        }
    }
};

// Q8_0: 32 columns = one block (four or eight rows of X).
template <int MB_>
struct BatchLane<QX_Q8_0, MB_> {
    static constexpr int C = 32;
    static constexpr int MB = MB_;
    uint32_t xq[MB][8];
    float dx[MB];
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int64_t qstride,
                                         int mvalid, int l) {
#pragma unroll
        for (int m = 0; m < MB; ++m) {
            const int64_t mm = m < mvalid ? m : mvalid - 1;
            const uint4* src = reinterpret_cast<const uint4*>(q + mm * qstride + int64_t(l) * C);
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint4 v = src[k];
                xq[m][4 * k + 0] = v.x;
                xq[m][4 * k + 1] = v.y;
                xq[m][4 * k + 2] = v.z;
                xq[m][4 * k + 3] = v.w;
            }
            dx[m] = d[mm * (qstride / 32) + l];
        }
    }
    __device__ __forceinline__ void row(const uint8_t* rp, int l, float (&out)[MB]) const {
        const uint8_t* bp = rp + l * 34;
        uint32_t qs[8];
        load_words<8>(bp + 2, qs);
        int P[MB];
#pragma unroll
        for (int m = 0; m < MB; ++m) P[m] = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int m = 0; m < MB; ++m) P[m] = dp4a(qs[i], xq[m][i], P[m]);
        const float dd = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp));
#pragma unroll
        for (int m = 0; m < MB; ++m) out[m] = dd * dx[m] * float(P[m]);
    }
};

// All rows of one stage for the batched lanes: team t takes rows t,
// t + nteams, ...; the partial of (row i, activation row m) goes to
// red[(i * MB + m) * RS + slice].
template <int FMT, int MB>
__device__ __forceinline__ void consume_stage_batch(const BatchLane<FMT, MB>& X, const Team& tm,
                                                    const uint8_t* sbuf, int nrows, uint32_t rb, float* red, int RS) {
    if (!tm.active) return;
    for (int i = tm.team; i < nrows; i += tm.nteams) {
        float v[MB];
        X.row(sbuf + uint32_t(i) * rb, tm.slice, v);
#pragma unroll
        for (int m = 0; m < MB; ++m) red[(i * MB + m) * RS + tm.slice] = v[m];
    }
}

// The reducer's share of one batched stage: one (row, activation row) pair
// per lane, its L partials added in the same fixed order as reduce_stage;
// y[m * y_stride + row] for m < mvalid.
template <int MB>
__device__ __forceinline__ void reduce_stage_batch(const float* red, int RS, int L, int nrows, float* y,
                                                   int64_t y_stride, int mvalid, int lane) {
    for (int pair = lane; pair < nrows * MB; pair += 32) {
        const int row = pair / MB, m = pair % MB;
        const float* pr = red + pair * RS;
        float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
        int s = 0;
        for (; s + 16 <= L; s += 16) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4*>(pr + s + 4 * u);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a0 += v[u].x;
                a1 += v[u].y;
                a2 += v[u].z;
                a3 += v[u].w;
            }
        }
        for (; s + 4 <= L; s += 4) {
            const float4 v = *reinterpret_cast<const float4*>(pr + s);
            a0 += v.x;
            a1 += v.y;
            a2 += v.z;
            a3 += v.w;
        }
        if (s < L) a0 += pr[s];
        if (s + 1 < L) a1 += pr[s + 1];
        if (s + 2 < L) a2 += pr[s + 2];
        if (m < mvalid) y[int64_t(m) * y_stride + row] = (a0 + a1) + (a2 + a3);
    }
}

// Load a lane's activation slice: from the quantised activation (W4A8) or
// the f32 activation.
template <int MODE, class LaneT>
__device__ __forceinline__ void load_slice(LaneT& X, const int8_t* q, const float* d, const int32_t* s,
                                           const float* xf, int slice, bool swz) {
    if constexpr (MODE == QX_MODE_W4A8) {
        X.load(q, d, s, slice, swz);
    } else {
        X.load(xf, slice);
    }
}

// Synchronise warps 0 .. WARPS - 1 only (the consumers; the producer and
// reducer warps never join).
template <int WARPS>
__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(WARPS * 32) : "memory");
}

// The same named barrier over the first `threads` threads (a multiple of 32,
// uniform over the CTA): the warps that quantise the activation in-kernel.
__device__ __forceinline__ void quantiser_barrier(int threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

}  // namespace lanes
}  // namespace qx
