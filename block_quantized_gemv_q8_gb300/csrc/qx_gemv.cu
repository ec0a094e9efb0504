// qx_gemv.cu -- batch-1 GEMV over GGUF-style block-quantised rows (Q4_K,
// Q6_K, Q8_0) for sm_103a, in f32 mode and W4A8 mode.
//
// Decode is weight-bandwidth-bound (VKNN wiki, "Running an LLM on VKNN",
// section "Performance": one token streams every weight once and the wide
// lm_head is the largest single op), so the kernel is a weight stream:
//
//   * Each CTA owns a contiguous range of rows (rows are independent:
//     llambda.lisp README, "Features & Architecture", the GEMV's outer loop
//     runs in parallel with isolated, lock-free writes).  Its rows are
//     contiguous bytes, streamed in stages of G whole rows by 1-D bulk copies
//     (TMA) into a ring of shared-memory slots, issued by one producer warp
//     and completed on mbarriers.  G is a multiple of the number of rows
//     whose bytes make a 16-byte multiple, so every copy is 16-byte aligned.
//   * Consumer lanes own a fixed slice of columns for the whole kernel, so
//     the activation slice stays in registers.  A "team" of lanes covers one
//     row; teams take the rows of a stage in turn and reduce with warp
//     shuffles (plus one shared-memory step when a row needs several warps).
//   * W4A8 (llamay docs, "Backends and hardware", sections "CPU" and
//     "CUDA"): per 32-weight sub-block (16 for Q6_K) the int8 x int4/int6/int8
//     products are summed exactly with dp4a, and only then scaled; the weight
//     rows are never materialised.
//   * f32 mode (llambda.lisp README, "Features & Architecture"): every quant
//     is converted exactly to f32 and fused-multiply-added with the f32
//     activation; the per-sub-block scale d*sc (and the Q4_K min term
//     dmin*m*sum(x)) is applied once per sub-block, which is the same sum
//     reassociated.
#include "qx_device.cuh"
#include "qx_internal.h"

namespace qx {

namespace {

constexpr int NW = kGemvConsumerWarps;

// Exact f32 value of a small non-negative integer n < 2^23, via the exponent
// trick: the float with bits 0x4B000000 | n is 2^23 + n.
__device__ __forceinline__ float small_uint_to_f32(uint32_t n) {
    return __int_as_float(0x4B000000u | n) - 8388608.0f;
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
    static constexpr int kRows = 2;    // rows per call
    uint32_t xq[32];
    float dxs[4];  // dx of sub-block u; the odd (high-nibble) ones divided by 16
    float t[4];    // dx * (sum of q_x) of sub-block u: weight of the min term
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t* s, int l) {
        const uint4* src = reinterpret_cast<const uint4*>(q + int64_t(l) * C);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = src[k];
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
    float x[64];
    float xsum[2];
    __device__ __forceinline__ void load(const float* xp, int l) {
        const float4* src = reinterpret_cast<const float4*>(xp + int64_t(l) * C);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const float4 v = src[k];
            x[4 * k + 0] = v.x;
            x[4 * k + 1] = v.y;
            x[4 * k + 2] = v.z;
            x[4 * k + 3] = v.w;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float s = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) s += x[32 * u + i];
            xsum[u] = s;
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 2, c = l & 3;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 144;
            const uint4 hdr = *reinterpret_cast<const uint4*>(bp);
            const uint4* qsp = reinterpret_cast<const uint4*>(bp + 16 + 32 * c);
            const uint4 a = qsp[0], b = qsp[1];
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
            float slo = 0.0f, shi = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    slo = fmaf(small_uint_to_f32((w[i] >> (8 * k)) & 15u), x[4 * i + k], slo);
                    shi = fmaf(small_uint_to_f32((w[i] >> (8 * k + 4)) & 15u), x[32 + 4 * i + k], shi);
                }
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
    uint32_t ql[16], qh[8];
    load_words<16>(bp + 64 * h, ql);
    load_words<8>(bp + 128 + 32 * h, qh);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        int pu[2] = {0, 0};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t src = ql[8 * (t & 1) + i];
            const uint32_t lo4 = (t < 2 ? src : (src >> 4)) & 0x0F0F0F0Fu;
            const uint32_t hi2 = ((qh[i] >> (2 * t)) & 0x03030303u) << 4;
            pu[i >> 2] = dp4a_us(lo4 | hi2, xq[8 * t + i], pu[i >> 2]);
        }
        P[2 * t] = pu[0] - 32 * s16[2 * t];
        P[2 * t + 1] = pu[1] - 32 * s16[2 * t + 1];
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
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int l) {
        const uint4* src = reinterpret_cast<const uint4*>(q + int64_t(l) * C);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = src[k];
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
    float x[64];
    __device__ __forceinline__ void load(const float* xp, int l) {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
        const int64_t c0 = int64_t(sb) * 256 + 128 * h + 32 * tp;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const float4* src = reinterpret_cast<const float4*>(xp + c0 + 64 * half);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float4 v = src[k];
                x[32 * half + 4 * k + 0] = v.x;
                x[32 * half + 4 * k + 1] = v.y;
                x[32 * half + 4 * k + 2] = v.z;
                x[32 * half + 4 * k + 3] = v.w;
            }
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
        const int sb = l >> 2, h = (l >> 1) & 1, tp = l & 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + sb * 210;
            uint32_t ql[8], qh[8], scw[2];
            load_words<8>(bp + 64 * h + 32 * tp, ql);
            load_words<8>(bp + 128 + 32 * h, qh);
            load_words<2>(bp + 192 + 8 * h, scw);
            float sg[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // lo g0, lo g1, hi g0, hi g1
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t nlo = ((ql[i] >> (8 * k)) & 15u) | (((qh[i] >> (8 * k + 2 * tp)) & 3u) << 4);
                    const uint32_t nhi =
                        ((ql[i] >> (8 * k + 4)) & 15u) | (((qh[i] >> (8 * k + 2 * tp + 4)) & 3u) << 4);
                    // exact q - 32 in f32: the float with bits 0x4B000000 | q is 2^23 + q
                    sg[i >> 2] = fmaf(__int_as_float(0x4B000000u | nlo) - 8388640.0f, x[4 * i + k], sg[i >> 2]);
                    sg[2 + (i >> 2)] =
                        fmaf(__int_as_float(0x4B000000u | nhi) - 8388640.0f, x[32 + 4 * i + k], sg[2 + (i >> 2)]);
                }
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

// Q8_0, W4A8: 32 columns = one block.
template <>
struct Lane<QX_Q8_0, QX_MODE_W4A8> {
    static constexpr int C = 32;
    static constexpr int kGroups = 1;
    static constexpr int kRows = 2;
    uint32_t xq[8];
    float dx;
    __device__ __forceinline__ void load(const int8_t* q, const float* d, const int32_t*, int l) {
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
    float x[32];
    __device__ __forceinline__ void load(const float* xp, int l) {
        const float4* src = reinterpret_cast<const float4*>(xp + int64_t(l) * C);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = src[k];
            x[4 * k + 0] = v.x;
            x[4 * k + 1] = v.y;
            x[4 * k + 2] = v.z;
            x[4 * k + 3] = v.w;
        }
    }
    template <int R>
    __device__ __forceinline__ void rows(const uint8_t* const (&rp)[R], int l, float (&out)[R]) const {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint8_t* bp = rp[r] + l * 34;
            uint32_t qs[8];
            load_words<8>(bp + 2, qs);
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // int8 -> f32 exactly: bias the byte by 128 into [0, 255].
                    const uint32_t u = ((qs[i] >> (8 * k)) & 0xFFu) ^ 0x80u;
                    acc = fmaf(__int_as_float(0x4B000000u | u) - 8388736.0f, x[4 * i + k], acc);
                }
            }
            out[r] = f16_bits_to_f32(*reinterpret_cast<const uint16_t*>(bp)) * acc;
        }
    }
};

// ----------------------------------------------------------------------------
// Work distribution
// ----------------------------------------------------------------------------

// First row (in the concatenated row space) of CTA i: an even split of the
// rows, rounded down within its entry to a multiple of the alignment quantum.
__device__ __forceinline__ int64_t cta_row_begin(const GemvParams& p, int i) {
    if (i >= p.n_cta) return p.total_rows;
    const int64_t raw = p.total_rows * int64_t(i) / p.n_cta;
    int e = 0;
    while (e + 1 < p.n_entries && raw >= p.e[e + 1].row0) ++e;
    const int64_t local = raw - p.e[e].row0;
    return p.e[e].row0 + (local - local % p.quantum);
}

// Walks one CTA's rows as a sequence of stages: at most G rows, never
// crossing an entry boundary.
struct StageWalker {
    int64_t g, gend;
    int e;
    __device__ __forceinline__ bool next(const GemvParams& p, int& entry, int64_t& lrow, int& nrows) {
        if (g >= gend) return false;
        while (g >= p.e[e].row0 + p.e[e].rows) ++e;
        const int64_t entry_end = p.e[e].row0 + p.e[e].rows;
        const int64_t stop = gend < entry_end ? gend : entry_end;
        const int64_t n = stop - g < p.G ? stop - g : p.G;
        entry = e;
        lrow = g - p.e[e].row0;
        nrows = static_cast<int>(n);
        g += n;
        return true;
    }
};

// W4A8 kernels and Q8_0 kernels fit two CTAs per SM (<= 112 registers), so
// that with programmatic dependent launch the next GEMV's CTA can be resident
// next to this one and stream its weights while this one finishes.
template <int FMT, int MODE>
constexpr int gemv_min_blocks() {
    return (MODE == QX_MODE_W4A8 || FMT == QX_Q8_0) ? 2 : 1;
}

// Synchronise the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

template <int FMT, int MODE, bool PART>
__global__ void __launch_bounds__(kGemvThreads, gemv_min_blocks<FMT, MODE>())
    gemv_kernel(const __grid_constant__ GemvParams p) {
    using LaneT = Lane<FMT, MODE>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int S = p.stages;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + S;
    // Cross-warp row sums (rows wider than one warp): per (slot, row of
    // stage) one partial per warp of the team and an arrival counter; the
    // last warp to arrive adds them in warp order and writes y, so no warp
    // ever waits on another.
    int* red_cnt = reinterpret_cast<int*>(smem + p.red_off);  // [S][G]
    float* red = reinterpret_cast<float*>(red_cnt + S * p.G);   // [S][G][team_warps]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = cta_row_begin(p, blockIdx.x), r1 = cta_row_begin(p, blockIdx.x + 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        if (p.team_warps > 1)
            for (int i = 0; i < S * p.G; ++i) red_cnt[i] = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();

    if (warp == NW) {
        // ---------------- producer: one lane issues every bulk copy ----------
        // Weights are never written by the preceding kernel, so they are
        // fetched before the programmatic dependency on it is resolved.
        if (lane != 0) return;
        StageWalker wk{r0, r1, 0};
        const uint64_t policy = policy_evict_first();
        int e, nrows;
        int64_t lrow;
        int issued = 0;
        unsigned tail_slots = 0;  // slots whose bytes were last written by plain stores
        for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
            const int slot = k % S;
            if (k >= S && !mbar_wait_bounded(&empty[slot], ((k / S) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                break;
            const uint8_t* src = p.e[e].W + lrow * p.row_bytes;
            const uint32_t bytes = static_cast<uint32_t>(int64_t(nrows) * p.row_bytes);
            const uint32_t abytes = bytes & ~15u;
            uint8_t* dst = smem + size_t(slot) * p.slot_bytes;
            if (bytes != abytes) {
                // The last < 16 bytes of a matrix whose size is not a 16-byte multiple.
                for (uint32_t t = abytes; t < bytes; ++t) dst[t] = src[t];
                tail_slots |= 1u << slot;
            } else if (tail_slots & (1u << slot)) {
                fence_proxy_async_smem();
                tail_slots &= ~(1u << slot);
            }
            mbar_arrive_expect_tx(&full[slot], abytes);
            if (abytes) bulk_g2s_evict_first(dst, src, abytes, &full[slot], policy);
            issued = k + 1;
        }
        // Keep the CTA alive until every copy it issued has landed.
        for (int k = issued > S ? issued - S : 0; k < issued; ++k)
            mbar_wait_bounded(&full[k % S], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
        return;
    }

    // ---------------- consumers ----------------------------------------------
    int team, slice;
    if (p.team_warps == 1) {
        team = warp * (32 / p.team_lanes) + lane / p.team_lanes;
        slice = lane % p.team_lanes;
    } else {
        team = warp / p.team_warps;
        slice = (warp % p.team_warps) * 32 + lane;
    }
    const bool in_team = team < p.nteams;
    const bool active = in_team && slice < p.L;

    pdl_wait_prior_grid();  // the activation may come from the previous kernel
    LaneT X;
    if constexpr (MODE == QX_MODE_W4A8) {
        const int8_t* q = p.xq;
        const float* d = p.xd;
        const int32_t* s = p.xs;
        if (p.xf != nullptr) {
            // Quantise the f32 activation once per CTA into shared memory,
            // with the same code as qx_quantize_act_q8.
            int8_t* sq = reinterpret_cast<int8_t*>(smem + p.act_off);
            float* sd = reinterpret_cast<float*>(sq + p.cols);
            int32_t* ss = reinterpret_cast<int32_t*>(sd + p.cols / 32);
            // two adjacent lanes per block of 32; all consumer lanes take part
            const int nblk = static_cast<int>(p.cols / 32);
            for (int base = 0; base < 2 * nblk; base += NW * 32)
                quantize_task(p.xf, nblk, base + threadIdx.x, sq, sd, ss);
            consumer_barrier();
            q = sq;
            d = sd;
            s = ss;
        }
        if (active) X.load(q, d, s, slice);
    } else {
        if (active) X.load(p.x, slice);
    }

    constexpr int R = PART ? 1 : LaneT::kRows;
    static_assert(PART || LaneT::kRows == gemv_rows_per_call(FMT, MODE), "row count must match the host geometry");
    const uint32_t rb = static_cast<uint32_t>(p.row_bytes);
    StageWalker wk{r0, r1, 0};
    int e, nrows;
    int64_t lrow;
    for (int k = 0; wk.next(p, e, lrow, nrows); ++k) {
        const int slot = k % S;
        if (!mbar_wait_bounded(&full[slot], (k / S) & 1, p.wait_ns, p.err, kErrTimeoutFull)) break;
        const uint8_t* sbuf = smem + size_t(slot) * p.slot_bytes;
        for (int ib = 0; ib < nrows; ib += p.nteams * R) {
            int ir[R];
            bool vr[R];
            const uint8_t* rp[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                ir[r] = ib + team + r * p.nteams;
                vr[r] = in_team && ir[r] < nrows;
                rp[r] = sbuf + (vr[r] ? uint32_t(ir[r]) : 0u) * rb;
            }
            if constexpr (PART) {
                if (vr[0] && active) {
                    int P[LaneT::kGroups];
                    X.partials(rp[0], slice, P);
                    const int64_t ng = p.cols / (FMT == QX_Q6_K ? 16 : 32);
                    int32_t* dst = p.e[e].P + (lrow + ir[0]) * ng;
#pragma unroll
                    for (int g = 0; g < LaneT::kGroups; ++g) dst[LaneT::part_index(slice, g)] = P[g];
                }
                continue;
            } else {
                float v[R];
                if (active) {
                    X.template rows<R>(rp, slice, v);
                } else {
#pragma unroll
                    for (int r = 0; r < R; ++r) v[r] = 0.0f;
                }
                float* yb = p.e[e].y + lrow;
                if (p.team_warps == 1) {
                    if (R == 2 && p.team_lanes == 32) {
                        // two rows in one butterfly: lanes 0-15 end with row 0, 16-31 with row 1
                        float a = (lane & 16) ? v[R - 1] : v[0];
                        const float b = (lane & 16) ? v[0] : v[R - 1];
                        a += __shfl_xor_sync(0xffffffffu, b, 16);
#pragma unroll
                        for (int o = 8; o >= 1; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                        if (lane == 0 && vr[0]) yb[ir[0]] = a;
                        if (lane == 16 && vr[R - 1]) yb[ir[R - 1]] = a;
                    } else {
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            for (int o = p.team_lanes >> 1; o >= 1; o >>= 1)
                                v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
                            if (vr[r] && slice == 0) yb[ir[r]] = v[r];
                        }
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < R; ++r) {
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) v[r] += __shfl_xor_sync(0xffffffffu, v[r], o);
                        if (vr[r] && lane == 0) {
                            const int ri = slot * p.G + ir[r];
                            float* rbuf = red + ri * p.team_warps;
                            rbuf[warp % p.team_warps] = v[r];
                            __threadfence_block();
                            if (atomicAdd(&red_cnt[ri], 1) == p.team_warps - 1) {
                                __threadfence_block();
                                float sum = 0.0f;
                                for (int w = 0; w < p.team_warps; ++w) sum += rbuf[w];
                                yb[ir[r]] = sum;
                                red_cnt[ri] = 0;
                            }
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }
}

// Largest dynamic shared memory a CTA may use on sm_103a.
constexpr int kMaxDynamicSmem = 227 * 1024;

// Raise the kernel's dynamic shared-memory limit to the maximum, once per
// kernel and device.  Occupancy and launches then depend only on the bytes
// each launch asks for.
template <int FMT, int MODE, bool PART>
cudaError_t configure_once() {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    err = cudaFuncSetAttribute(gemv_kernel<FMT, MODE, PART>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMaxDynamicSmem);
    if (err == cudaSuccess) done[dev] = true;
    return err;
}

template <int FMT, int MODE, bool PART>
cudaError_t launch_one(const GemvParams& p, size_t smem, cudaStream_t s, bool pdl) {
    cudaError_t err = configure_once<FMT, MODE, PART>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.n_cta);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<FMT, MODE, PART>, p);
}

template <int FMT, int MODE, bool PART>
cudaError_t occupancy_one(size_t smem, int* out) {
    cudaError_t err = configure_once<FMT, MODE, PART>();
    if (err != cudaSuccess) return err;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, gemv_kernel<FMT, MODE, PART>, kGemvThreads, smem);
}

}  // namespace

cudaError_t launch_gemv(int fmt, int mode, bool partials, const GemvParams& p, size_t smem, cudaStream_t s,
                        bool pdl) {
    switch (fmt * 4 + mode * 2 + (partials ? 1 : 0)) {
        case QX_Q4_K * 4 + 0: return launch_one<QX_Q4_K, QX_MODE_F32, false>(p, smem, s, pdl);
        case QX_Q4_K * 4 + 2: return launch_one<QX_Q4_K, QX_MODE_W4A8, false>(p, smem, s, pdl);
        case QX_Q4_K * 4 + 3: return launch_one<QX_Q4_K, QX_MODE_W4A8, true>(p, smem, s, pdl);
        case QX_Q6_K * 4 + 0: return launch_one<QX_Q6_K, QX_MODE_F32, false>(p, smem, s, pdl);
        case QX_Q6_K * 4 + 2: return launch_one<QX_Q6_K, QX_MODE_W4A8, false>(p, smem, s, pdl);
        case QX_Q6_K * 4 + 3: return launch_one<QX_Q6_K, QX_MODE_W4A8, true>(p, smem, s, pdl);
        case QX_Q8_0 * 4 + 0: return launch_one<QX_Q8_0, QX_MODE_F32, false>(p, smem, s, pdl);
        case QX_Q8_0 * 4 + 2: return launch_one<QX_Q8_0, QX_MODE_W4A8, false>(p, smem, s, pdl);
        case QX_Q8_0 * 4 + 3: return launch_one<QX_Q8_0, QX_MODE_W4A8, true>(p, smem, s, pdl);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t gemv_max_ctas_per_sm(int fmt, int mode, bool partials, size_t smem, int* out) {
    switch (fmt * 4 + mode * 2 + (partials ? 1 : 0)) {
        case QX_Q4_K * 4 + 0: return occupancy_one<QX_Q4_K, QX_MODE_F32, false>(smem, out);
        case QX_Q4_K * 4 + 2: return occupancy_one<QX_Q4_K, QX_MODE_W4A8, false>(smem, out);
        case QX_Q4_K * 4 + 3: return occupancy_one<QX_Q4_K, QX_MODE_W4A8, true>(smem, out);
        case QX_Q6_K * 4 + 0: return occupancy_one<QX_Q6_K, QX_MODE_F32, false>(smem, out);
        case QX_Q6_K * 4 + 2: return occupancy_one<QX_Q6_K, QX_MODE_W4A8, false>(smem, out);
        case QX_Q6_K * 4 + 3: return occupancy_one<QX_Q6_K, QX_MODE_W4A8, true>(smem, out);
        case QX_Q8_0 * 4 + 0: return occupancy_one<QX_Q8_0, QX_MODE_F32, false>(smem, out);
        case QX_Q8_0 * 4 + 2: return occupancy_one<QX_Q8_0, QX_MODE_W4A8, false>(smem, out);
        case QX_Q8_0 * 4 + 3: return occupancy_one<QX_Q8_0, QX_MODE_W4A8, true>(smem, out);
        default: return cudaErrorInvalidValue;
    }
}

// ----------------------------------------------------------------------------
// Bounded-wait probe: one warp waits on an mbarrier that nothing completes.
// ----------------------------------------------------------------------------
__global__ void timeout_probe_kernel(unsigned* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    mbar_wait_bounded(&bar, 0, limit_ns, err, kErrTimeoutProbe);
}

cudaError_t launch_timeout_probe(unsigned* err, uint64_t limit_ns, cudaStream_t s) {
    timeout_probe_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

}  // namespace qx
