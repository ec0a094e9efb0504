// qx_tc.cu -- the prefill contraction on the fifth-generation tensor cores
// (tcgen05 MMA, accumulator in tensor memory, operands staged by TMA).
//
// The W4A8 prefill product (llamay docs, "Backends and hardware", sections
// "CPU" and "CUDA") is Y[m, n] = sum_k xhat[m, k] * what[n, k] with
// xhat = dx * q_x (the dequantised int8 activation) and what the dequantised
// weight (Q4_K: d*sc*q - dmin*m, Q6_K: d*sc*(q - 32), Q8_0: d*q).  sm_103a has
// no integer tensor-core MMA, and the per-block scales differ along K, so the
// integer partial sums cannot be scaled inside the MMA accumulation.  Instead
// each operand is written as two bf16 terms whose sum carries 16 significant
// bits (hi = bf16(v), lo = bf16(v - hi)), and
//     Y = Xh Wh^T + Xh Wl^T + Xl Wh^T
// is accumulated in f32 in tensor memory.  The dropped Xl Wl^T term and the
// split rounding bound the error of every product by about 2^-15 of
// |xhat * what|, well inside the tolerance of 1e-4 * sum |w * x| per output.
//
// One kernel per format, and no pass outside it.  A CTA computes a 256 x 128
// tile of Y (256 rows of X, 128 weight rows) as two 128 x 128 accumulators in
// tensor memory that share every converted weight slice.  Per K group TMA
// brings the raw blocks of the 128 weight rows into shared memory; sixteen
// converter warps dequantise them and the int8 activation codes of the 256
// rows, 32 columns (one activation block) per K slice, split both into hi and
// lo bf16 and write them straight into the 64-byte-swizzled K-major tiles the
// tensor cores read; one thread issues the split products (M = 128, N = 128,
// K = 16 each).  The activation codes and scales go from global memory (L2:
// every CTA of an M tile reads them) straight into the converters' registers,
// several slices ahead; three operand stages let the conversion run up to two
// slices ahead of the tensor cores.  The
// library needs no workspace, so the call allocates nothing and may be
// captured in a CUDA graph on first use.
//
// Weight rows (llamay docs, "Backends and hardware", section "CUDA": the
// prefill kernel should stage the next weight tile behind the current
// multiply): rows that are a 16-byte multiple (Q4_K always; Q6_K and Q8_0 at
// 2048 and 256 columns and their multiples) come as one 2-D box per group and
// tile.  Otherwise each row's group is fetched by a 1-D box that starts at the
// 16-byte boundary at or below it (the group plus up to 14 bytes before it),
// and the converter indexes from the remainder.  Boxes that run past the end
// of a row or of the matrix are zero-filled by the copy engine, never read
// out of bounds.
//
// Every wait is bounded and reports through the device error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>

#include "qx_device.cuh"
#include "qx_internal.h"

namespace qx {

namespace {

constexpr int TBM = 256, TBN = 128, TBK = 32;  // CTA tile; K slice
constexpr int OP_STAGES = 3;               // operand stages: conversion runs up to two slices ahead of the MMAs
constexpr int T_TILE = 128 * TBK * 2;       // one 128-row x 32 bf16 tile: 8 KB
// one K slice of operands: Xh (two 128-row halves), Xl (two halves), Wh, Wl
constexpr int OP_XH = 0, OP_XL = 2 * T_TILE, OP_WH = 4 * T_TILE, OP_WL = 5 * T_TILE, OP_BYTES = 6 * T_TILE;
constexpr int kXAhead = 4;                  // slices of activation codes and scales in flight per thread
constexpr int kConvWarps = 16;              // converter warps; the first eight drain the accumulators
constexpr int kTcThreads = 32 * (2 + kConvWarps);
constexpr int kRowStride1d = 256;           // shared-memory row stride of the per-row boxes (128-byte aligned)
constexpr uint32_t kIdesc =  // kind::f16: f32 accumulator, bf16 A and B, both K-major, M = 128, N = 128
    (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(TBN >> 3) << 17) | (uint32_t(128 >> 4) << 24);

// Raw weight groups per format: K columns per group, its bytes in a row, the
// box fetched per row (bytes, a 16-byte multiple covering the group from the
// 16-byte boundary at or below it), and the number of shared-memory slots.
template <int FMT>
struct RawGeom;
template <>
struct RawGeom<QX_Q4_K> {
    static constexpr int kGroupK = 256, kGroupBytes = 144, kBox = 144, kSlots = 3;
};
template <>
struct RawGeom<QX_Q6_K> {
    static constexpr int kGroupK = 256, kGroupBytes = 210, kBox = 224, kSlots = 2;
};
template <>
struct RawGeom<QX_Q8_0> {
    static constexpr int kGroupK = 128, kGroupBytes = 136, kBox = 160, kSlots = 2;
};
// Bytes of one raw slot (128 rows): dense rows of the 2-D box, or the per-row
// boxes at kRowStride1d.
template <int FMT>
__host__ __device__ constexpr int raw_slot_bytes() {
    return (FMT == QX_Q4_K ? RawGeom<FMT>::kBox : kRowStride1d) * TBN;
}

template <int FMT>
constexpr size_t tc_smem_bytes() {
    return size_t(OP_STAGES) * OP_BYTES + size_t(RawGeom<FMT>::kSlots) * raw_slot_bytes<FMT>() + 1024 + 256;
}
static_assert(tc_smem_bytes<QX_Q6_K>() <= 227 * 1024 && tc_smem_bytes<QX_Q8_0>() <= 227 * 1024 &&
                  tc_smem_bytes<QX_Q4_K>() <= 227 * 1024,
              "a CTA's shared memory");

struct TcParams {
    CUtensorMap w_map;  // [N rows, row_bytes] bytes, boxes kBox x 128 (w2d); else all N * row_bytes bytes, 1-D boxes
    const int8_t* xq;   // [M, K] activation codes, 16-byte aligned (K a multiple of 32)
    const float* xd;    // [M, K / 32] activation scales
    int M, N, K;
    int w2d;            // 1: weight rows are a 16-byte multiple, one 2-D box per group
    int tiles_m;        // M tiles; tile i is M tile i % tiles_m of N tile i / tiles_m
    int tile_base;      // the launch's first tile
    int split;          // 0, or the CTAs per tile (a cluster of 2 or 4), each taking its share of the K groups
    int64_t row_bytes;
    float* Y;           // [M, N] f32
    unsigned* err;
    unsigned long long wait_ns;
};

// ---------------------------------------------------------------------------
// tcgen05 and TMA helpers
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor of a K-major tile with the 64-byte swizzle:
// rows of 64 bytes (32 bf16), 8-row atoms 512 bytes apart; within an atom the
// 16-byte chunk j of row r sits at chunk j ^ ((r / 2) % 4).
__device__ __forceinline__ uint64_t sw64_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFF) >> 4);  // start address
    d |= uint64_t(1) << 16;                  // leading byte offset (unused for swizzled K-major)
    d |= uint64_t(512 >> 4) << 32;           // stride byte offset: one 8-row atom
    d |= uint64_t(1) << 46;                  // descriptor version
    d |= uint64_t(4) << 61;                  // 64-byte swizzle
    return d;
}
// Byte offset of 16-byte chunk j of row r in such a tile.
__device__ __forceinline__ uint32_t sw64_off(int r, int j) {
    return uint32_t(r) * 64u + uint32_t((j ^ ((r >> 1) & 3)) << 4);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_addr(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}
// x: a byte offset that is a multiple of 16 (the copy engine's rule for the
// innermost coordinate); bytes past the end of the tensor arrive as zeros.
__device__ __forceinline__ void tma_load_1d(void* dst, const CUtensorMap* map, int x, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2}], [%3];" ::"r"(
            smem_addr(dst)),
        "l"(map), "r"(x), "r"(smem_addr(bar))
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
// Thread-block clusters: this CTA's rank, the address of one of this CTA's
// shared-memory locations in the cluster's CTA `rank`, a 16-byte store there,
// and a barrier over every thread of the cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t peer_addr(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_peer_v4(uint32_t raddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(raddr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_peer_v4(uint32_t raddr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(raddr)
                 : "memory");
    return v;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
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

// ---------------------------------------------------------------------------
// operand conversion: 16 consecutive K values of one row into hi / lo bf16
// (two 16-byte chunks each)
// ---------------------------------------------------------------------------

// Split 2N f32 values, pairs in packed f32x2 form, into hi = bf16(v) and
// lo = bf16(v - hi), both rounded to nearest (v - hi is exact in f32): hi + lo
// is within 2^-17 |v| of v.  (The subtraction is a scalar round-to-nearest
// intrinsic: ptxas may fold packed two-wide cancellation patterns such as
// g - (g - v) at -O3.)
template <int N>
__device__ __forceinline__ void split_pairs(const uint64_t (&v)[N], uint32_t (&h)[N], uint32_t (&l)[N]) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float2 f = f32x2_unpack(v[i]);
        const __nv_bfloat162 hb = __floats2bfloat162_rn(f.x, f.y);
        h[i] = *reinterpret_cast<const uint32_t*>(&hb);
        const float h0 = __uint_as_float(h[i] << 16), h1 = __uint_as_float(h[i] & 0xFFFF0000u);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(__fsub_rn(f.x, h0), __fsub_rn(f.y, h1));
        l[i] = *reinterpret_cast<const uint32_t*>(&lb);
    }
}
__device__ __forceinline__ void split16(const uint64_t (&v)[8], uint4 (&hi)[2], uint4 (&lo)[2]) {
    uint32_t h[8], l[8];
    split_pairs<8>(v, h, l);
    hi[0] = make_uint4(h[0], h[1], h[2], h[3]);
    hi[1] = make_uint4(h[4], h[5], h[6], h[7]);
    lo[0] = make_uint4(l[0], l[1], l[2], l[3]);
    lo[1] = make_uint4(l[4], l[5], l[6], l[7]);
}
__device__ __forceinline__ void split8(const uint64_t (&v)[4], uint4& hi, uint4& lo) {
    uint32_t h[4], l[4];
    split_pairs<4>(v, h, l);
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// Byte k of w as the float 2^23 + byte (one byte-permute into the exponent
// pattern 0x4B); the caller subtracts 2^23 (plus any offset) exactly.
__device__ __forceinline__ float byte_biased(uint32_t w, int k) {
    return __int_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + uint32_t(k)));
}

// N little-endian words at the 2-byte-aligned shared-memory address p: N + 1
// aligned words, funnel-shifted (reads up to 4 bytes past the N words).
template <int N>
__device__ __forceinline__ void words_a2(const uint8_t* p, uint32_t (&out)[N]) {
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

__device__ __forceinline__ float f16_at_a2(const uint8_t* p) {
    return __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(p)));
}

// Bytes k, k + 1 of w as the packed floats (2^23 + byte_k, 2^23 + byte_k+1).
__device__ __forceinline__ uint64_t byte_pair_biased(uint32_t w, int k) {
    return f32x2_pack(byte_biased(w, k), byte_biased(w, k + 1));
}

// The activation: xhat = dx * q for the 16 codes in c (little-endian bytes);
// q comes out exactly (bytes offset by 128 into 2^23 + 128 + q, minus the
// same), then one rounding in the multiply.
__device__ __forceinline__ void convert_x16(const uint4 c, float dx, uint4 (&hi)[2], uint4 (&lo)[2]) {
    const uint32_t w[4] = {c.x ^ 0x80808080u, c.y ^ 0x80808080u, c.z ^ 0x80808080u, c.w ^ 0x80808080u};
    const uint64_t bias = f32x2_pack(8388736.0f, 8388736.0f), dx2 = f32x2_pack(dx, dx);  // 2^23 + 128
    uint64_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = f32x2_mul(f32x2_sub(byte_pair_biased(w[i >> 1], 2 * (i & 1)), bias), dx2);
    split16(v, hi, lo);
}

// The weights: elements 8 qq .. 8 qq + 7 of K slice c (32 wide) of the group
// whose bytes start at `blk` (2-byte aligned), as one 16-byte chunk of hi and
// one of lo.
template <int FMT>
__device__ __forceinline__ void convert_w8(const uint8_t* blk, int c, int qq, uint4& hi, uint4& lo);

// Q4_K (super-block: d, dmin, 12 bytes of 6-bit scales / mins, 128 bytes of
// nibbles).  Slice c is sub-block c: the low (c even) or high (c odd) nibbles
// of quant chunk c / 2.  w = d * sc * q - dmin * m.
template <>
__device__ __forceinline__ void convert_w8<QX_Q4_K>(const uint8_t* blk, int c, int qq, uint4& hi, uint4& lo) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
    const uint2 qv = *reinterpret_cast<const uint2*>(blk + 16 + 32 * (c >> 1) + 8 * qq);
    const float d = __half2float(__ushort_as_half(uint16_t(hdr.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half(uint16_t(hdr.x >> 16)));
    int sc, m;
    if (c < 4) {
        sc = (hdr.y >> (8 * c)) & 63;
        m = (hdr.z >> (8 * c)) & 63;
    } else {
        const int u = c - 4;
        sc = ((hdr.w >> (8 * u)) & 15) | (((hdr.y >> (8 * u + 6)) & 3) << 4);
        m = ((hdr.w >> (8 * u + 4)) & 15) | (((hdr.z >> (8 * u + 6)) & 3) << 4);
    }
    const float a = d * float(sc), cm = dmin * float(m);  // exact products
    const uint32_t sh = 4u * uint32_t(c & 1);
    const uint32_t nb[2] = {(qv.x >> sh) & 0x0F0F0F0Fu, (qv.y >> sh) & 0x0F0F0F0Fu};
    const uint64_t bias = f32x2_pack(8388608.0f, 8388608.0f), a2 = f32x2_pack(a, a), ncm = f32x2_pack(-cm, -cm);
    uint64_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)  // d * sc * q - dmin * m with one rounding (a fused multiply-add)
        v[i] = f32x2_fma(a2, f32x2_sub(byte_pair_biased(nb[i >> 1], 2 * (i & 1)), bias), ncm);
    split8(v, hi, lo);
}

// Q6_K (ql[128], qh[64], scales[16] int8, d f16; element e = 128 h + 32 t + l
// has its low four bits in ql[64 h + 32 (t & 1) + l] -- the low nibble for
// t < 2 -- and its high two bits at bits 2t of qh[32 h + l]).  Slice c is
// h = c / 4, t = c % 4; the thread's l = 8 qq .. 8 qq + 7 share scale
// 2c + qq / 2.  w = d * sc * (q - 32).
template <>
__device__ __forceinline__ void convert_w8<QX_Q6_K>(const uint8_t* blk, int c, int qq, uint4& hi, uint4& lo) {
    const int h = c >> 2, t = c & 3, l0 = 8 * qq;
    uint32_t ql[2], qh[2];
    words_a2<2>(blk + 64 * h + 32 * (t & 1) + l0, ql);
    words_a2<2>(blk + 128 + 32 * h + l0, qh);
    const float a = f16_at_a2(blk + 208) * float(reinterpret_cast<const int8_t*>(blk)[192 + 2 * c + (qq >> 1)]);
    const uint32_t nsh = (t >= 2) ? 4u : 0u, hsh = 2u * uint32_t(t);
    const uint64_t bias = f32x2_pack(8388640.0f, 8388640.0f), a2 = f32x2_pack(a, a);  // 2^23 + 32
    uint64_t v[4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const uint32_t q = ((ql[j] >> nsh) & 0x0F0F0F0Fu) | (((qh[j] >> hsh) & 0x03030303u) << 4);
        v[2 * j] = f32x2_mul(a2, f32x2_sub(byte_pair_biased(q, 0), bias));
        v[2 * j + 1] = f32x2_mul(a2, f32x2_sub(byte_pair_biased(q, 2), bias));
    }
    split8(v, hi, lo);
}

// Q8_0 (blocks of d f16 and 32 int8), four blocks per group: slice c is
// block c.  w = d * q.
template <>
__device__ __forceinline__ void convert_w8<QX_Q8_0>(const uint8_t* blk, int c, int qq, uint4& hi, uint4& lo) {
    const uint8_t* b = blk + 34 * c;
    uint32_t qw[2];
    words_a2<2>(b + 2 + 8 * qq, qw);
    const float d = f16_at_a2(b);
    const uint64_t bias = f32x2_pack(8388736.0f, 8388736.0f), d2 = f32x2_pack(d, d);  // 2^23 + 128
    uint64_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v[i] = f32x2_mul(d2, f32x2_sub(byte_pair_biased(qw[i >> 1] ^ 0x80808080u, 2 * (i & 1)), bias));
    split8(v, hi, lo);
}

// ---------------------------------------------------------------------------
// the GEMM
// ---------------------------------------------------------------------------

// Tiles are numbered M tile fastest, so the CTAs that share a weight tile run
// together and read it from DRAM once.  A launch takes tiles tile_base ..:
// one CTA per tile, or (split) a cluster of two or four CTAs per tile, each
// taking an equal share of the K groups, whose f32 partial sums meet in the
// first CTA through distributed shared memory: Y = a0 + a1 for two, and
// (a0 + a1) + (a2 + a3) for four, in that order.  The host splits the tiles
// of a last, at most half-full wave in two, so that it takes half as long;
// every tile in two when all of them fill at most half a wave, and in four
// when they fill at most a quarter (and K has four groups or more).
//   warp 0: TMA producer (the whole warp: per-row boxes take four rows a lane);
//   warp 1: tensor memory (two 128-column accumulators) and the MMA issuer;
//   warps 2-17: converters -- per K slice, thread ct converts X row ct / 2
//           (16 codes, half ct % 2; zeros past M, nothing stored for an
//           unused half) and weight row ct / 4 (8 values, quarter
//           ct % 4); warps 2-9 then drain the accumulators (warp w: rows
//           128 ((w - 2) / 4) + 32 (w % 4) .. + 31 of the tile).
template <int FMT>
__global__ void __launch_bounds__(kTcThreads, 1) tc_prefill_kernel(const __grid_constant__ TcParams p) {
    using G = RawGeom<FMT>;
    constexpr int SPG = G::kGroupK / TBK;        // K slices per raw group
    constexpr int RAW_BYTES = raw_slot_bytes<FMT>();
    constexpr int RAW_TX = G::kBox * TBN;        // bytes the copies of one group bring
    constexpr int RS = G::kSlots;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t rawaddr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (rawaddr & 1023)) & 1023);
    uint8_t* ops = smem;                               // [OP_STAGES][Xh0, Xh1, Xl0, Xl1, Wh, Wl]
    uint8_t* wr = ops + OP_STAGES * OP_BYTES;          // [RS][128 rows of raw blocks]
    uint64_t* full_op = reinterpret_cast<uint64_t*>(wr + RS * RAW_BYTES);
    uint64_t* empty_op = full_op + OP_STAGES;
    uint64_t* full_wr = empty_op + OP_STAGES;
    uint64_t* empty_wr = full_wr + RS;
    uint64_t* acc_full = empty_wr + RS;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = p.tile_base + (p.split ? int(blockIdx.x / unsigned(p.split)) : int(blockIdx.x));
    const int m0 = (tile % p.tiles_m) * TBM, n0 = (tile / p.tiles_m) * TBN;
    const int halves = (m0 + 128 < p.M) ? 2 : 1;  // 128-row halves of the tile with rows of X
    const int n_k = p.K / TBK, n_groups = (p.K + G::kGroupK - 1) / G::kGroupK;
    // this CTA's K groups [g0, g1) and slices [t0, t1); ring positions count from g0 and t0
    const uint32_t rank = p.split ? cluster_rank() : 0u;
    const int ks = p.split ? p.split : 1;  // CTAs sharing the tile's K groups
    const int g0 = int(int64_t(n_groups) * int(rank) / ks), g1 = int(int64_t(n_groups) * (int(rank) + 1) / ks);
    const int t0 = g0 * SPG, t1 = g1 * SPG < n_k ? g1 * SPG : n_k;
    const bool w2d = FMT == QX_Q4_K || p.w2d != 0;
    const int wstride = w2d ? G::kBox : kRowStride1d;
    if (!p.split) pdl_launch_dependents();  // a split launch of the last tiles may start beside this one

    if (threadIdx.x == 0) {
        for (int s = 0; s < OP_STAGES; ++s) {
            mbar_init(&full_op[s], kConvWarps);
            mbar_init(&empty_op[s], 1);
        }
        for (int r = 0; r < RS; ++r) {
            mbar_init(&full_wr[r], 1);
            mbar_init(&empty_wr[r], kConvWarps);
        }
        mbar_init(acc_full, 1);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                     "r"(2 * TBN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;  // converter warps: every wait of the main loop succeeded

    if (warp == 0) {
        // ---- producer: raw weight groups, up to RS ahead of the group being converted
        int wr_issued = 0;  // ring positions issued
        for (int g = g0; g < g1; ++g) {
            const int lg = g - g0, r = lg % RS;
            if (lg >= RS && !warp_wait(&empty_wr[r], ((lg / RS) - 1) & 1, p.wait_ns, p.err, kErrTimeoutEmpty)) break;
            uint8_t* dst = wr + r * RAW_BYTES;
            if (lane == 0) mbar_arrive_expect_tx(&full_wr[r], RAW_TX);
            __syncwarp();
            if (w2d) {
                // the same offset in every row: one box, from the 16-byte boundary at or below the group
                if (lane == 0)
                    tma_load_2d(dst, &p.w_map, (g * G::kGroupBytes) & ~15, n0, &full_wr[r]);
            } else {
#pragma unroll
                for (int i = 0; i < TBN / 32; ++i) {
                    const int row = lane + 32 * i;
                    const int64_t a = int64_t(n0 + row) * p.row_bytes + int64_t(g) * G::kGroupBytes;
                    tma_load_1d(dst + row * kRowStride1d, &p.w_map, static_cast<int>(a & ~int64_t(15)), &full_wr[r]);
                }
            }
            wr_issued = lg + 1;
        }
        // keep the CTA alive until every copy it issued has landed
        if (lane == 0)
            for (int g = wr_issued > RS ? wr_issued - RS : 0; g < wr_issued; ++g)
                mbar_wait_bounded(&full_wr[g % RS], (g / RS) & 1, p.wait_ns, p.err, kErrTimeoutDrain);
    } else if (warp == 1) {
        if (lane == 0) {
            // ---- MMA issuer: per half, Xh Wh + Xh Wl + Xl Wh per K slice of 32
            for (int lt = 0; lt < t1 - t0; ++lt) {
                const int s = lt % OP_STAGES;
                if (!mbar_wait_bounded(&full_op[s], (lt / OP_STAGES) & 1, p.wait_ns, p.err, kErrTimeoutMma)) break;
                tc_fence_after();
                const uint32_t base = smem_addr(ops + s * OP_BYTES);
                const uint64_t wh = sw64_desc(base + OP_WH), wl = sw64_desc(base + OP_WL);
                for (int a = 0; a < halves; ++a) {
                    const uint64_t xh = sw64_desc(base + OP_XH + a * T_TILE), xl = sw64_desc(base + OP_XL + a * T_TILE);
                    const uint32_t acc = tmem + uint32_t(a * TBN);
#pragma unroll
                    for (int k = 0; k < TBK / 16; ++k) {  // K = 16 per MMA: 32 bytes further along the swizzled row
                        const uint64_t o = uint64_t(2 * k);
                        tc_mma(acc, xh + o, wh + o, kIdesc, (lt | k) != 0 ? 1u : 0u);
                        tc_mma(acc, xh + o, wl + o, kIdesc, 1u);
                        tc_mma(acc, xl + o, wh + o, kIdesc, 1u);
                    }
                }
                tc_commit(&empty_op[s]);  // arrives once these MMAs have read the stage
            }
            tc_commit(acc_full);  // also after a failed wait: arrives once the issued MMAs are done
        }
    } else {
        // ---- converters
        const int ct = threadIdx.x - 64;
        const int xrow = ct >> 1, xh = ct & 1;  // X: row of the tile, half of the slice
        const int wrow = ct >> 2, wq = ct & 3;  // W: row of the tile, quarter of the slice
        const int xm = m0 + xrow;
        const bool xlive = xm < p.M;             // rows of X past M are zeros
        const bool xstore = (xrow >> 7) < halves;  // (warp-uniform) rows of an unused half are never read
        // The thread's 16 codes of slice t are word 2 t + xh of its row (K is a multiple of 32 and the
        // codes are 16-byte aligned); codes and scales of kXAhead slices are in flight at a time.
        const uint4* xq_row = reinterpret_cast<const uint4*>(p.xq + int64_t(xlive ? xm : 0) * p.K) + xh;
        const float* xd_row = p.xd + int64_t(xlive ? xm : 0) * (p.K / 32);
        uint4 qa[kXAhead];
        float da[kXAhead];
#pragma unroll
        for (int i = 0; i < kXAhead; ++i) {
            const bool live = xlive && t0 + i < t1;
            qa[i] = live ? __ldg(xq_row + 2 * (t0 + i)) : make_uint4(0u, 0u, 0u, 0u);
            da[i] = live ? __ldg(xd_row + t0 + i) : 0.0f;
        }
        const uint32_t xa = uint32_t(OP_XH + (xrow >> 7) * T_TILE), xla = uint32_t(OP_XL + (xrow >> 7) * T_TILE);
        const int xr7 = xrow & 127;
        // Ring positions, advanced slice by slice (no divisions): operand stage s and the parity of
        // its release phase to wait for, K slice c of group g, raw slot r and its fill parity.
        int s = 0, lap = 0, c = 0, g = g0, r = 0, wph = 0;
        const int64_t wrow_byte0 = int64_t(n0 + wrow) * p.row_bytes;  // this thread's weight row in the matrix
        const uint8_t* blk = nullptr;  // the thread's row of the current raw group in its slot
        // slice t (ring position lt = t - t0), its codes and scale in slot j = lt % kXAhead (the loop
        // is unrolled by kXAhead so that j is static), which then takes slice t + kXAhead
        const auto convert_slice = [&](int t, uint4& qx, float& dx) -> bool {
            if (c == 0) {
                if (!warp_wait(&full_wr[r], wph, p.wait_ns, p.err, kErrTimeoutFull)) return false;
                const int64_t a = wrow_byte0 + int64_t(g) * G::kGroupBytes;
                blk = wr + r * RAW_BYTES + wrow * wstride + (a & 15);  // the group in its box
            }
            if (t - t0 >= OP_STAGES && !warp_wait(&empty_op[s], lap ^ 1, p.wait_ns, p.err, kErrTimeoutEmpty))
                return false;
            uint4 xhi[2], xlo[2], whi, wlo;
            if (xlive) {
                convert_x16(qx, dx, xhi, xlo);
            } else {
                xhi[0] = xhi[1] = xlo[0] = xlo[1] = make_uint4(0u, 0u, 0u, 0u);
            }
            if (xlive && t + kXAhead < t1) {
                qx = __ldg(xq_row + 2 * (t + kXAhead));
                dx = __ldg(xd_row + t + kXAhead);
            }
            convert_w8<FMT>(blk, c, wq, whi, wlo);
            uint8_t* st = ops + s * OP_BYTES;
            if (xstore) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t off = sw64_off(xr7, 2 * xh + i);
                    *reinterpret_cast<uint4*>(st + xa + off) = xhi[i];
                    *reinterpret_cast<uint4*>(st + xla + off) = xlo[i];
                }
            }
            const uint32_t woff = sw64_off(wrow, wq);
            *reinterpret_cast<uint4*>(st + OP_WH + woff) = whi;
            *reinterpret_cast<uint4*>(st + OP_WL + woff) = wlo;
            fence_proxy_async_smem();  // generic-proxy stores, read by the tensor cores
            __syncwarp();
            const bool group_done = c == SPG - 1 || t == t1 - 1;
            if (lane == 0) {
                mbar_arrive(&full_op[s]);
                if (group_done) mbar_arrive(&empty_wr[r]);
            }
            if (++s == OP_STAGES) {
                s = 0;
                lap ^= 1;
            }
            if (group_done) {
                c = 0;
                ++g;
                if (++r == RS) {
                    r = 0;
                    wph ^= 1;
                }
            } else {
                ++c;
            }
            return true;
        };
        for (int tb = t0; tb < t1 && ok; tb += kXAhead) {
#pragma unroll
            for (int j = 0; j < kXAhead; ++j) {
                if (ok && tb + j < t1) ok = convert_slice(tb + j, qa[j], da[j]);
            }
        }
    }
    // ---- epilogue: warps 2-9; warp w drains rows 32 (w % 4) .. + 31 of accumulator (w - 2) / 4
    const int half = (warp - 2) >> 2, q = warp & 3;
    const bool drains = warp >= 2 && warp < 10 && half < halves;
    const bool acc_ok = warp >= 2 && warp < 10 && warp_wait(acc_full, 0, p.wait_ns, p.err, kErrTimeoutMma) && ok;
    if (acc_ok) tc_fence_after();
    // Split tiles: the partial sums of the second CTA go into the first CTA's operand stages (free
    // once its MMAs are done), row r of accumulator h at byte 65536 h + 512 r, 16-byte chunk j at
    // position j ^ (r % 32) (so that the 32 rows a warp touches fall on different banks).
    const uint32_t xbuf = smem_addr(ops);
    const int row = 32 * q + lane;  // of the warp's accumulator
    const auto xchunk = [&](int j) -> uint32_t {
        return uint32_t(half * 65536 + row * 512 + ((j ^ lane) << 4));
    };
    // Two CTAs: the second hands its sums to the first, which adds them to its own.  Four: the odd
    // ranks hand theirs to the rank below; rank 2 adds them to its own and hands the result to
    // rank 1's (idle) buffer, while rank 0 adds rank 1's into its own buffer; rank 0 stores
    // (a0 + a1) + (a2 + a3).
    if (p.split) {
        cluster_sync_all();  // every CTA's MMAs are done: their stages are free
        if ((rank & 1u) && drains && acc_ok) {
            const uint32_t dst = peer_addr(xbuf, rank - 1u);
#pragma unroll 1
            for (int cc = 0; cc < TBN / 32; ++cc) {
                uint32_t v[32];
                tc_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(half * TBN + 32 * cc), v);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    st_peer_v4(dst + xchunk(8 * cc + i), v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            }
        }
        cluster_sync_all();  // the odd ranks' sums have landed
        if (p.split == 4) {
            if ((rank == 0u || rank == 2u) && drains && acc_ok) {
#pragma unroll 1
                for (int cc = 0; cc < TBN / 32; ++cc) {
                    uint32_t v[32];
                    tc_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(half * TBN + 32 * cc), v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float4 o = *reinterpret_cast<const float4*>(ops + xchunk(8 * cc + i));
                        o.x = __uint_as_float(v[4 * i]) + o.x;
                        o.y = __uint_as_float(v[4 * i + 1]) + o.y;
                        o.z = __uint_as_float(v[4 * i + 2]) + o.z;
                        o.w = __uint_as_float(v[4 * i + 3]) + o.w;
                        if (rank == 2u)
                            st_peer_v4(peer_addr(xbuf, 1u) + xchunk(8 * cc + i), __float_as_uint(o.x),
                                       __float_as_uint(o.y), __float_as_uint(o.z), __float_as_uint(o.w));
                        else
                            *reinterpret_cast<float4*>(ops + xchunk(8 * cc + i)) = o;
                    }
                }
            }
            cluster_sync_all();  // rank 0 holds a0 + a1, rank 1 holds a2 + a3
        }
    }
    if (rank == 0 && drains && acc_ok) {
        const int yr = m0 + 128 * half + row;
        const bool row_ok = yr < p.M;
        // vector stores only where every row of the tile starts 16-byte aligned (Y is only
        // required to be 4-byte aligned)
        const bool vec = (n0 + TBN <= p.N) && (p.N % 4 == 0) && (reinterpret_cast<uintptr_t>(p.Y) & 15) == 0;
        float* yrow = p.Y + size_t(row_ok ? yr : 0) * p.N + n0;
        const uint32_t src1 = p.split == 4 ? peer_addr(xbuf, 1u) : 0u;
#pragma unroll 1
        for (int cc = 0; cc < TBN / 32; ++cc) {
            uint32_t v[32];
            if (p.split == 4) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 o = *reinterpret_cast<const float4*>(ops + xchunk(8 * cc + i));
                    const uint4 r = ld_peer_v4(src1 + xchunk(8 * cc + i));
                    v[4 * i] = __float_as_uint(o.x + __uint_as_float(r.x));
                    v[4 * i + 1] = __float_as_uint(o.y + __uint_as_float(r.y));
                    v[4 * i + 2] = __float_as_uint(o.z + __uint_as_float(r.z));
                    v[4 * i + 3] = __float_as_uint(o.w + __uint_as_float(r.w));
                }
            } else {
                tc_ld32(tmem + (uint32_t(32 * q) << 16) + uint32_t(half * TBN + 32 * cc), v);
                if (p.split) {
                    const auto add = [](uint32_t& a, float b) { a = __float_as_uint(__uint_as_float(a) + b); };
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 o = *reinterpret_cast<const float4*>(ops + xchunk(8 * cc + i));
                        add(v[4 * i], o.x);
                        add(v[4 * i + 1], o.y);
                        add(v[4 * i + 2], o.z);
                        add(v[4 * i + 3], o.w);
                    }
                }
            }
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
    if (p.split == 4) cluster_sync_all();  // rank 1's buffer stays until rank 0 has read it
    // A split launch beside the launch of the other tiles (programmatic
    // dependent launch) completes only after that one has; launched alone,
    // this wait returns at once.
    if (p.split) pdl_wait_prior_grid();
    tc_fence_before();
    __syncthreads();
    __syncwarp();
    if (warp == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(2 * TBN) : "memory");
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

// A byte matrix [rows, row_bytes] (row_bytes a 16-byte multiple), boxes of
// box_x bytes x box_rows rows, no swizzle.
bool encode_bytes_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t row_bytes, int box_x, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cuuint64_t(row_bytes), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
    cuuint32_t box[2] = {cuuint32_t(box_x), cuuint32_t(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// `bytes` bytes as a one-dimensional tensor, boxes of box_x bytes.
bool encode_bytes_1d(CUtensorMap* m, const void* ptr, int64_t bytes, int box_x) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[1] = {cuuint64_t(bytes)};
    cuuint64_t strides[1] = {0};  // no outer dimension, but the encoder wants the array
    cuuint32_t box[1] = {cuuint32_t(box_x)};
    cuuint32_t es[1] = {1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT>
cudaError_t launch_fmt(TcParams& p, const uint8_t* W, int64_t N, const int8_t* xq, int64_t M, int64_t K,
                       int sm_count, cudaStream_t s) {
    using G = RawGeom<FMT>;
    if ((reinterpret_cast<uintptr_t>(xq) & 15) != 0 || K % TBK != 0) return cudaErrorInvalidValue;
    p.xq = xq;
    p.w2d = (FMT == QX_Q4_K || p.row_bytes % 16 == 0) ? 1 : 0;
    const bool wok = p.w2d ? encode_bytes_2d(&p.w_map, W, N, p.row_bytes, G::kBox, TBN)
                           : encode_bytes_1d(&p.w_map, W, N * p.row_bytes, G::kBox);
    if (!wok) return cudaErrorInvalidValue;
    static int per_sm[64] = {0};  // resident CTAs per SM, per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (per_sm[dev] == 0) {
        e = cudaFuncSetAttribute(tc_prefill_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(tc_smem_bytes<FMT>()));
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tc_prefill_kernel<FMT>, kTcThreads, tc_smem_bytes<FMT>());
        if (e != cudaSuccess) return e;
        per_sm[dev] = n > 0 ? n : 1;
    }
    // Waves of tiles: when the last wave is at most half full (and there is
    // more than one), its tiles are split in two along K and run as clusters
    // of two CTAs beside the others' last wave, so that it takes half as long.
    // When all the tiles fill at most half a wave, every tile is split (one
    // launch of clusters, after the preceding work like any launch), in four
    // when they fill at most a quarter of one and there are four K groups.
    const int64_t tiles_m = (M + TBM - 1) / TBM, tiles_n = (N + TBN - 1) / TBN, tiles = tiles_m * tiles_n;
    const int64_t slots = int64_t(sm_count > 0 ? sm_count : 1) * per_sm[dev];
    const int n_groups = int((K + G::kGroupK - 1) / G::kGroupK);
    int64_t tail = 0;
    int ks = 2;
    if (n_groups >= 2) {
        if (tiles > slots && 2 * (tiles % slots) <= slots) {
            tail = tiles % slots;
        } else if (n_groups >= 4 && 4 * tiles <= slots) {
            tail = tiles;
            ks = 4;
        } else if (2 * tiles <= slots) {
            tail = tiles;
        }
    }
    p.tiles_m = int(tiles_m);
    if (tiles - tail > 0) {
        p.tile_base = 0;
        p.split = 0;
        tc_prefill_kernel<FMT><<<unsigned(tiles - tail), kTcThreads, tc_smem_bytes<FMT>(), s>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (tail > 0) {
        p.tile_base = int(tiles - tail);
        p.split = ks;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(ks * tail));
        cfg.blockDim = dim3(kTcThreads);
        cfg.dynamicSmemBytes = tc_smem_bytes<FMT>();
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = unsigned(ks);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        // beside the first launch (which lets it start at its own start, so
        // after the preceding work); alone, an ordinary stream-ordered launch
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = tiles > tail ? 2 : 1;
        if ((e = cudaLaunchKernelEx(&cfg, tc_prefill_kernel<FMT>, p)) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

bool prefill_tc_serves(int fmt, int64_t N, int64_t K, int64_t M, int64_t row_bytes) {
    if (fmt != QX_Q4_K && fmt != QX_Q6_K && fmt != QX_Q8_0) return false;
    // copy coordinates are 32-bit: the last box of the last tile must start below 2^31
    const int64_t limit = (int64_t(1) << 31) - 4096;
    const int64_t tiles_n = (N + TBN - 1) / TBN;
    const int64_t tiles = tiles_n * ((M + TBM - 1) / TBM);
    return M <= INT32_MAX && N <= INT32_MAX && K <= INT32_MAX && 4 * tiles <= INT32_MAX &&
           tiles_n * TBN * row_bytes < limit;
}

cudaError_t launch_prefill_tc(int fmt, const uint8_t* W, int64_t N, int64_t K, int64_t row_bytes, const int8_t* xq,
                              const float* xd, int64_t M, float* Y, unsigned* err, int sm_count, cudaStream_t s) {
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.xd = xd;
    p.M = int(M);
    p.N = int(N);
    p.K = int(K);
    p.row_bytes = row_bytes;
    p.Y = Y;
    p.err = err;
    p.wait_ns = 2000000000ull;
    switch (fmt) {
        case QX_Q4_K: return launch_fmt<QX_Q4_K>(p, W, N, xq, M, K, sm_count, s);
        case QX_Q6_K: return launch_fmt<QX_Q6_K>(p, W, N, xq, M, K, sm_count, s);
        case QX_Q8_0: return launch_fmt<QX_Q8_0>(p, W, N, xq, M, K, sm_count, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qx
