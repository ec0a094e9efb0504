/*
 * qx_oracle.c -- plain, slow CPU oracle for the block-quantised GEMV.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library; it is written from the
 * definitions below so that a reader can check it against them by eye.
 *
 * What it computes (two methods, each with its own reference -- llamay
 * "Backends and hardware", "Accelerate is not bit-identical": dequantising the
 * weights to float and quantising the activation to int8 are two methods, not
 * one method plus a rounding error):
 *
 *   f32 mode : every weight is dequantised exactly (in double) and the row dot
 *              product  y[r] = sum_i w[r,i] * x[i]  is summed in double.
 *   W4A8 mode: the activation is quantised to int8 once per matmul, per block
 *              of 32 with an f32 absmax scale (llamay "Backends and hardware",
 *              "CPU": the W4A8 fused dot product); per weight sub-block the
 *              integer products are summed exactly (int64, checked to fit
 *              int32), then scaled per block and summed in double.
 *
 * Block layouts (the GGUF block convention; the pages name the formats --
 * llambda.lisp README, "Features & Architecture" and opening paragraph: Q4_K_M
 * and Q6_K tensors whose 4-bit/6-bit nibbles are unpacked -- but print no byte
 * layout, so the on-disk GGUF convention is the reading taken):
 *
 *   Q4_K (256 weights, 144 B): d f16 @0, dmin f16 @2, scales[12] @4, qs[128] @16.
 *        Sub-block j (32 weights) has a 6-bit scale sc_j and 6-bit min m_j:
 *          j < 4 : sc_j = s[j] & 63,  m_j = s[j+4] & 63
 *          j >= 4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4)
 *                  m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4)
 *        Element e: byte qs[32*(e/64) + e%32], low nibble if (e%64) < 32 else
 *        high nibble.  w = d*sc_j*q - dmin*m_j.
 *   Q6_K (256 weights, 210 B): ql[128] @0, qh[64] @128, scales[16] int8 @192,
 *        d f16 @208.  Element e = 128h + 32t + l (h in 0..1, t in 0..3,
 *        l in 0..31): low 4 bits from ql[64h + 32*(t&1) + l] (low nibble if
 *        t < 2 else high nibble), high 2 bits are bits 2t..2t+1 of qh[32h + l].
 *        w = d * scales[e/16] * (q - 32).
 *   Q8_0 (32 weights, 34 B): d f16 @0, qs[32] int8 @2.  w = d*q.
 *
 * Activation quantisation (per block of 32, decisions in f32, the precision of
 * the kernel; the pages fix none):
 *   amax = max |x_i|;  d = amax / 127 (correctly rounded f32);
 *   q_i = round-half-to-even(x_i / d) (correctly rounded f32 quotient),
 *         clamped to [-127, 127];  q_i = 0 when d == 0;
 *   sum = sum_i q_i.
 *
 * Rows are independent (llambda.lisp README, "Features & Architecture": the
 * GEMV's outer loop runs in parallel with isolated, lock-free writes), so the
 * only parallelism here is an OpenMP loop over rows; nothing inside a row is
 * blocked, fused or reordered.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_Q8_0 8
#define ORC_Q4_K 12
#define ORC_Q6_K 14

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_NONFINITE (-2)
#define ORC_ERR_OVERFLOW (-3)

/* IEEE 754 binary16 -> double, from the format's definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is subnormal
 * (f * 2^-24), exponent 31 is infinity / NaN. */
double orc_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

static double f16_at(const uint8_t* p) {
    return orc_f16_to_f64((uint16_t)(p[0] | (p[1] << 8)));
}

int orc_block_weights(int fmt) {
    if (fmt == ORC_Q8_0) return 32;
    if (fmt == ORC_Q4_K || fmt == ORC_Q6_K) return 256;
    return 0;
}

int orc_block_bytes(int fmt) {
    if (fmt == ORC_Q8_0) return 34;
    if (fmt == ORC_Q4_K) return 144;
    if (fmt == ORC_Q6_K) return 210;
    return 0;
}

/* Number of integer partial sums per row: one per 32-weight sub-block for
 * Q4_K and Q8_0, one per 16-weight scale group for Q6_K. */
int orc_partial_group(int fmt) {
    if (fmt == ORC_Q6_K) return 16;
    if (fmt == ORC_Q4_K || fmt == ORC_Q8_0) return 32;
    return 0;
}

int64_t orc_row_bytes(int fmt, int64_t cols) {
    int bw = orc_block_weights(fmt);
    if (bw == 0 || cols <= 0 || cols % bw) return -1;
    return cols / bw * orc_block_bytes(fmt);
}

/* ---- per-format element decode (integer quant and its scale terms) ---- */

static void q4k_scale_min(const uint8_t* s, int j, int* sc, int* m) {
    if (j < 4) {
        *sc = s[j] & 63;
        *m = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

static int q4k_quant(const uint8_t* blk, int e) {
    uint8_t b = blk[16 + 32 * (e / 64) + e % 32];
    return (e % 64) < 32 ? (b & 15) : (b >> 4);
}

static int q6k_quant(const uint8_t* blk, int e) {
    int h = e / 128, t = (e % 128) / 32, l = e % 32;
    uint8_t lo = blk[64 * h + 32 * (t & 1) + l];
    int low4 = t < 2 ? (lo & 15) : (lo >> 4);
    int high2 = (blk[128 + 32 * h + l] >> (2 * t)) & 3;
    return low4 | (high2 << 4);
}

static int q6k_scale(const uint8_t* blk, int e) {
    return (int)(int8_t)blk[192 + e / 16];
}

static int q8_0_quant(const uint8_t* blk, int e) {
    return (int)(int8_t)blk[2 + e];
}

/* Dequantise one row of `cols` weights into w (double), by the closed forms
 * w = d*sc*q - dmin*m (Q4_K), w = d*sc*(q-32) (Q6_K), w = d*q (Q8_0). */
int orc_dequant_row(int fmt, const uint8_t* row, int64_t cols, double* w) {
    int bw = orc_block_weights(fmt), bb = orc_block_bytes(fmt);
    if (!row || !w || bw == 0 || cols <= 0 || cols % bw) return ORC_ERR_ARG;
    for (int64_t b = 0; b < cols / bw; b++) {
        const uint8_t* blk = row + b * bb;
        double* wb = w + b * bw;
        if (fmt == ORC_Q4_K) {
            double d = f16_at(blk), dmin = f16_at(blk + 2);
            for (int e = 0; e < 256; e++) {
                int sc, m;
                q4k_scale_min(blk + 4, e / 32, &sc, &m);
                wb[e] = d * sc * q4k_quant(blk, e) - dmin * m;
            }
        } else if (fmt == ORC_Q6_K) {
            double d = f16_at(blk + 208);
            for (int e = 0; e < 256; e++)
                wb[e] = d * q6k_scale(blk, e) * (q6k_quant(blk, e) - 32);
        } else {
            double d = f16_at(blk);
            for (int e = 0; e < 32; e++) wb[e] = d * q8_0_quant(blk, e);
        }
    }
    return ORC_OK;
}

/* ---- activation quantisation ---- */

int orc_quantize_act_q8(const float* x, int64_t m, int64_t cols, int8_t* q,
                        float* d, int32_t* sum) {
    if (!x || !q || !d || !sum || m <= 0 || cols <= 0 || cols % 32)
        return ORC_ERR_ARG;
    for (int64_t i = 0; i < m * cols; i++)
        if (!isfinite(x[i])) return ORC_ERR_NONFINITE;
    for (int64_t blk = 0; blk < m * cols / 32; blk++) {
        const float* xb = x + blk * 32;
        float amax = 0.0f;
        for (int i = 0; i < 32; i++)
            if (fabsf(xb[i]) > amax) amax = fabsf(xb[i]);
        float db = amax / 127.0f;
        int32_t s = 0;
        for (int i = 0; i < 32; i++) {
            int v = 0;
            if (db != 0.0f) {
                float r = nearbyintf(xb[i] / db);
                v = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);
            }
            q[blk * 32 + i] = (int8_t)v;
            s += v;
        }
        d[blk] = db;
        sum[blk] = s;
    }
    return ORC_OK;
}

/* ---- f32 mode: y[r] = sum_i w[r,i] * x[i], all in double ---- */

int orc_gemv_f64x(int fmt, const uint8_t* W, int64_t rows, int64_t cols,
                  const double* x, double* y, double* absdot, int nthreads) {
    int64_t rb = orc_row_bytes(fmt, cols);
    if (!W || !x || !y || rows <= 0 || rb < 0) return ORC_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    int err = ORC_OK;
#pragma omp parallel num_threads(nthreads)
    {
        double* w = (double*)malloc(sizeof(double) * (size_t)cols);
        if (!w) {
#pragma omp atomic write
            err = ORC_ERR_ARG;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; r++) {
            if (!w) continue;
            orc_dequant_row(fmt, W + r * rb, cols, w);
            double acc = 0.0, aacc = 0.0;
            for (int64_t i = 0; i < cols; i++) {
                acc += w[i] * x[i];
                aacc += fabs(w[i] * x[i]);
            }
            y[r] = acc;
            if (absdot) absdot[r] = aacc;
        }
        free(w);
    }
    return err;
}

int orc_gemv_f32(int fmt, const uint8_t* W, int64_t rows, int64_t cols,
                 const float* x, double* y, double* absdot, int nthreads) {
    if (!x || cols <= 0) return ORC_ERR_ARG;
    double* xd = (double*)malloc(sizeof(double) * (size_t)cols);
    if (!xd) return ORC_ERR_ARG;
    for (int64_t i = 0; i < cols; i++) xd[i] = (double)x[i];
    int rc = orc_gemv_f64x(fmt, W, rows, cols, xd, y, absdot, nthreads);
    free(xd);
    return rc;
}

/* ---- W4A8 mode ---- */

/* Integer partial sums of one row: P[g] = sum over group g of q_w * q_x, with
 * q_w the unsigned 4-bit quant for Q4_K, (q - 32) for Q6_K and the int8 quant
 * for Q8_0.  Summed in int64; ORC_ERR_OVERFLOW if a sum leaves int32. */
static int row_partials(int fmt, const uint8_t* row, int64_t cols,
                        const int8_t* qx, int64_t* P) {
    int bw = orc_block_weights(fmt), bb = orc_block_bytes(fmt);
    int gs = orc_partial_group(fmt);
    int64_t ng = cols / gs;
    for (int64_t g = 0; g < ng; g++) {
        int64_t col0 = g * gs;
        const uint8_t* blk = row + (col0 / bw) * bb;
        int e0 = (int)(col0 % bw);
        int64_t acc = 0;
        for (int i = 0; i < gs; i++) {
            int qw;
            if (fmt == ORC_Q4_K)
                qw = q4k_quant(blk, e0 + i);
            else if (fmt == ORC_Q6_K)
                qw = q6k_quant(blk, e0 + i) - 32;
            else
                qw = q8_0_quant(blk, e0 + i);
            acc += (int64_t)qw * qx[col0 + i];
        }
        if (acc > INT32_MAX || acc < INT32_MIN) return ORC_ERR_OVERFLOW;
        P[g] = acc;
    }
    return ORC_OK;
}

int orc_partials(int fmt, const uint8_t* W, int64_t rows, int64_t cols,
                 const int8_t* qx, int32_t* P) {
    int64_t rb = orc_row_bytes(fmt, cols);
    if (!W || !qx || !P || rows <= 0 || rb < 0) return ORC_ERR_ARG;
    int gs = orc_partial_group(fmt);
    int64_t ng = cols / gs;
    int64_t* tmp = (int64_t*)malloc(sizeof(int64_t) * (size_t)ng);
    if (!tmp) return ORC_ERR_ARG;
    int rc = ORC_OK;
    for (int64_t r = 0; r < rows && rc == ORC_OK; r++) {
        rc = row_partials(fmt, W + r * rb, cols, qx, tmp);
        for (int64_t g = 0; g < ng && rc == ORC_OK; g++)
            P[r * ng + g] = (int32_t)tmp[g];
    }
    free(tmp);
    return rc;
}

/* y[r] = sum over blocks of (block scale) * (integer partial), in double:
 *   Q4_K: sum_j d*sc_j*dx_j*P_j - dmin*m_j*dx_j*S_j,  S_j = sum of q_x in j
 *   Q6_K: sum_k d*sc_k*dx_{k/2}*P_k
 *   Q8_0: sum_b d*dx_b*P_b
 * absdot[r] = sum_i |w_i * dx_i*q_x_i| (the tolerance scale). */
int orc_gemv_w4a8(int fmt, const uint8_t* W, int64_t rows, int64_t cols,
                  const int8_t* qx, const float* dx, double* y, double* absdot,
                  int nthreads) {
    int64_t rb = orc_row_bytes(fmt, cols);
    if (!W || !qx || !dx || !y || rows <= 0 || rb < 0) return ORC_ERR_ARG;
    if (nthreads < 1) nthreads = 1;
    int gs = orc_partial_group(fmt);
    int64_t ng = cols / gs;
    int err = ORC_OK;
#pragma omp parallel num_threads(nthreads)
    {
        int64_t* P = (int64_t*)malloc(sizeof(int64_t) * (size_t)ng);
        double* w = (double*)malloc(sizeof(double) * (size_t)cols);
        if (!P || !w) {
#pragma omp atomic write
            err = ORC_ERR_ARG;
        }
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; r++) {
            if (!P || !w) continue;
            const uint8_t* row = W + r * rb;
            if (row_partials(fmt, row, cols, qx, P) != ORC_OK) {
#pragma omp atomic write
                err = ORC_ERR_OVERFLOW;
                continue;
            }
            double acc = 0.0;
            for (int64_t g = 0; g < ng; g++) {
                int64_t col0 = g * gs;
                const uint8_t* blk = row + (col0 / orc_block_weights(fmt)) * orc_block_bytes(fmt);
                double dxg = (double)dx[col0 / 32];
                if (fmt == ORC_Q4_K) {
                    int j = (int)((col0 % 256) / 32), sc, m;
                    q4k_scale_min(blk + 4, j, &sc, &m);
                    int64_t S = 0;
                    for (int i = 0; i < 32; i++) S += qx[col0 + i];
                    acc += f16_at(blk) * sc * dxg * (double)P[g]
                         - f16_at(blk + 2) * m * dxg * (double)S;
                } else if (fmt == ORC_Q6_K) {
                    int sc = q6k_scale(blk, (int)(col0 % 256));
                    acc += f16_at(blk + 208) * sc * dxg * (double)P[g];
                } else {
                    acc += f16_at(blk) * dxg * (double)P[g];
                }
            }
            y[r] = acc;
            if (absdot) {
                orc_dequant_row(fmt, row, cols, w);
                double aacc = 0.0;
                for (int64_t i = 0; i < cols; i++)
                    aacc += fabs(w[i] * ((double)dx[i / 32] * qx[i]));
                absdot[r] = aacc;
            }
        }
        free(P);
        free(w);
    }
    return err;
}

/* Prefill: the rows of X are independent W4A8 GEMVs (colibri GPU_BACKENDS.md,
 * XDNA lane: C = A x B is row-independent).  Y is [m, rows] row-major. */
int orc_gemm_w4a8(int fmt, const uint8_t* W, int64_t rows, int64_t cols,
                  int64_t m, const int8_t* qx, const float* dx, double* Y,
                  double* absdot, int nthreads) {
    if (m <= 0) return ORC_ERR_ARG;
    for (int64_t i = 0; i < m; i++) {
        int rc = orc_gemv_w4a8(fmt, W, rows, cols, qx + i * cols, dx + i * (cols / 32),
                               Y + i * rows, absdot ? absdot + i * rows : NULL, nthreads);
        if (rc != ORC_OK) return rc;
    }
    return ORC_OK;
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
