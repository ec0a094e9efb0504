/* A plain C99 consumer of include/qx.h and include/qx_debug.h: the header compiles as C, the library
 * links and loads from C, and the calls that need no GPU behave as declared
 * (row sizes, status strings, version, argument errors returned before any
 * device work).  Built and run by tests/test_abi.py, also against a build of
 * the library whose host code carries AddressSanitizer and
 * UndefinedBehaviorSanitizer; prints "ok" on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "qx.h"
#include "qx_debug.h"

static int failures = 0;

static void expect(int cond, const char* what) {
    if (!cond) {
        fprintf(stderr, "FAIL: %s\n", what);
        ++failures;
    }
}

int main(void) {
    void* const a16 = (void*)(uintptr_t)(1u << 20); /* 16-byte aligned, never dereferenced */
    void* const a2 = (void*)(uintptr_t)((1u << 20) + 2u);
    float* const y = (float*)a16;
    qx_act_q8 act;
    act.q = (int8_t*)a16;
    act.d = (float*)a16;
    act.sum = (int32_t*)a16;
    act.m = 1;
    act.cols = 64;

    expect(qx_row_bytes(QX_Q4_K, 4096) == 16 * 144, "Q4_K row bytes");
    expect(qx_row_bytes(QX_Q6_K, 14336) == 56 * 210, "Q6_K row bytes");
    expect(qx_row_bytes(QX_Q8_0, 896) == 28 * 34, "Q8_0 row bytes");
    expect(qx_row_bytes(QX_Q6_K_SOA, 4096) == qx_row_bytes(QX_Q6_K, 4096), "Q6_K_SOA row bytes at 4096");
    expect(qx_row_bytes(QX_Q4_K, 896) == 0, "Q4_K partial super-block");
    expect(strncmp(qx_status_string(QX_ERR_SHAPE), "QX_", 3) == 0, "status string");
    expect(strstr(qx_version(), "sm_103a") != NULL, "version names sm_103a");

    expect(qx_gemv((qx_fmt)99, a16, 4, 256, a16, y, QX_MODE_F32, NULL) == QX_ERR_FMT, "unknown format");
    expect(qx_gemv(QX_Q4_K, a16, 4, 256, a16, y, (qx_mode)7, NULL) == QX_ERR_MODE, "unknown mode");
    expect(qx_gemv(QX_Q4_K, a16, 4, 896, a16, y, QX_MODE_F32, NULL) == QX_ERR_SHAPE, "cols not whole blocks");
    expect(qx_gemv(QX_Q4_K, NULL, 4, 256, a16, y, QX_MODE_F32, NULL) == QX_ERR_ARG, "null weights");
    expect(qx_gemv(QX_Q4_K, a2, 4, 256, a16, y, QX_MODE_F32, NULL) == QX_ERR_ALIGN, "misaligned weights");
    expect(qx_quantize_act_q8((const float*)a16, 1, 40, &act, NULL) == QX_ERR_SHAPE, "activation cols");
    expect(qx_quantize_act_q8(NULL, 1, 64, &act, NULL) == QX_ERR_ARG, "null activation");
    expect(qx_gemv_chain(0, NULL, NULL, NULL) == QX_ERR_ARG, "empty chain");
    expect(qx_gemv_chain_noalloc(0, NULL, NULL) == QX_ERR_ARG, "empty chain without scratch");

    /* byte counts that would overflow: refused as a shape, nothing computed */
    expect(qx_gemv(QX_Q4_K, a16, INT64_MAX / 2, 256, a16, y, QX_MODE_F32, NULL) == QX_ERR_SHAPE, "huge rows");
    expect(qx_gemv(QX_Q4_K, a16, 4, INT64_MAX - 255, a16, y, QX_MODE_F32, NULL) == QX_ERR_SHAPE, "huge cols");
    expect(qx_quantize_act_q8((const float*)a16, INT64_MAX / 64, 64, &act, NULL) == QX_ERR_SHAPE,
           "huge activation");

    {
        qx_fmt f9[9];
        int i;
        for (i = 0; i < 9; ++i) f9[i] = QX_Q4_K;
        expect(qx_gemv_multi(0, f9, NULL, NULL, 256, a16, NULL, QX_MODE_F32, NULL) == QX_ERR_ARG, "multi of 0");
        expect(qx_gemv_multi(9, f9, NULL, NULL, 256, a16, NULL, QX_MODE_F32, NULL) == QX_ERR_ARG, "multi of 9");
    }
    {
        qx_act_q8 bad = act;
        bad.d = NULL;
        expect(qx_gemv_partials(QX_Q4_K, a16, 4, 256, &bad, (int32_t*)a16, NULL) == QX_ERR_ARG, "partials, no d");
    }
    {
        qx_act_q8 x4 = act;
        x4.m = 4;
        x4.cols = 256;
        expect(qx_gemm_prefill_ex(QX_Q4_K, a16, 4, 256, &x4, y, 5, NULL) == QX_ERR_ARG, "prefill path 5");
        expect(qx_gemm_prefill_ex(QX_Q6_K_SOA, a16, 4, 256, &x4, y, 3, NULL) == QX_ERR_FMT, "prefill of SOA");
    }
    expect(qx_repack(QX_Q4_K, QX_Q6_K_SOA, a16, 4, 256, (void*)(2 * (uintptr_t)a16), NULL) == QX_ERR_FMT,
           "repack from Q4_K");
    expect(qx_repack(QX_Q6_K, QX_Q6_K_SOA, a16, 4, 256, (void*)((uintptr_t)a16 + 256), NULL) == QX_ERR_ARG,
           "overlapping repack");
    {
        qx_gemv_job job;
        memset(&job, 0, sizeof(job));
        job.fmt = QX_Q6_K_SOA;
        job.n = 1;
        job.W[0] = a16;
        job.rows[0] = 4;
        job.y[0] = y;
        job.cols = 256;
        job.x = (const float*)a16;
        expect(qx_gemv_chain(1, &job, a16, NULL) == QX_ERR_FMT, "chain of SOA");
        job.fmt = QX_Q4_K;
        job.n = QX_CHAIN_MAX_ENTRIES + 1;
        expect(qx_gemv_chain(1, &job, a16, NULL) == QX_ERR_ARG, "chain job with too many entries");
    }
    {
        double rate = 0.0;
        expect(qx_debug_mma_rate(2, &rate, NULL) == QX_ERR_ARG, "mma rate kind");
        expect(qx_debug_mma_rate(0, NULL, NULL) == QX_ERR_ARG, "mma rate output");
    }
    expect(qx_debug_timeout_probe(10, NULL) == QX_ERR_ARG, "timeout probe limit");

#ifdef QX_PLANT_OOB
    /* sanitizer builds only: one byte read past a heap block must be reported */
    {
        volatile char* p = (volatile char*)malloc(16);
        volatile char c = p[16];
        (void)c;
        free((void*)p);
    }
#endif
    if (failures) return 1;
    printf("ok\n");
    return 0;
}
