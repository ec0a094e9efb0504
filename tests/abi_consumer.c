/* A plain C99 consumer of include/qx.h: the header compiles as C, the library
 * links and loads from C, and the calls that need no GPU behave as declared
 * (row sizes, status strings, version, argument errors returned before any
 * device work).  Built and run by tests/test_abi.py; prints "ok" on success. */
#include <stdio.h>
#include <string.h>

#include "qx.h"

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

    if (failures) return 1;
    printf("ok\n");
    return 0;
}
