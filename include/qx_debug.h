/*
 * qx_debug.h -- test and measurement hooks of libqx.so, kept apart from the
 * product calls in qx.h.  The test suite and the benchmark use them; an
 * application has no reason to.  Same conventions as qx.h (status codes,
 * streams, current device).
 */
#ifndef QX_DEBUG_H
#define QX_DEBUG_H

#include "qx.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launch one CTA that waits on a barrier nothing will complete, with a wait
 * limit of `limit_ns` nanoseconds (1 ms .. 10 s), so that the bounded-wait
 * path runs without any fault.  qx_device_check() then returns
 * QX_ERR_DEVICE_TIMEOUT.  QX_ERR_ARG for a limit outside that range. */
qx_status qx_debug_timeout_probe(uint64_t limit_ns, qx_stream_t s);

/* The device's warp-level tensor-core rate, multiply-adds x 2 per second, of
 * mma.sync int8 m16n8k32 (kind 0) or f16 m16n8k16 with an f32 accumulator
 * (kind 1), run from registers by every SM; sm_103a has no int8 tcgen05 MMA,
 * so kind 0 is the int8 tensor rate a prefill can use.  It allocates and
 * frees a small device buffer and synchronises stream s: not for use inside
 * a graph capture.  QX_ERR_ARG for a null out pointer or another kind. */
qx_status qx_debug_mma_rate(int kind, double* ops_per_s, qx_stream_t s);

/* Fill every word of the arrival-counter array that qx_gemv_chain_noalloc
 * keeps inside the library (on the current device) with `value`, on stream
 * s, so that a test can show that the entry point starts from whatever an
 * earlier call left there. */
qx_status qx_debug_noalloc_fill(uint32_t value, qx_stream_t s);

/* Measurement builds only (compiled with QX_TRACE): copy up to `bytes` of
 * the chain kernel's per-(CTA, job, event) timestamps to host memory.  Other
 * builds return QX_ERR_CUDA. */
qx_status qx_debug_trace_read(void* host, size_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* QX_DEBUG_H */
