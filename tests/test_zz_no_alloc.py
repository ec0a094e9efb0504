"""qx_gemv_chain_noalloc: the chain entry point that allocates nothing.

Some callers cannot allocate device memory where they run a chain (during
CUDA graph capture, in pool-only runtimes, in plug-ins barred from the
process allocator); this entry point keeps the chain's arrival counters in a
fixed array inside the library instead of caller scratch.  The test calls it
through the C ABI twice in a row and checks each result against
qx_gemv_chain (caller scratch) within the tolerance the parity tests use,
1e-4 * sum_i |w_i * x_i| per row.  It runs last (file name) and also alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_quantized_gemv_q8_gb300 as qx
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module")
def lib():
    qx.build_library()
    L = qx.lib()
    L.qx_gemv_chain_noalloc.argtypes = [ctypes.c_int, ctypes.POINTER(qx._Job), ctypes.c_void_p]
    L.qx_gemv_chain_noalloc.restype = ctypes.c_int
    return L


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_noalloc_chain_matches_chain_with_scratch(lib):
    specs = [(synth.Q4_K, [300, 64], 4096), (synth.Q6_K, [129], 14336), (synth.Q8_0, [151, 33], 896),
             (synth.Q4_K, [4096], 4096)]
    host = []
    jobs = []
    for i, (fmt, rows, cols) in enumerate(specs):
        Ws = [synth.weights(fmt, r, cols, seed=900 + 10 * i + k) for k, r in enumerate(rows)]
        x = synth.activation(1, cols, seed=950 + i)
        host.append((fmt, Ws, rows, cols, x))
        jobs.append(qx.GemvJob(fmt, [dev(W) for W in Ws], rows, cols, dev(x[0])))

    # the existing entry point, with caller-owned scratch
    qx.qx_gemv_chain(jobs, qx.chain_scratch(len(jobs)))
    torch.cuda.synchronize()
    ref = [[y.cpu().numpy().astype(np.float64) for y in job.y] for job in jobs]

    # tolerance scale per row from the oracle (inputs from the generators only)
    absdot = []
    for fmt, Ws, rows, cols, x in host:
        q, d, _ = oracle.quantize_act_q8(x)
        absdot.append([oracle.gemv_w4a8(fmt, W, r, cols, q[0], d[0])[1] for W, r in zip(Ws, rows)])

    stream = torch.cuda.current_stream()
    for call in range(2):
        outs = []
        for job in jobs:
            job.y = [torch.full((r,), float("nan"), dtype=torch.float32, device="cuda") for r in job.rows]
            outs.append(job.y)
        arr = qx.make_chain(jobs)
        st = lib.qx_gemv_chain_noalloc(len(arr), arr, ctypes.c_void_p(stream.cuda_stream))
        assert st == qx.QX_OK, qx.qx_status_string(st)
        assert qx.qx_device_check(stream) == qx.QX_OK
        for j, ys in enumerate(outs):
            for k, y in enumerate(ys):
                got = y.cpu().numpy().astype(np.float64)
                err = np.abs(got - ref[j][k])
                assert np.all(err <= TOL * absdot[j][k]), f"call {call} job {j} entry {k}: max err {err.max()}"


@pytest.mark.parametrize("left_over", [1, 152, 0x7FFFFFFF])
def test_noalloc_chain_starts_from_stale_counters(lib, left_over):
    """The library's counter array keeps whatever the last call left (a chain
    stopped by a wait that ran out leaves counts behind).  Fill it with such
    values, then run the entry point: it clears the counters itself, so the
    outputs match qx_gemv_chain with fresh caller scratch, bit for bit."""
    specs = [(synth.Q4_K, [256, 64], 2048), (synth.Q8_0, [96], 896), (synth.Q6_K, [40], 4096)]
    jobs, again = [], []
    for i, (fmt, rows, cols) in enumerate(specs):
        Ws = [dev(synth.weights(fmt, r, cols, seed=1200 + 10 * i + k)) for k, r in enumerate(rows)]
        x = dev(synth.activation(1, cols, seed=1250 + i)[0])
        jobs.append(qx.GemvJob(fmt, Ws, rows, cols, x))
        again.append(qx.GemvJob(fmt, Ws, rows, cols, x))
    qx.qx_gemv_chain(jobs, qx.chain_scratch(len(jobs)))
    qx.qx_debug_noalloc_fill(left_over)
    for job in again:
        job.y = [torch.full((r,), float("nan"), dtype=torch.float32, device="cuda") for r in job.rows]
    stream = torch.cuda.current_stream()
    arr = qx.make_chain(again)
    assert lib.qx_gemv_chain_noalloc(len(arr), arr, ctypes.c_void_p(stream.cuda_stream)) == qx.QX_OK
    assert qx.qx_device_check(stream) == qx.QX_OK
    for a, b in zip(jobs, again):
        for ya, yb in zip(a.y, b.y):
            assert torch.equal(ya.view(torch.int32), yb.view(torch.int32))


def test_noalloc_chain_rejects_too_many_jobs(lib):
    W = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    jobs = [qx.GemvJob(synth.Q4_K, [W], [4], 256, x) for _ in range(qx.QX_CHAIN_MAX_JOBS + 1)]
    arr = qx.make_chain(jobs)
    assert lib.qx_gemv_chain_noalloc(len(arr), arr, None) == qx.QX_ERR_ARG


def test_noalloc_chain_through_the_binding(lib):
    """The binding's qx_gemv_chain_noalloc gives the scratch chain's outputs bit for bit,
    and refuses an over-long chain with a named status."""
    specs = [(synth.Q4_K, [200, 56], 2048), (synth.Q8_0, [96], 896)]
    jobs, again = [], []
    for i, (fmt, rows, cols) in enumerate(specs):
        Ws = [dev(synth.weights(fmt, r, cols, seed=970 + 10 * i + k)) for k, r in enumerate(rows)]
        x = dev(synth.activation(1, cols, seed=990 + i)[0])
        jobs.append(qx.GemvJob(fmt, Ws, rows, cols, x))
        again.append(qx.GemvJob(fmt, Ws, rows, cols, x))
    qx.qx_gemv_chain(jobs, qx.chain_scratch(len(jobs)))
    qx.qx_gemv_chain_noalloc(again)
    torch.cuda.synchronize()
    for a, b in zip(jobs, again):
        for ya, yb in zip(a.y, b.y):
            assert torch.equal(ya.view(torch.int32), yb.view(torch.int32))
    assert qx.qx_device_check() == qx.QX_OK
    W = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    too_many = [qx.GemvJob(synth.Q4_K, [W], [4], 256, x) for _ in range(qx.QX_CHAIN_MAX_JOBS + 1)]
    with pytest.raises(qx.QxError) as e:
        qx.qx_gemv_chain_noalloc(too_many)
    assert e.value.status == qx.QX_ERR_ARG
