"""GPU tests of qx_gemv_chain: a chain of dependent W4A8 GEMVs in one launch.

Every row of a chain job is computed by the same lane code, team layout and
reduction order as a single qx_gemv launch in QX_MODE_W4A8_FUSED, so the
outputs must be equal bit for bit; the single launch is itself checked
against the oracle (test_gpu_parity.py), and one chain is checked against
the oracle directly here.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_q8_gb300 as qx
import oracle
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qx.build_library()
    qx.lib()
    assert qx.qx_device_check() == qx.QX_OK


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits(t):
    torch.cuda.synchronize()
    return t.cpu().numpy().view(np.uint32)


def single(job):
    return qx.qx_gemv_multi([job.fmt] * len(job.W), job.W, job.rows, job.cols, job.x,
                            mode=qx.QX_MODE_W4A8_FUSED)


def test_chain_of_independent_jobs_matches_single_launches():
    specs = [(synth.Q4_K, [4096, 1024, 1024], 4096), (synth.Q4_K, [4096], 4096),
             (synth.Q4_K, [1000, 77], 4096), (synth.Q6_K, [300], 14336), (synth.Q8_0, [151, 33], 896),
             (synth.Q4_K, [64], 1024)]
    jobs = []
    for i, (fmt, rows, cols) in enumerate(specs):
        Ws = [dev(synth.weights(fmt, r, cols, seed=200 + 10 * i + k)) for k, r in enumerate(rows)]
        x = dev(synth.activation(1, cols, seed=300 + i)[0])
        jobs.append(qx.GemvJob(fmt, Ws, rows, cols, x))
    scratch = qx.chain_scratch(len(jobs))
    qx.qx_gemv_chain(jobs, scratch)
    for job in jobs:
        for y_chain, y_single in zip(job.y, single(job)):
            assert np.array_equal(bits(y_chain), bits(y_single))
    assert qx.qx_device_check() == qx.QX_OK
    assert int(scratch.sum()) == 0, "a completed chain leaves its scratch zero-filled"


def test_dependent_chain_reads_previous_output():
    """x of job j + 1 is y of job j: same results as sequential launches."""
    fmt, n, cols = synth.Q4_K, 4096, 4096
    Ws = [dev(synth.weights(fmt, n, cols, seed=400 + i)) for i in range(6)]
    x0 = dev(synth.activation(1, cols, seed=401)[0])
    ys = [torch.empty(n, dtype=torch.float32, device="cuda") for _ in Ws]
    jobs = [qx.GemvJob(fmt, [W], [n], cols, x0 if i == 0 else ys[i - 1], [ys[i]]) for i, W in enumerate(Ws)]
    scratch = qx.chain_scratch(len(jobs))
    for rep in range(2):  # the same scratch serves consecutive calls
        for y in ys:
            y.fill_(float("nan"))
        qx.qx_gemv_chain(jobs, scratch)
        x = x0
        for W, y in zip(Ws, ys):
            ref = qx.qx_gemv(fmt, W, n, cols, x, mode=qx.QX_MODE_W4A8_FUSED)
            assert np.array_equal(bits(y), bits(ref)), f"rep {rep}"
            x = ref
    assert qx.qx_device_check() == qx.QX_OK
    assert int(scratch.sum()) == 0


def test_chain_against_oracle():
    fmt, rows, cols = synth.Q6_K, 257, 4096
    W = synth.weights(fmt, rows, cols, seed=500)
    x = synth.activation(1, cols, seed=501)
    job = qx.GemvJob(fmt, [dev(W)], [rows], cols, dev(x[0]))
    qx.qx_gemv_chain([job], qx.chain_scratch(1))
    q, d, _ = oracle.quantize_act_q8(x)
    ref, absdot = oracle.gemv_w4a8(fmt, W, rows, cols, q[0], d[0])
    torch.cuda.synchronize()
    err = np.abs(job.y[0].cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 1e-4 * absdot)


def test_chain_quantises_subnormal_scale_blocks_like_the_oracle():
    """A chain job over an activation whose block scales are f32 subnormals (the
    codes clamp to +-127): same int8 codes as the oracle, so the same y as the
    two-step path with the oracle-checked standalone quantiser."""
    from tests.test_gpu_parity import subnormal_scale_activation
    fmt, rows = synth.Q4_K, 96
    x = subnormal_scale_activation(128, seed=9)
    cols = x.shape[1]
    W = dev(synth.weights(fmt, rows, cols, seed=510))
    a = qx.qx_quantize_act_q8(dev(x))
    q, d, s = oracle.quantize_act_q8(x)
    torch.cuda.synchronize()
    assert np.array_equal(a.q.cpu().numpy(), q) and np.array_equal(a.sum.cpu().numpy(), s)
    y_two_step = qx.qx_gemv(fmt, W, rows, cols, a, mode=qx.QX_MODE_W4A8)
    job = qx.GemvJob(fmt, [W], [rows], cols, dev(x[0]))
    qx.qx_gemv_chain([job], qx.chain_scratch(1))
    assert np.array_equal(bits(job.y[0]), bits(y_two_step))
    assert qx.qx_device_check() == qx.QX_OK


def test_chain_argument_errors():
    W = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, dtype=torch.float32, device="cuda")
    job = qx.GemvJob(synth.Q4_K, [W], [4], 256, x)
    with pytest.raises(qx.QxError) as ei:
        qx.qx_gemv_chain([job], qx.chain_scratch(1)[1:])  # misaligned scratch
    assert ei.value.status == qx.QX_ERR_ALIGN
    bad = qx.GemvJob(synth.Q4_K, [W], [4], 896, x)
    with pytest.raises(qx.QxError) as ei:
        qx.qx_gemv_chain([bad], qx.chain_scratch(1))
    assert ei.value.status == qx.QX_ERR_SHAPE
    assert qx.qx_gemv_chain_scratch_bytes(0) == 0
    assert qx.qx_gemv_chain_scratch_bytes(qx.QX_CHAIN_MAX_JOBS + 1) == 0
