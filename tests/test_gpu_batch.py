"""Small-batch GEMV (qx_gemm_prefill_ex path 4): several rows of a quantised
activation against one stream of the weights, compared with the oracle.

The rows of X are independent W4A8 GEMVs (colibri GPU_BACKENDS.md, XDNA
lane: C = A x B is row-independent), so the oracle's prefill is one W4A8
GEMV per row of X; every output must lie within 1e-4 * sum|w * x'| of it.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_q8_gb300 as qx
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qx.build_library()
    qx.lib()
    assert qx.qx_device_check() == qx.QX_OK


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def check(fmt, W, rows, cols, X, what, sample_rows=None):
    a = qx.qx_quantize_act_q8(dev(X))
    q, d, s = oracle.quantize_act_q8(X)
    assert np.array_equal(host(a.q), q) and np.array_equal(host(a.d).view(np.uint32), d.view(np.uint32))
    m = X.shape[0]
    # one guard row after Y: the kernel must write exactly Y[m, rows]
    Yg = torch.full((m + 1, rows), float("nan"), device="cuda")
    qx.qx_gemm_prefill_ex(fmt, dev(W), rows, cols, a, Y=Yg[:m], path=4)
    Yh = host(Yg)
    assert np.all(np.isnan(Yh[m])), f"{what}: wrote past Y"
    Y = Yh[:m]
    assert np.all(np.isfinite(Y)), f"{what}: unwritten or non-finite outputs"
    wr = np.arange(rows) if sample_rows is None else sample_rows
    ref, absdot = oracle.gemm_w4a8(fmt, np.ascontiguousarray(W[wr]), len(wr), cols, q, d)
    y = Y[:, wr].astype(np.float64)
    err = np.abs(y - ref)
    bad = np.argwhere(~(err <= TOL * absdot))
    assert bad.size == 0, (f"{what}: {len(bad)} outputs out of tolerance, e.g. {tuple(bad[0])}: "
                           f"y={y[tuple(bad[0])]} ref={ref[tuple(bad[0])]}")
    return Y


# ragged batches (1..16 rows of X: whole and partial groups of four or eight),
# ragged row counts (not multiples of the CTA split, of the stage or of the
# 16-row groups of the tensor path), narrow and wide rows.  Groups of five to
# eight rows of X against rows of up to 4096 columns in whole 256-column units
# whose bytes are a 16-byte multiple take the integer tensor path: Q4_K with
# 2, 3, 4, 9 and 16 units a row (8, 5, 4, 1 and 1 row groups a stage, some
# consumer warps idle), Q6_K at 2048 and 4096 columns, Q8_0 at 256 to 4096;
# the others, and groups of up to four rows, the dp4a lanes.
@pytest.mark.parametrize("fmt,m,rows,cols", [
    (synth.Q4_K, 1, 70, 1024), (synth.Q4_K, 2, 300, 4096), (synth.Q4_K, 6, 129, 256),
    (synth.Q4_K, 4, 1000, 4096), (synth.Q4_K, 5, 77, 14336), (synth.Q4_K, 8, 513, 1024),
    (synth.Q4_K, 9, 200, 768), (synth.Q4_K, 16, 45, 2304), (synth.Q4_K, 7, 1, 4096), (synth.Q4_K, 5, 1111, 512),
    (synth.Q6_K, 2, 300, 1024), (synth.Q6_K, 4, 129, 14336), (synth.Q6_K, 7, 33, 256),
    (synth.Q6_K, 6, 300, 2048), (synth.Q6_K, 8, 129, 4096), (synth.Q6_K, 16, 45, 2048),
    (synth.Q8_0, 2, 151, 896), (synth.Q8_0, 4, 300, 32), (synth.Q8_0, 6, 513, 864), (synth.Q8_0, 9, 128, 4096),
    (synth.Q8_0, 5, 77, 256), (synth.Q8_0, 8, 1000, 2048), (synth.Q8_0, 6, 3, 512),
])
def test_batch_matches_oracle(fmt, m, rows, cols):
    W = synth.weights(fmt, rows, cols, seed=80 + m + rows)
    X = synth.activation(m, cols, seed=81 + m)
    check(fmt, W, rows, cols, X, f"batch {synth.NAMES[fmt]} m={m} rows={rows} cols={cols}")


def test_batch_zero_rows_of_x_and_tail_bytes():
    """A zero row of X gives exact zeros; a matrix whose size is not a
    16-byte multiple (Q8_0, 3 rows of 34 bytes) takes its tail by plain loads."""
    fmt, rows, cols = synth.Q8_0, 3, 32
    W = synth.weights(fmt, rows, cols, seed=90)
    X = synth.activation(3, cols, seed=91)
    X[1] = 0.0
    Y = check(fmt, W, rows, cols, X, "zero row / tail bytes")
    assert np.all(Y[1] == 0.0)


def test_batch_tensor_path_zero_weights_give_exact_zeros():
    """Q4_K rows whose quants and dmin are zero (d and the 6-bit scales left
    as they are) are zero weights: the integer tensor path must give exact
    zeros there (integer partials of zero, a min term of zero), and the
    oracle's values elsewhere."""
    fmt, rows, cols, m = synth.Q4_K, 200, 4096, 8
    W = synth.weights(fmt, rows, cols, seed=95)
    blocks = W.reshape(rows, cols // 256, 144)
    zero_rows = np.array([0, 17, 63, 64, 150, 199])
    blocks[zero_rows, :, 2:4] = 0      # dmin
    blocks[zero_rows, :, 16:] = 0      # quants
    X = synth.activation(m, cols, seed=96)
    Y = check(fmt, W, rows, cols, X, "zero weight rows")
    assert np.all(Y[:, zero_rows] == 0.0)


@pytest.mark.parametrize("fmt", [synth.Q6_K, synth.Q8_0])
def test_batch_tensor_path_full_width(fmt):
    """Q6_K and Q8_0 rows of 4096 columns on the integer tensor path, eight
    rows of X, 2000 weight rows (several stages a CTA), sampled rows."""
    rows, cols, m = 2000, 4096, 8
    W = synth.weights(fmt, rows, cols, seed=97)
    X = synth.activation(m, cols, seed=98)
    rng = np.random.default_rng(99)
    wr = np.sort(np.concatenate([rng.choice(rows, 200, replace=False), [0, rows - 1]]))
    check(fmt, W, rows, cols, X, f"tensor path {synth.NAMES[fmt]}", sample_rows=wr)


@pytest.mark.parametrize("m", [4, 8])
def test_batch_full_size_sampled(m):
    """Llama-3.1-8B gate projection shape, Q4_K [14336, 4096], sampled rows."""
    fmt, rows, cols = synth.Q4_K, 14336, 4096
    W = synth.weights(fmt, rows, cols, seed=92)
    X = synth.activation(m, cols, seed=93 + m)
    rng = np.random.default_rng(94)
    wr = np.sort(np.concatenate([rng.choice(rows, 300, replace=False), [0, rows - 1]]))
    check(fmt, W, rows, cols, X, f"full size m={m}", sample_rows=wr)


def test_batch_and_repack_capture_in_a_graph():
    """The small-batch path and the repack allocate nothing: captured in a CUDA
    graph they replay to the eager bits."""
    fmt, rows, cols, m = synth.Q4_K, 300, 1024, 6
    W = dev(synth.weights(fmt, rows, cols, seed=130))
    X = qx.qx_quantize_act_q8(dev(synth.activation(m, cols, seed=131)))
    y_eager = host(qx.qx_gemm_prefill_ex(fmt, W, rows, cols, X, path=4))
    W6 = dev(synth.weights(synth.Q6_K, rows, cols, seed=132))
    x6 = dev(synth.activation(1, cols, seed=133)[0])
    y6_eager = host(qx.qx_gemv(synth.Q6_K, W6, rows, cols, x6, mode=qx.QX_MODE_W4A8_FUSED))
    Y = torch.full((m, rows), float("nan"), device="cuda")
    R = torch.zeros(rows * qx.qx_row_bytes(qx.QX_Q6_K_SOA, cols), dtype=torch.uint8, device="cuda")
    y6 = torch.full((rows,), float("nan"), device="cuda")
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        qx.qx_gemm_prefill_ex(fmt, W, rows, cols, X, Y=Y, path=4, stream=stream)
        qx.qx_repack(synth.Q6_K, qx.QX_Q6_K_SOA, W6, rows, cols, out=R, stream=stream)
        qx.qx_gemv(qx.QX_Q6_K_SOA, R, rows, cols, x6, y=y6, mode=qx.QX_MODE_W4A8_FUSED, stream=stream)
    g.replay()
    assert np.array_equal(host(Y).view(np.uint32), y_eager.view(np.uint32))
    assert np.array_equal(host(y6).view(np.uint32), y6_eager.view(np.uint32))
    assert qx.qx_device_check() == qx.QX_OK
