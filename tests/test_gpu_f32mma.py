"""f32 mode on the tensor pipe: Q6_K rows (GGUF blocks and QX_Q6_K_SOA) of
2048 and 4096 columns and Q4_K rows of 256 to 4096 columns, whose
f32-mode GEMV runs as bf16 mma.sync over the exact quants (q - 32; q) and
the activation split into hi + lo bf16 terms (scaled per 256-column
super-block by a power of two); the Q4_K min term from each sub-block's sum
of the activation.

Gates: the f32-mode tolerance |y - y_ref| <= 1e-4 * sum_i |w_i x_i| per row
against the oracle, and the kernel's own error bound (2^-16 of the same sum,
about four times its analysis) wherever every activation lies within 2^-100
of its super-block's largest magnitude; both layouts bit-identical; a CUDA
graph and the multi-matrix launch give the eager bits.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_q8_gb300 as qx
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4
TIGHT = 2.0 ** -16
Q6, SOA = synth.Q6_K, qx.QX_Q6_K_SOA


@pytest.fixture(scope="module", autouse=True)
def _lib():
    qx.build_library()
    qx.lib()
    assert qx.qx_device_check() == qx.QX_OK


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    return host(t).view(np.uint32)


def check(y, ref, absdot, what, tight=True):
    err = np.abs(np.asarray(y, dtype=np.float64) - ref)
    bad = np.nonzero(~(err <= TOL * absdot))[0]
    assert bad.size == 0, f"{what}: row {bad[0]} err {err[bad[0]]} bound {TOL * absdot[bad[0]]}"
    if tight:
        bad = np.nonzero(~(err <= TIGHT * absdot))[0]
        assert bad.size == 0, f"{what}: row {bad[0]} err {err[bad[0]]} above 2^-16 of {absdot[bad[0]]}"


def both_layouts(W, rows, cols, x, mode=qx.QX_MODE_F32):
    Wg = dev(W)
    Ws = qx.qx_repack(Q6, SOA, Wg, rows, cols)
    xf = dev(x)
    yg = qx.qx_gemv(Q6, Wg, rows, cols, xf, mode=mode)
    ys = qx.qx_gemv(SOA, Ws, rows, cols, xf, mode=mode)
    assert np.array_equal(bits(ys), bits(yg)), "GGUF and repacked layouts differ"
    return host(yg)


@pytest.mark.parametrize("rows,cols", [(1, 2048), (17, 4096), (1005, 4096), (333, 2048), (2500, 4096)])
def test_f32_tensor_parity(rows, cols):
    W = synth.weights(Q6, rows, cols, seed=7 * rows + cols)
    x = synth.activation(1, cols, seed=cols + 17)[0]
    y = both_layouts(W, rows, cols, x)
    ref, absdot = oracle.gemv_f32(Q6, W, rows, cols, x)
    check(y, ref, absdot, f"{rows}x{cols}")
    yp = both_layouts(W, rows, cols, x, mode=qx.QX_MODE_F32 | qx.QX_FLAG_PDL)
    assert np.array_equal(yp.view(np.uint32), y.view(np.uint32))
    assert qx.qx_device_check() == qx.QX_OK


@pytest.mark.parametrize("k", [-130, -100, -60, 60, 100])
def test_f32_tensor_activation_scale(k):
    """The activation times 2^k: the per-super-block power of two keeps both
    bf16 terms normal, from blocks whose largest value is an f32 subnormal
    (k = -130) to values near 2^100."""
    rows, cols = 200, 4096
    W = synth.weights(Q6, rows, cols, seed=50)
    x = (synth.activation(1, cols, seed=51)[0].astype(np.float64) * 2.0 ** k).astype(np.float32)
    y = both_layouts(W, rows, cols, x)
    ref, absdot = oracle.gemv_f32(Q6, W, rows, cols, x)
    assert np.all(np.isfinite(y))
    # 2^-130: y itself lies among the f32 subnormals, whose spacing 2^-149 is
    # above 2^-16 of some rows' sums: only the f32-mode tolerance applies there
    check(y, ref, absdot, f"2^{k}", tight=k > -130)


def test_f32_tensor_mixed_magnitudes():
    """Activations spread over 2^-40 .. 2^40 inside every super-block, zeros,
    and one super-block entirely zero."""
    rows, cols = 300, 4096
    rng = np.random.default_rng(52)
    W = synth.weights(Q6, rows, cols, seed=53)
    x = rng.standard_normal(cols) * 2.0 ** rng.integers(-40, 41, cols)
    x[rng.choice(cols, 300, replace=False)] = 0.0
    x[256 * 5:256 * 6] = 0.0
    x = x.astype(np.float32)
    y = both_layouts(W, rows, cols, x)
    ref, absdot = oracle.gemv_f32(Q6, W, rows, cols, x)
    check(y, ref, absdot, "mixed")


def test_f32_tensor_zero_cases():
    """All-zero weights or activation give exact zeros; a zero activation
    outside one 16-column group reads only that group's products."""
    rows, cols = 40, 2048
    W = synth.weights(Q6, rows, cols, seed=54)
    x = synth.activation(1, cols, seed=55)[0]
    assert np.all(both_layouts(np.zeros_like(W), rows, cols, x) == 0)
    assert np.all(both_layouts(W, rows, cols, np.zeros_like(x)) == 0)
    xg = np.zeros_like(x)
    xg[256 * 3 + 16 * 9:256 * 3 + 16 * 10] = x[:16]
    y = both_layouts(W, rows, cols, xg)
    ref, absdot = oracle.gemv_f32(Q6, W, rows, cols, xg)
    check(y, ref, absdot, "one group")


def test_f32_tensor_multi_and_graph():
    """Two matrices in one launch (ragged rows) equal the separate launches;
    a captured CUDA graph replays the eager bits."""
    cols = 4096
    rows = [300, 77]
    Wh = [synth.weights(Q6, r, cols, seed=60 + r) for r in rows]
    Wg = [dev(w) for w in Wh]
    x = dev(synth.activation(1, cols, seed=61)[0])
    F = qx.QX_MODE_F32
    ys = qx.qx_gemv_multi([Q6, Q6], Wg, rows, cols, x, mode=F)
    for W, r, y in zip(Wg, rows, ys):
        assert np.array_equal(bits(y), bits(qx.qx_gemv(Q6, W, r, cols, x, mode=F)))
    stream = torch.cuda.Stream()
    yg = [torch.full((r,), float("nan"), device="cuda") for r in rows]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        qx.qx_gemv_multi([Q6, Q6], Wg, rows, cols, x, ys=yg, mode=F | qx.QX_FLAG_PDL, stream=stream)
    g.replay()
    for a, b in zip(yg, ys):
        assert np.array_equal(bits(a), bits(b))
    assert qx.qx_device_check() == qx.QX_OK


# ----------------------------------------------------------------- Q4_K ----
Q4 = synth.Q4_K
# Q4_K: w = d sc q - dmin m; the two terms of a sub-block may cancel, so the
# kernel's own bound is looser relative to sum |w x| than for Q6_K
TIGHT_Q4 = 2.0 ** -13


def check_q4(y, ref, absdot, what):
    err = np.abs(np.asarray(y, dtype=np.float64) - ref)
    bad = np.nonzero(~(err <= TOL * absdot))[0]
    assert bad.size == 0, f"{what}: row {bad[0]} err {err[bad[0]]} bound {TOL * absdot[bad[0]]}"
    bad = np.nonzero(~(err <= TIGHT_Q4 * absdot))[0]
    assert bad.size == 0, f"{what}: row {bad[0]} err {err[bad[0]]} above 2^-13 of {absdot[bad[0]]}"


@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 768), (300, 1024), (1005, 4096), (14336, 4096)])
def test_f32_tensor_q4k_parity(rows, cols):
    """Ragged rows, one to sixteen super-blocks a row (three: 15 of 16 warps
    in use); a large launch under programmatic dependent launch gives the
    same bits (small ones take the merged lanes, checked elsewhere)."""
    W = synth.weights(Q4, rows, cols, seed=11 * rows + cols)
    x = synth.activation(1, cols, seed=cols + 23)[0]
    Wd, xd = dev(W), dev(x)
    y = host(qx.qx_gemv(Q4, Wd, rows, cols, xd, mode=qx.QX_MODE_F32))
    ref, absdot = oracle.gemv_f32(Q4, W, rows, cols, x)
    check_q4(y, ref, absdot, f"q4_k {rows}x{cols}")
    if rows * cols >= 14336 * 4096:  # more than 192 KB a SM: the tensor pipe under PDL too
        yp = host(qx.qx_gemv(Q4, Wd, rows, cols, xd, mode=qx.QX_MODE_F32 | qx.QX_FLAG_PDL))
        assert np.array_equal(yp.view(np.uint32), y.view(np.uint32))
    assert qx.qx_device_check() == qx.QX_OK


@pytest.mark.parametrize("k", [-130, -100, 60, 100])
def test_f32_tensor_q4k_activation_scale(k):
    rows, cols = 200, 4096
    W = synth.weights(Q4, rows, cols, seed=56)
    x = (synth.activation(1, cols, seed=57)[0].astype(np.float64) * 2.0 ** k).astype(np.float32)
    y = host(qx.qx_gemv(Q4, dev(W), rows, cols, dev(x), mode=qx.QX_MODE_F32))
    ref, absdot = oracle.gemv_f32(Q4, W, rows, cols, x)
    assert np.all(np.isfinite(y))
    if k > -130:
        check_q4(y, ref, absdot, f"q4_k 2^{k}")
    else:  # y among the f32 subnormals: the f32-mode tolerance only
        err = np.abs(y.astype(np.float64) - ref)
        assert np.all(err <= TOL * absdot)


def test_f32_tensor_q4k_zero_cases_and_multi():
    """Zero weights or activation give exact zeros; two Q4_K matrices in one
    launch equal the separate launches; a CUDA graph replays the eager bits."""
    rows, cols = 40, 1024
    W = synth.weights(Q4, rows, cols, seed=58)
    x = synth.activation(1, cols, seed=59)[0]
    assert np.all(host(qx.qx_gemv(Q4, dev(np.zeros_like(W)), rows, cols, dev(x), mode=qx.QX_MODE_F32)) == 0)
    assert np.all(host(qx.qx_gemv(Q4, dev(W), rows, cols, dev(np.zeros_like(x)), mode=qx.QX_MODE_F32)) == 0)
    cols = 4096
    rows2 = [3000, 77]
    Wh = [synth.weights(Q4, r, cols, seed=70 + r) for r in rows2]
    Wg = [dev(w) for w in Wh]
    xg = dev(synth.activation(1, cols, seed=71)[0])
    F = qx.QX_MODE_F32
    ys = qx.qx_gemv_multi([Q4, Q4], Wg, rows2, cols, xg, mode=F)
    for Wd, r, y in zip(Wg, rows2, ys):
        assert np.array_equal(bits(y), bits(qx.qx_gemv(Q4, Wd, r, cols, xg, mode=F)))
    stream = torch.cuda.Stream()
    yg = [torch.full((r,), float("nan"), device="cuda") for r in rows2]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        qx.qx_gemv_multi([Q4, Q4], Wg, rows2, cols, xg, ys=yg, mode=F, stream=stream)
    g.replay()
    for a, b in zip(yg, ys):
        assert np.array_equal(bits(a), bits(b))
    assert qx.qx_device_check() == qx.QX_OK
