"""Load-time repack of Q6_K into the aligned QX_Q6_K_SOA layout (qx_repack),
and the GEMV on it.

The pages make block repacking a per-device load-time decision (llamay docs,
"Backends and hardware", section "Repacking is a per-device decision now").
The repacked layout holds the same values, so every result on it must equal
the GGUF-layout result bit for bit, and the integer partial sums must equal
the oracle's."""
import numpy as np
import pytest
import torch

import block_quantized_gemv_q8_gb300 as qx
import oracle
import synth

pytestmark = pytest.mark.gpu
Q6, SOA = qx.QX_Q6_K, qx.QX_Q6_K_SOA


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


def bits(t):
    return host(t).view(np.uint32)


def expected_soa(W: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """The documented layout, restated with numpy slicing (test code)."""
    nsb = cols // 256
    rb = qx.qx_row_bytes(SOA, cols)
    G = W.reshape(rows, nsb, 210)
    out = np.zeros((rows, rb), np.uint8)
    out[:, : 208 * nsb] = G[:, :, :208].reshape(rows, 208 * nsb)
    out[:, 208 * nsb: 208 * nsb + 2 * nsb] = G[:, :, 208:].reshape(rows, 2 * nsb)
    return out


# nsb a multiple of 8 (same row size as GGUF) and not (9 super-blocks: padded d area)
SHAPES = [(1, 256), (129, 1024), (300, 4096), (65, 14336), (9, 2304), (64, 32768)]


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_repack_layout_and_round_trip(rows, cols):
    W = synth.weights(Q6, rows, cols, seed=rows + cols)
    R = qx.qx_repack(Q6, SOA, dev(W), rows, cols)
    assert np.array_equal(host(R).reshape(rows, -1), expected_soa(W, rows, cols))
    back = qx.qx_repack(SOA, Q6, R, rows, cols)
    assert np.array_equal(host(back), W.reshape(-1)), "round trip changed bytes"


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_repacked_gemv_is_bit_identical(rows, cols):
    W = synth.weights(Q6, rows, cols, seed=3 * rows + cols)
    Wg = dev(W)
    Ws = qx.qx_repack(Q6, SOA, Wg, rows, cols)
    x = synth.activation(1, cols, seed=cols + 11)
    a = qx.qx_quantize_act_q8(dev(x))
    xf = dev(x[0])
    FU, PDL = qx.QX_MODE_W4A8_FUSED, qx.QX_FLAG_PDL
    modes = [(qx.QX_MODE_W4A8, a), (FU, xf), (FU | PDL, xf)]
    if cols <= 16384:  # the f32-mode lanes serve rows up to 16384 columns
        modes += [(qx.QX_MODE_F32, xf), (qx.QX_MODE_F32 | PDL, xf)]
    for mode, arg in modes:
        yg = qx.qx_gemv(Q6, Wg, rows, cols, arg, mode=mode)
        ys = qx.qx_gemv(SOA, Ws, rows, cols, arg, mode=mode)
        assert np.array_equal(bits(ys), bits(yg)), f"mode {mode:#x}"
    q, d, s = oracle.quantize_act_q8(x)
    P = host(qx.qx_gemv_partials(SOA, Ws, rows, cols, a))
    assert np.array_equal(P, oracle.partials(Q6, W, rows, cols, q[0]))
    ref, absdot = oracle.gemv_w4a8(Q6, W, rows, cols, q[0], d[0])
    y = host(qx.qx_gemv(SOA, Ws, rows, cols, a, mode=qx.QX_MODE_W4A8)).astype(np.float64)
    assert np.all(np.abs(y - ref) <= 1e-4 * absdot)


def test_repacked_multi_and_prefill():
    cols = 1024
    rows = [300, 77]
    Wh = [synth.weights(Q6, r, cols, seed=40 + r) for r in rows]
    Wg = [dev(w) for w in Wh]
    Ws = [qx.qx_repack(Q6, SOA, w, r, cols) for w, r in zip(Wg, rows)]
    x = synth.activation(1, cols, seed=41)
    xf = dev(x[0])
    FU = qx.QX_MODE_W4A8_FUSED
    ys = qx.qx_gemv_multi([SOA, SOA], Ws, rows, cols, xf, mode=FU)
    yg = qx.qx_gemv_multi([Q6, Q6], Wg, rows, cols, xf, mode=FU)
    for a, b in zip(ys, yg):
        assert np.array_equal(bits(a), bits(b))
    # prefill: the automatic path and path 1 serve the repacked layout, one GEMV per row of X
    X = synth.activation(3, cols, seed=42)
    act = qx.qx_quantize_act_q8(dev(X))
    Yg = qx.qx_gemm_prefill_ex(Q6, Wg[0], rows[0], cols, act, path=1)
    for path in (0, 1):
        Ys = qx.qx_gemm_prefill_ex(SOA, Ws[0], rows[0], cols, act, path=path)
        assert np.array_equal(bits(Ys), bits(Yg))
    assert qx.qx_device_check() == qx.QX_OK
