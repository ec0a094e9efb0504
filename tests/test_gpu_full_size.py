"""GPU parity at the benchmark's full sizes, in the launch configuration the
benchmark times (in-kernel quantisation, programmatic dependent launch,
q/k/v and gate/up fused through qx_gemv_multi): sampled output rows against
the oracle, row by row.

Same gates as test_gpu_parity: activation codes bit-exact (checked through
qx_quantize_act_q8, whose codes the fused launches reproduce bit for bit),
f32 outputs within 1e-4 * sum_i |w_i * x_i| per row.
"""
import numpy as np
import pytest
import torch

import block_quantized_gemv_q8_gb300 as qx
import oracle
import synth

pytestmark = pytest.mark.gpu
TOL = 1e-4
FUSED_PDL = qx.QX_MODE_W4A8_FUSED | qx.QX_FLAG_PDL


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


def sample_rows(rows: int, n: int, seed: int) -> np.ndarray:
    """n distinct rows, always including the first and the last."""
    rng = np.random.default_rng(seed)
    pick = rng.choice(rows, min(n, rows), replace=False)
    return np.unique(np.concatenate([pick, [0, rows - 1]]))


def check_w4a8_rows(fmt, W, cols, x, y, rows_sel, what):
    """y[rows_sel] against the oracle's W4A8 product on those rows."""
    q, d, _ = oracle.quantize_act_q8(x.reshape(1, -1))
    ref, absdot = oracle.gemv_w4a8(fmt, np.ascontiguousarray(W[rows_sel]), len(rows_sel), cols, q[0], d[0])
    check(y[rows_sel], ref, absdot, what)


def check_f32_rows(fmt, W, cols, x, y, rows_sel, what):
    ref, absdot = oracle.gemv_f32(fmt, np.ascontiguousarray(W[rows_sel]), len(rows_sel), cols, x)
    check(y[rows_sel], ref, absdot, what)


def check(y, ref, absdot, what):
    err = np.abs(np.asarray(y, dtype=np.float64) - ref)
    bad = np.nonzero(~(err <= TOL * absdot))[0]
    assert bad.size == 0, f"{what}: {bad.size} sampled rows out of tolerance (first: err {err[bad[0]]})"


def assert_codes_match(x: np.ndarray):
    """The GPU's int8 codes, scales and block sums for x equal the oracle's."""
    a = qx.qx_quantize_act_q8(dev(x.reshape(1, -1)))
    q, d, s = oracle.quantize_act_q8(x.reshape(1, -1))
    assert np.array_equal(host(a.q), q)
    assert np.array_equal(host(a.d).view(np.uint32), d.view(np.uint32))
    assert np.array_equal(host(a.sum), s)


def test_llama8b_layer_full_size_sampled():
    """One Llama-3.1-8B decode layer (q,k,v,o,gate,up Q4_K; down Q6_K) as the
    benchmark launches it: four PDL launches in sequence on one stream."""
    shapes = {n: (f, r, c) for n, f, r, c in synth.LLAMA8B_LAYER}
    Wh = {n: synth.weights(f, r, c, seed=synth.seed_for(1, 0, j)) for j, (n, (f, r, c)) in enumerate(shapes.items())}
    xs = [synth.activation(1, c, seed=synth.seed_for(1, 0, 200 + k))[0] for k, c in enumerate([4096, 4096, 4096, 14336])]
    Wd = {n: dev(W) for n, W in Wh.items()}
    xd = [dev(x) for x in xs]
    y = {n: torch.empty(r, dtype=torch.float32, device="cuda") for n, (f, r, c) in shapes.items()}
    stream = torch.cuda.Stream()
    F = synth.Q4_K
    qx.qx_gemv_multi([F, F, F], [Wd["q"], Wd["k"], Wd["v"]], [4096, 1024, 1024], 4096, xd[0],
                     ys=[y["q"], y["k"], y["v"]], mode=FUSED_PDL, stream=stream)
    qx.qx_gemv(F, Wd["o"], 4096, 4096, xd[1], y=y["o"], mode=FUSED_PDL, stream=stream)
    qx.qx_gemv_multi([F, F], [Wd["gate"], Wd["up"]], [14336, 14336], 4096, xd[2],
                     ys=[y["gate"], y["up"]], mode=FUSED_PDL, stream=stream)
    # the benchmark's down projection: repacked at load into QX_Q6_K_SOA; the
    # GGUF-layout launch must give the same bits
    down_soa = qx.qx_repack(synth.Q6_K, qx.QX_Q6_K_SOA, Wd["down"], 4096, 14336)
    qx.qx_gemv(qx.QX_Q6_K_SOA, down_soa, 4096, 14336, xd[3], y=y["down"], mode=FUSED_PDL, stream=stream)
    y_down_gguf = torch.empty(4096, dtype=torch.float32, device="cuda")
    qx.qx_gemv(synth.Q6_K, Wd["down"], 4096, 14336, xd[3], y=y_down_gguf, mode=FUSED_PDL, stream=stream)
    stream.synchronize()
    assert qx.qx_device_check() == qx.QX_OK
    assert np.array_equal(host(y["down"]).view(np.uint32), host(y_down_gguf).view(np.uint32))
    xin = {"q": 0, "k": 0, "v": 0, "o": 1, "gate": 2, "up": 2, "down": 3}
    for k in range(4):
        assert_codes_match(xs[k])
    for j, (n, (f, r, c)) in enumerate(shapes.items()):
        sel = sample_rows(r, 96, seed=300 + j)
        check_w4a8_rows(f, Wh[n], c, xs[xin[n]], host(y[n]), sel, f"llama8b {n}")


@pytest.mark.parametrize("layout", ["gguf", "soa"])
@pytest.mark.parametrize("mode", ["w4a8", "f32"])
def test_lm_head_q6k_full_size_sampled(mode, layout):
    """The Q6_K lm_head, 128256 x 4096 (431 MB): the launches the benchmark
    times, on the GGUF blocks and repacked at load (W4A8: the merged
    producer/reducer variant, taken from 128 MB)."""
    _, fmt, rows, cols = synth.LLAMA8B_LM_HEAD_Q6K
    W = synth.weights(fmt, rows, cols, seed=20)
    x = synth.activation(1, cols, seed=21)[0]
    flag = FUSED_PDL if mode == "w4a8" else qx.QX_MODE_F32 | qx.QX_FLAG_PDL
    Wd = dev(W)
    if layout == "soa":
        y = host(qx.qx_gemv(qx.QX_Q6_K_SOA, qx.qx_repack(fmt, qx.QX_Q6_K_SOA, Wd, rows, cols), rows, cols, dev(x),
                            mode=flag))
        y_gguf = host(qx.qx_gemv(fmt, Wd, rows, cols, dev(x), mode=flag))
        assert np.array_equal(y.view(np.uint32), y_gguf.view(np.uint32))
    else:
        y = host(qx.qx_gemv(fmt, Wd, rows, cols, dev(x), mode=flag))
    assert qx.qx_device_check() == qx.QX_OK
    sel = sample_rows(rows, 256, seed=22)
    if mode == "w4a8":
        assert_codes_match(x)
        check_w4a8_rows(fmt, W, cols, x, y, sel, "lm_head w4a8")
    else:
        check_f32_rows(fmt, W, cols, x, y, sel, "lm_head f32")


def test_qwen05b_step_full_size_sampled():
    """A Qwen2-0.5B decode step's shapes (Q8_0 attention, Q4_K MLP, Q8_0 lm_head
    151936 x 896), launched as the benchmark does, each launch checked."""
    Q8, Q4 = synth.Q8_0, synth.Q4_K
    shapes = {n: (f, r, c) for n, f, r, c in synth.QWEN05B_LAYER}
    Wh = {n: synth.weights(f, r, c, seed=synth.seed_for(3, 0, j)) for j, (n, (f, r, c)) in enumerate(shapes.items())}
    _, lf, lr, lc = synth.QWEN05B_LM_HEAD
    Wlm = synth.weights(lf, lr, lc, seed=31)
    xs = [synth.activation(1, 1024, seed=40 + k, valid_cols=896 if k == 2 else None)[0] for k in range(3)]
    xdn = synth.activation(1, 4864, seed=44)[0]
    Wd = {n: dev(W) for n, W in Wh.items()}
    x_dev = [dev(x) for x in xs]
    xdn_dev = dev(xdn)
    y = {n: torch.empty(r, dtype=torch.float32, device="cuda") for n, (f, r, c) in shapes.items()}
    ylm = torch.empty(lr, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    qx.qx_gemv_multi([Q8] * 3, [Wd["q"], Wd["k"], Wd["v"]], [896, 128, 128], 896, x_dev[0][:896],
                     ys=[y["q"], y["k"], y["v"]], mode=FUSED_PDL, stream=stream)
    qx.qx_gemv(Q8, Wd["o"], 896, 896, x_dev[1][:896], y=y["o"], mode=FUSED_PDL, stream=stream)
    qx.qx_gemv_multi([Q4, Q4], [Wd["gate"], Wd["up"]], [4864, 4864], 1024, x_dev[2],
                     ys=[y["gate"], y["up"]], mode=FUSED_PDL, stream=stream)
    qx.qx_gemv(Q4, Wd["down"], 896, 4864, xdn_dev, y=y["down"], mode=FUSED_PDL, stream=stream)
    qx.qx_gemv(Q8, dev(Wlm), lr, lc, x_dev[0][:896], y=ylm, mode=FUSED_PDL, stream=stream)
    stream.synchronize()
    assert qx.qx_device_check() == qx.QX_OK
    xin = {"q": xs[0][:896], "k": xs[0][:896], "v": xs[0][:896], "o": xs[1][:896], "gate": xs[2], "up": xs[2],
           "down": xdn}
    for j, (n, (f, r, c)) in enumerate(shapes.items()):
        sel = sample_rows(r, 96, seed=400 + j)
        check_w4a8_rows(f, Wh[n], c, xin[n], host(y[n]), sel, f"qwen {n}")
    check_w4a8_rows(lf, Wlm, lc, xs[0][:896], host(ylm), sample_rows(lr, 256, seed=499), "qwen lm_head")
