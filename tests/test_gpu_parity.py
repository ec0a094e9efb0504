"""GPU parity: the CUDA path against the CPU oracle on the same seeded inputs.

Gates (the same in every test):
  * activation quants, scales and block sums: bit-exact;
  * integer partial sums of the W4A8 product: bit-exact;
  * f32 outputs: |y - y_ref| <= 1e-4 * sum_i |w_i * x_i| per row, where x is
    the f32 activation in f32 mode and the dequantised int8 activation in
    W4A8 mode.
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


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close(y, ref, absdot, what):
    y = np.asarray(y, dtype=np.float64)
    err = np.abs(y - ref)
    bound = TOL * absdot
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{what}: {bad.size} rows out of tolerance, e.g. row {bad[0]}: "
                           f"y={y[bad[0]]} ref={ref[bad[0]]} err={err[bad[0]]} bound={bound[bad[0]]}")


def quantize_both(x: np.ndarray):
    """GPU and oracle quantisation of the same activation; asserts bit-exactness."""
    a = qx.qx_quantize_act_q8(dev(x))
    q, d, s = oracle.quantize_act_q8(x)
    assert np.array_equal(host(a.q), q), "activation quants differ"
    assert np.array_equal(host(a.d).view(np.uint32), d.view(np.uint32)), "activation scales differ"
    assert np.array_equal(host(a.sum), s), "activation block sums differ"
    return a, q, d, s


# -------------------------------------------------------- activation quant ----

@pytest.mark.parametrize("m,cols", [(1, 32), (1, 896), (1, 4096), (3, 1024), (512, 4096), (1, 14336)])
def test_actq8_bit_exact(m, cols):
    x = synth.activation(m, cols, seed=100 + m + cols)
    quantize_both(x)


def test_actq8_special_values():
    x = np.zeros((1, 256), np.float32)
    x[0, 32] = 1e-44                      # block whose scale underflows to 0
    x[0, 64:96] = np.linspace(-1e30, 1e30, 32)
    x[0, 96] = 127 / 8                    # ties: x/d = k + 1/2 with d = 1/8
    x[0, 97:103] = np.array([2.5, 3.5, -2.5, 0.5, 1.5, -126.5]) / 8
    x[0, 128:160] = -3.0                  # constant block
    x[0, 160:192] = np.float32(1e-30) * np.arange(32)
    # subnormal scales: amax = 178 and 383 times 2^-149 give d = 1 and 3 times
    # 2^-149, so x / d reaches 178 and 127.7; the codes clamp to +-127
    sub = lambda k: np.array([k], np.uint32).view(np.float32)[0]
    x[0, 192:196] = [sub(178), -sub(178), sub(50), -sub(3)]
    x[0, 224:228] = [sub(383), sub(192), sub(190), -sub(383)]
    a, q, d, s = quantize_both(x)
    assert list(q[0, 192:196]) == [127, -127, 50, -3] and list(q[0, 224:228]) == [127, 64, 63, -127]


def subnormal_scale_activation(nblocks: int, seed: int) -> np.ndarray:
    """Blocks whose scale d = amax / 127 is an f32 subnormal, amax swept from the
    smallest subnormal up to 127 * 2^-126 (so d passes through every subnormal
    precision); there x / d can exceed 127 and the clamp decides the code."""
    rng = np.random.default_rng(seed)
    top = int(np.array([np.float32(127.0 * 2.0 ** -126)], np.float32).view(np.uint32)[0])
    first = np.arange(1, nblocks // 2 + 1)
    rest = np.exp(rng.uniform(np.log(nblocks // 2 + 1), np.log(top), nblocks - first.size)).astype(np.int64)
    amax = np.concatenate([first, rest]).astype(np.uint32).view(np.float32)
    x = (rng.uniform(-1, 1, (nblocks, 32)) * amax[:, None]).astype(np.float32)
    col = rng.integers(0, 32, nblocks)
    sign = np.where(rng.integers(0, 2, nblocks) == 1, 1, -1).astype(np.float32)
    x[np.arange(nblocks), col] = sign * amax
    return x.reshape(1, -1)


def test_actq8_subnormal_scales_clamp():
    x = subnormal_scale_activation(4096, seed=8)
    a, q, d, s = quantize_both(x)
    assert np.abs(q.astype(np.int32)).max() == 127
    # the sweep reaches blocks where the clamp binds (and, at its low end, blocks
    # whose scale underflows to 0)
    xb, dd = x.reshape(-1, 32).astype(np.float64), d.reshape(-1).astype(np.float64)
    live = dd > 0
    assert np.any(np.abs(xb[live] / dd[live, None]) >= 127.5) and np.any(~live)


def near_tie_activation(nblocks: int, seed: int) -> np.ndarray:
    """Blocks whose every value sits within 4 ulps of a half-integer multiple of
    the block's scale d = amax / 127: the hardest inputs for the rounding rule."""
    rng = np.random.default_rng(seed)
    x = np.zeros((nblocks, 32), np.float32)
    for b in range(nblocks):
        amax = np.float32(rng.uniform(1e-3, 1e3))
        d = np.float32(amax / np.float32(127))
        k = rng.integers(-127, 127, size=31).astype(np.float64)
        v = ((k + 0.5) * np.float64(d)).astype(np.float32)
        v = (v.view(np.int32) + rng.integers(-4, 5, size=31).astype(np.int32)).view(np.float32)
        v = np.clip(v, -amax, amax)
        x[b, 0] = amax
        x[b, 1:] = v
    return x.reshape(1, -1)


def test_actq8_near_ties_bit_exact():
    quantize_both(near_tie_activation(4096, seed=5))


# 4096 columns: two lanes per block; 2048: four; 896: eight (narrow activations)
@pytest.mark.parametrize("nblocks", [128, 64, 28])
@pytest.mark.parametrize("kind", ["near_ties", "subnormal_scales"])
def test_fused_quantisation_hard_blocks(nblocks, kind):
    """In-kernel quantisation of near-tie and subnormal-scale activations matches
    the standalone kernel (itself bit-exact against the oracle)."""
    fmt, rows = synth.Q8_0, 64
    gen = near_tie_activation if kind == "near_ties" else subnormal_scale_activation
    x = gen(nblocks, seed=6 + nblocks)
    cols = x.shape[1]
    W = dev(synth.weights(fmt, rows, cols, seed=7))
    a, q, d, s = quantize_both(x)
    y_two_step = qx.qx_gemv(fmt, W, rows, cols, a, mode=qx.QX_MODE_W4A8)
    y_fused = qx.qx_gemv(fmt, W, rows, cols, dev(x[0]), mode=qx.QX_MODE_W4A8_FUSED)
    assert np.array_equal(host(y_fused).view(np.uint32), host(y_two_step).view(np.uint32))


# ------------------------------------------------------------------ GEMV ----

SHAPES = {
    synth.Q4_K: [(1, 256), (7, 256), (37, 1024), (300, 4096), (129, 14336), (64, 32768), (1000, 1024)],
    synth.Q6_K: [(1, 256), (5, 512), (37, 1024), (300, 4096), (65, 14336), (9, 2048)],
    synth.Q8_0: [(1, 32), (7, 896), (33, 4096), (301, 896), (5, 8192), (3, 64)],
}
CASES = [(f, r, c) for f, shapes in SHAPES.items() for (r, c) in shapes]
IDS = [f"{synth.NAMES[f]}-{r}x{c}" for f, r, c in CASES]


@pytest.mark.parametrize("fmt,rows,cols", CASES, ids=IDS)
def test_partials_bit_exact(fmt, rows, cols):
    W = synth.weights(fmt, rows, cols, seed=rows * 7 + cols)
    x = synth.activation(1, cols, seed=cols + 3)
    a, q, d, s = quantize_both(x)
    P = qx.qx_gemv_partials(fmt, dev(W), rows, cols, a)
    ref = oracle.partials(fmt, W, rows, cols, q[0])
    got = host(P)
    assert got.shape == ref.shape
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{bad.shape[0]} partials differ, first at {bad[0]}: {got[tuple(bad[0])]} vs {ref[tuple(bad[0])]}"


@pytest.mark.parametrize("fmt,rows,cols", CASES, ids=IDS)
def test_gemv_w4a8(fmt, rows, cols):
    W = synth.weights(fmt, rows, cols, seed=rows * 11 + cols)
    x = synth.activation(1, cols, seed=cols + 5)
    a, q, d, s = quantize_both(x)
    y = qx.qx_gemv(fmt, dev(W), rows, cols, a, mode=qx.QX_MODE_W4A8)
    ref, absdot = oracle.gemv_w4a8(fmt, W, rows, cols, q[0], d[0])
    assert_close(host(y), ref, absdot, f"w4a8 {synth.NAMES[fmt]} {rows}x{cols}")


@pytest.mark.parametrize("fmt,rows,cols", [c for c in CASES if c[2] <= 16384],
                         ids=[i for c, i in zip(CASES, IDS) if c[2] <= 16384])
def test_gemv_f32(fmt, rows, cols):
    W = synth.weights(fmt, rows, cols, seed=rows * 13 + cols)
    x = synth.activation(1, cols, seed=cols + 7)[0]
    y = qx.qx_gemv(fmt, dev(W), rows, cols, dev(x), mode=qx.QX_MODE_F32)
    ref, absdot = oracle.gemv_f32(fmt, W, rows, cols, x)
    assert_close(host(y), ref, absdot, f"f32 {synth.NAMES[fmt]} {rows}x{cols}")


@pytest.mark.parametrize("fmt,rows,cols", CASES, ids=IDS)
def test_gemv_fused_quantisation_is_bit_identical(fmt, rows, cols):
    """In-kernel quantisation gives the same int8 codes, hence the same y, bit for bit."""
    W = dev(synth.weights(fmt, rows, cols, seed=rows * 17 + cols))
    x = synth.activation(1, cols, seed=cols + 9)
    a, q, d, s = quantize_both(x)
    y_two_step = qx.qx_gemv(fmt, W, rows, cols, a, mode=qx.QX_MODE_W4A8)
    y_fused = qx.qx_gemv(fmt, W, rows, cols, dev(x[0]), mode=qx.QX_MODE_W4A8_FUSED)
    y_fused_pdl = qx.qx_gemv(fmt, W, rows, cols, dev(x[0]), mode=qx.QX_MODE_W4A8_FUSED | qx.QX_FLAG_PDL)
    assert np.array_equal(host(y_fused).view(np.uint32), host(y_two_step).view(np.uint32))
    assert np.array_equal(host(y_fused_pdl).view(np.uint32), host(y_two_step).view(np.uint32))


def test_pdl_chain_matches_plain_launches():
    """A chain of PDL launches where each activation is produced by the previous kernel."""
    fmt, rows, cols = synth.Q4_K, 4096, 4096
    Ws = [dev(synth.weights(fmt, rows, cols, seed=70 + i)) for i in range(4)]
    x0 = dev(synth.activation(1, cols, seed=75)[0])
    outs = {}
    for flag in (0, qx.QX_FLAG_PDL):
        x = x0.clone()
        ys = []
        for W in Ws:
            y = qx.qx_gemv(fmt, W, rows, cols, x, mode=qx.QX_MODE_W4A8_FUSED | flag)
            ys.append(y)
            x = y  # the next launch reads what this one wrote
        outs[flag] = [host(t).view(np.uint32) for t in ys]
    for a, b in zip(outs[0], outs[qx.QX_FLAG_PDL]):
        assert np.array_equal(a, b)
    assert qx.qx_device_check() == qx.QX_OK


def test_two_step_chain_reads_after_the_producer():
    """GEMV -> quantise -> GEMV, each activation written by the kernel before.

    The quantisation kernel may become resident while the GEMV before it
    drains and the W4A8 GEMV after it runs under QX_FLAG_PDL; each must still
    read what its predecessor wrote.  The output buffers start out filled with
    a constant, so an early read would change the codes.  Checked eagerly and
    replayed from a CUDA graph against the fused launches, bit for bit."""
    fmt, rows, cols = synth.Q4_K, 4096, 4096
    Ws = [dev(synth.weights(fmt, rows, cols, seed=80 + i)) for i in range(4)]
    x0 = dev(synth.activation(1, cols, seed=85)[0])
    PDL = qx.QX_FLAG_PDL
    ys = [torch.full((rows,), 7.0, dtype=torch.float32, device="cuda") for _ in Ws]
    acts = [qx.ActQ8.empty(1, cols) for _ in Ws]

    def two_step():
        x = x0
        for W, y, a in zip(Ws, ys, acts):
            qx.qx_quantize_act_q8(x, out=a)
            qx.qx_gemv(fmt, W, rows, cols, a, y=y, mode=qx.QX_MODE_W4A8 | PDL)
            x = y

    x, ref = x0, []
    for W in Ws:
        x = qx.qx_gemv(fmt, W, rows, cols, x, mode=qx.QX_MODE_W4A8_FUSED | PDL)
        ref.append(host(x).view(np.uint32))
    two_step()
    for y, r in zip(ys, ref):
        assert np.array_equal(host(y).view(np.uint32), r)
    for y in ys:
        y.fill_(7.0)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            two_step()
    for y in ys:
        y.fill_(7.0)
    torch.cuda.current_stream().wait_stream(stream)
    g.replay()
    torch.cuda.synchronize()
    for y, r in zip(ys, ref):
        assert np.array_equal(host(y).view(np.uint32), r)
    assert qx.qx_device_check() == qx.QX_OK


@pytest.mark.parametrize("fmt,rows,cols", [(synth.Q4_K, 1024, 1024), (synth.Q4_K, 77, 4096), (synth.Q6_K, 65, 14336),
                                           (synth.Q6_K, 300, 1024), (qx.QX_Q6_K_SOA, 129, 1024)])
def test_gemv_f32_small_pdl_launch(fmt, rows, cols):
    """Small f32 launches under programmatic dependent launch run the merged
    variant (8 warps, so that the next launch's CTA fits beside it): the
    same lanes and reduction as the standard kernel, bit for bit (Q4_K rows
    of up to 4096 columns run on the tensor pipe without the flag: both
    against the oracle), and the oracle's tolerance."""
    base = synth.Q6_K if fmt == qx.QX_Q6_K_SOA else fmt
    W = synth.weights(base, rows, cols, seed=rows + 3 * cols)
    x = synth.activation(1, cols, seed=cols + 19)[0]
    Wd = dev(W)
    if fmt == qx.QX_Q6_K_SOA:
        Wd = qx.qx_repack(synth.Q6_K, qx.QX_Q6_K_SOA, Wd, rows, cols)
    y0 = host(qx.qx_gemv(fmt, Wd, rows, cols, dev(x), mode=qx.QX_MODE_F32))
    y1 = host(qx.qx_gemv(fmt, Wd, rows, cols, dev(x), mode=qx.QX_MODE_F32 | qx.QX_FLAG_PDL))
    ref, absdot = oracle.gemv_f32(base, W, rows, cols, x)
    assert_close(y1, ref, absdot, f"f32 pdl {fmt} {rows}x{cols}")
    if fmt == synth.Q4_K:
        # without the flag, Q4_K rows of up to 4096 columns run on the tensor pipe
        assert_close(y0, ref, absdot, f"f32 {fmt} {rows}x{cols}")
    else:
        assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))
    assert qx.qx_device_check() == qx.QX_OK


def test_gemv_zero_and_edge_values():
    """All-zero weights, all-zero activation, a zero-scale super-block."""
    rows, cols = 16, 1024
    for fmt in (synth.Q4_K, synth.Q6_K, synth.Q8_0):
        W = synth.weights(fmt, rows, cols, seed=3)
        x = synth.activation(1, cols, seed=4)
        Wz = np.zeros_like(W)
        y = qx.qx_gemv(fmt, dev(Wz), rows, cols, dev(x[0]), mode=qx.QX_MODE_F32)
        assert np.all(host(y) == 0)
        a = qx.qx_quantize_act_q8(dev(np.zeros_like(x)))
        y = qx.qx_gemv(fmt, dev(W), rows, cols, a, mode=qx.QX_MODE_W4A8)
        assert np.all(host(y) == 0)


def test_gemv_unaligned_base_offset():
    """W and y at a 16-byte offset inside larger allocations; misaligned pointers are refused."""
    fmt, rows, cols = synth.Q8_0, 9, 896
    W = synth.weights(fmt, rows, cols, seed=8)
    x = synth.activation(1, cols, seed=9)[0]
    buf = torch.zeros(W.size + 48, dtype=torch.uint8, device="cuda")
    buf[16:16 + W.size] = dev(W.reshape(-1))
    y = torch.zeros(rows + 8, dtype=torch.float32, device="cuda")
    qx.qx_gemv(fmt, buf[16:16 + W.size], rows, cols, dev(x), y=y[4:4 + rows], mode=qx.QX_MODE_F32)
    ref, absdot = oracle.gemv_f32(fmt, W, rows, cols, x)
    assert_close(host(y[4:4 + rows]), ref, absdot, "offset")
    assert np.all(host(y[:4]) == 0) and np.all(host(y[4 + rows:]) == 0)
    with pytest.raises(qx.QxError) as ei:
        qx.qx_gemv(fmt, buf[8:8 + W.size], rows, cols, dev(x), mode=qx.QX_MODE_F32)
    assert ei.value.status == qx.QX_ERR_ALIGN


# ------------------------------------------------------------- multi GEMV ----

@pytest.mark.parametrize("mode", [qx.QX_MODE_W4A8, qx.QX_MODE_F32])
def test_gemv_multi_matches_separate(mode):
    cols = 1024
    shapes = [(synth.Q4_K, 200), (synth.Q4_K, 37), (synth.Q4_K, 64), (synth.Q8_0, 33), (synth.Q6_K, 5)]
    Ws = [synth.weights(f, r, cols, seed=40 + i) for i, (f, r) in enumerate(shapes)]
    x = synth.activation(1, cols, seed=41)
    if mode == qx.QX_MODE_W4A8:
        a, q, d, s = quantize_both(x)
        xin = a
    else:
        xin = dev(x[0])
    ys = qx.qx_gemv_multi([f for f, _ in shapes], [dev(W) for W in Ws], [r for _, r in shapes], cols, xin,
                          mode=mode)
    for (f, r), W, y in zip(shapes, Ws, ys):
        if mode == qx.QX_MODE_W4A8:
            ref, absdot = oracle.gemv_w4a8(f, W, r, cols, q[0], d[0])
        else:
            ref, absdot = oracle.gemv_f32(f, W, r, cols, x[0])
        assert_close(host(y), ref, absdot, f"multi {synth.NAMES[f]} {r}")


# ------------------------------------------------------------- prefill ----

@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("m,rows,cols", [(1, 70, 1024), (3, 128, 256), (8, 300, 1024), (64, 129, 512),
                                         (65, 256, 4096), (130, 70, 2048)])
def test_prefill_paths(path, m, rows, cols):
    fmt = synth.Q4_K
    W = synth.weights(fmt, rows, cols, seed=50 + m + rows)
    X = synth.activation(m, cols, seed=51 + m)
    a, q, d, s = quantize_both(X)
    Y = qx.qx_gemm_prefill_ex(fmt, dev(W), rows, cols, a, path=path)
    ref, absdot = oracle.gemm_w4a8(fmt, W, rows, cols, q, d)
    assert_close(host(Y).reshape(-1), ref.reshape(-1), absdot.reshape(-1), f"prefill path {path} m={m}")


# The tcgen05 path serves every format; ragged M (partial 128-row tiles), N
# (partial 256-column tiles) and K (a last 64-wide K tile read past the end,
# zero-filled: Q8_0 with cols = 96 or 864).
@pytest.mark.parametrize("fmt,m,rows,cols", [(synth.Q6_K, 16, 300, 1024), (synth.Q6_K, 129, 257, 256),
                                             (synth.Q6_K, 33, 4096, 14336),
                                             (synth.Q8_0, 16, 151, 896), (synth.Q8_0, 40, 33, 96),
                                             (synth.Q8_0, 200, 513, 864),
                                             (synth.Q4_K, 300, 1000, 4864)])
def test_prefill_tcgen05_formats(fmt, m, rows, cols):
    W = synth.weights(fmt, rows, cols, seed=70 + m + rows)
    X = synth.activation(m, cols, seed=71 + m)
    a, q, d, s = quantize_both(X)
    Y = host(qx.qx_gemm_prefill_ex(fmt, dev(W), rows, cols, a, path=3))
    assert np.all(np.isfinite(Y))
    ref, absdot = oracle.gemm_w4a8(fmt, W, rows, cols, q, d)
    assert_close(Y.reshape(-1), ref.reshape(-1), absdot.reshape(-1), f"tcgen05 prefill {synth.NAMES[fmt]} m={m}")


def test_prefill_auto_and_refusals():
    fmt, rows, cols = synth.Q4_K, 96, 1024
    W = dev(synth.weights(fmt, rows, cols, seed=60))
    # automatic path: a GEMV for one row, the small-batch GEMV for 2..40 rows (Q4_K rows the integer
    # tensor path serves; Q8_0 32, Q6_K 24; 16 on the lanes: Q6_K at 1024 columns), tcgen05 above
    W6 = dev(synth.weights(synth.Q6_K, rows, cols, seed=62))
    W8 = dev(synth.weights(synth.Q8_0, rows, cols, seed=63))
    for Wm, f, m, forced in ((W, fmt, 1, 1), (W, fmt, 2, 4), (W, fmt, 16, 4), (W, fmt, 40, 4), (W, fmt, 41, 3),
                             (W, fmt, 200, 3), (W8, synth.Q8_0, 32, 4), (W8, synth.Q8_0, 33, 3),
                             (W6, synth.Q6_K, 15, 4), (W6, synth.Q6_K, 17, 3)):
        a, q, d, s = quantize_both(synth.activation(m, cols, seed=61 + m))
        y_auto = host(qx.qx_gemm_prefill(f, Wm, rows, cols, a))
        y_forced = host(qx.qx_gemm_prefill_ex(f, Wm, rows, cols, a, path=forced))
        assert np.array_equal(y_auto.view(np.uint32), y_forced.view(np.uint32)), f"m={m}"
    with pytest.raises(qx.QxError) as ei:
        qx.qx_gemm_prefill_ex(synth.Q6_K, W6, rows, cols, a, path=2)
    assert ei.value.status == qx.QX_ERR_FMT
    with pytest.raises(qx.QxError) as ei:
        qx.qx_gemm_prefill_ex(fmt, W, rows, cols, a, path=5)
    assert ei.value.status == qx.QX_ERR_ARG


def test_prefill_tcgen05_capturable_on_first_use_and_on_two_streams():
    """The tcgen05 path allocates nothing: its very first call on a fresh shape
    can be captured in a CUDA graph, and two streams can run it at once (no
    shared workspace), each giving the eager result bit for bit."""
    cases = []
    for i, (fmt, rows, cols, m) in enumerate([(synth.Q6_K, 200, 2048, 48), (synth.Q8_0, 136, 864, 40),
                                             (synth.Q4_K, 256, 1024, 33)]):
        W = dev(synth.weights(fmt, rows, cols, seed=66 + i))
        a, q, d, s = quantize_both(synth.activation(m, cols, seed=67 + i))
        cases.append((fmt, W, rows, cols, m, a, q, d))
    stream = torch.cuda.Stream()
    for fmt, W, rows, cols, m, a, q, d in cases:
        Y = torch.full((m, rows), float("nan"), device="cuda")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):  # the first call of this shape and format
            qx.qx_gemm_prefill_ex(fmt, W, rows, cols, a, Y=Y, path=3, stream=stream)
        g.replay()
        y_graph = host(Y).copy()
        y_eager = host(qx.qx_gemm_prefill_ex(fmt, W, rows, cols, a, path=3))
        assert np.array_equal(y_graph.view(np.uint32), y_eager.view(np.uint32)), synth.NAMES[fmt]
        ref, absdot = oracle.gemm_w4a8(fmt, host(W), rows, cols, q, d)
        assert_close(y_eager.reshape(-1), ref.reshape(-1), absdot.reshape(-1), f"captured {synth.NAMES[fmt]}")
    # two streams, interleaved launches of two different problems, many times over
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    (f1, W1, r1, c1, m1, a1, _, _), (f2, W2, r2, c2, m2, a2, _, _) = cases[0], cases[1]
    want1 = host(qx.qx_gemm_prefill_ex(f1, W1, r1, c1, a1, path=3))
    want2 = host(qx.qx_gemm_prefill_ex(f2, W2, r2, c2, a2, path=3))
    Y1 = [torch.empty((m1, r1), device="cuda") for _ in range(8)]
    Y2 = [torch.empty((m2, r2), device="cuda") for _ in range(8)]
    torch.cuda.synchronize()
    for k in range(8):
        qx.qx_gemm_prefill_ex(f1, W1, r1, c1, a1, Y=Y1[k], path=3, stream=s1)
        qx.qx_gemm_prefill_ex(f2, W2, r2, c2, a2, Y=Y2[k], path=3, stream=s2)
    torch.cuda.synchronize()
    for k in range(8):
        assert np.array_equal(host(Y1[k]).view(np.uint32), want1.view(np.uint32))
        assert np.array_equal(host(Y2[k]).view(np.uint32), want2.view(np.uint32))
    assert qx.qx_device_check() == qx.QX_OK


@pytest.mark.parametrize("fmt,cols", [(synth.Q6_K, 512), (synth.Q8_0, 384), (synth.Q4_K, 768)])
def test_prefill_tcgen05_split_last_wave(fmt, cols):
    """More tiles than SMs, the last wave under half full: its tiles run as
    two CTAs each, one per half of the K groups (Q8_0 with three groups: one
    and two), the second handing its partial sums to the first.  Ragged M
    (the second M tile has one 128-row half) and ragged N (the last tile has
    57 rows).  Every row of the split tiles and sampled rows of the others
    against the oracle; a CUDA graph of the call gives the eager bits."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    m = 300                                   # two M tiles of 256
    tiles_n = (sm + 28 + 1) // 2              # sm + 28 (or 29) tiles: a last wave of 28 or 29
    rows = (tiles_n - 1) * 128 + 57
    W = synth.weights(fmt, rows, cols, seed=80 + cols)
    X = synth.activation(m, cols, seed=81 + cols)
    a, q, d, s = quantize_both(X)
    Wd = dev(W)
    Y = host(qx.qx_gemm_prefill_ex(fmt, Wd, rows, cols, a, path=3))
    first_split = (sm // 2) * 128             # tiles sm .. (M tile fastest): N tiles sm / 2 ..
    rng = np.random.default_rng(82)
    wr = np.sort(np.concatenate([np.arange(first_split, rows), rng.choice(first_split, 100, replace=False)]))
    ref, absdot = oracle.gemm_w4a8(fmt, np.ascontiguousarray(W[wr]), len(wr), cols, q, d)
    assert_close(Y[:, wr].reshape(-1), ref.reshape(-1), absdot.reshape(-1), f"split {synth.NAMES[fmt]}")
    stream = torch.cuda.Stream()
    Yg = torch.full((m, rows), float("nan"), device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        qx.qx_gemm_prefill_ex(fmt, Wd, rows, cols, a, Y=Yg, path=3, stream=stream)
    g.replay()
    assert np.array_equal(host(Yg).view(np.uint32), Y.view(np.uint32))
    assert qx.qx_device_check() == qx.QX_OK


@pytest.mark.parametrize("fmt,cols", [(synth.Q4_K, 1280), (synth.Q6_K, 1792), (synth.Q8_0, 512), (synth.Q8_0, 384)])
def test_prefill_tcgen05_split_small_grid(fmt, cols):
    """Twenty tiles (ragged M: 300 rows; ragged N: the last tile has 57 rows),
    at most a quarter of a wave: every tile runs as a cluster of four CTAs
    with shares of 1, 1, 1, 2 (Q4_K, five K groups), 1, 2, 2, 2 (Q6_K, seven)
    and 1 each (Q8_0, four groups), the sums meeting as (a0 + a1) +
    (a2 + a3); with three K groups (Q8_0, 384 columns) as clusters of two.
    Sampled rows and the last tile against the oracle; a CUDA graph of the
    call gives the eager bits."""
    sm = torch.cuda.get_device_properties(0).multi_processor_count
    assert 20 * 4 <= sm
    m, rows = 300, 9 * 128 + 57
    W = synth.weights(fmt, rows, cols, seed=90 + cols)
    X = synth.activation(m, cols, seed=91 + cols)
    a, q, d, s = quantize_both(X)
    Wd = dev(W)
    Y = host(qx.qx_gemm_prefill_ex(fmt, Wd, rows, cols, a, path=3))
    rng = np.random.default_rng(92)
    wr = np.sort(np.concatenate([np.arange(9 * 128, rows), rng.choice(9 * 128, 120, replace=False)]))
    ref, absdot = oracle.gemm_w4a8(fmt, np.ascontiguousarray(W[wr]), len(wr), cols, q, d)
    assert_close(Y[:, wr].reshape(-1), ref.reshape(-1), absdot.reshape(-1), f"small grid {synth.NAMES[fmt]}")
    stream = torch.cuda.Stream()
    Yg = torch.full((m, rows), float("nan"), device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        qx.qx_gemm_prefill_ex(fmt, Wd, rows, cols, a, Y=Yg, path=3, stream=stream)
    g.replay()
    assert np.array_equal(host(Yg).view(np.uint32), Y.view(np.uint32))
    assert qx.qx_device_check() == qx.QX_OK


@pytest.mark.parametrize("path", [2, 3])
def test_prefill_full_size_sampled(path):
    """X [512, 4096] against Q4_K [14336, 4096]: sampled rows of X and of W against the oracle."""
    fmt, rows, cols, m = synth.Q4_K, 14336, 4096, 512
    W = synth.weights(fmt, rows, cols, seed=63)
    X = synth.activation(m, cols, seed=64)
    a, q, d, s = quantize_both(X)
    Y = host(qx.qx_gemm_prefill_ex(fmt, dev(W), rows, cols, a, path=path))
    rng = np.random.default_rng(65)
    xr = np.sort(rng.choice(m, 6, replace=False))
    wr = np.sort(np.concatenate([rng.choice(rows, 250, replace=False), [0, rows - 1]]))
    ref, absdot = oracle.gemm_w4a8(fmt, np.ascontiguousarray(W[wr]), len(wr), cols, q[xr], d[xr])
    assert_close(Y[np.ix_(xr, wr)].reshape(-1), ref.reshape(-1), absdot.reshape(-1), f"prefill full size path {path}")


# ------------------------------------------------- binding size checks ----

def test_binding_refuses_short_buffers():
    """The binding checks every tensor's byte count before passing a raw pointer."""
    W = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros(256, device="cuda")
    with pytest.raises(ValueError):
        qx.qx_gemv(qx.QX_Q4_K, W, 5, 256, x, mode=qx.QX_MODE_F32)                  # W holds 4 rows
    with pytest.raises(ValueError):
        qx.qx_gemv(qx.QX_Q4_K, W, 4, 256, x, y=torch.zeros(3, device="cuda"), mode=qx.QX_MODE_F32)
    with pytest.raises(ValueError):
        qx.qx_gemv(qx.QX_Q4_K, W, 4, 256, x[:128], mode=qx.QX_MODE_W4A8_FUSED)      # x too short
    with pytest.raises(ValueError):
        qx.qx_repack(qx.QX_Q6_K, qx.QX_Q6_K_SOA, torch.zeros(210, dtype=torch.uint8, device="cuda"), 1, 256,
                     out=torch.zeros(16, dtype=torch.uint8, device="cuda"))


# ------------------------------------------------------- mma rate probe ----

def test_mma_rate_probe():
    """The measured mma.sync rates are finite, positive and ordered (f16 above int8 on GB300)."""
    int8 = qx.qx_debug_mma_rate(0)
    f16 = qx.qx_debug_mma_rate(1)
    assert 1e12 < int8 < 1e16 and 1e12 < f16 < 1e16
    assert f16 > int8


# ---------------------------------------------------- device error word ----

def test_bounded_wait_reports_timeout_and_recovers():
    assert qx.qx_device_check() == qx.QX_OK
    qx.qx_debug_timeout_probe(5_000_000)  # 5 ms on a barrier nothing completes
    assert qx.qx_device_check() == qx.QX_ERR_DEVICE_TIMEOUT
    assert qx.qx_device_check() == qx.QX_OK  # cleared, context still usable
    fmt, rows, cols = synth.Q4_K, 8, 256
    W = synth.weights(fmt, rows, cols, seed=60)
    x = synth.activation(1, cols, seed=61)[0]
    y = qx.qx_gemv(fmt, dev(W), rows, cols, dev(x), mode=qx.QX_MODE_F32)
    ref, absdot = oracle.gemv_f32(fmt, W, rows, cols, x)
    assert_close(host(y), ref, absdot, "after probe")


# ------------------------------------------------------------ width limits ----

def test_wide_rows_take_a_variant_that_fits():
    """A >= 128 MB Q6_K W4A8 launch normally takes the merged variant, whose
    lanes cover 28672 columns: 32768-column rows take the standard kernel;
    the automatic prefill path leaves the small-batch path for rows wider
    than its lanes; the documented limits refuse wider rows by name."""
    fmt, rows, cols = synth.Q6_K, 5120, 32768          # 137.6 MB of weights
    W = synth.weights(fmt, rows, cols, seed=120)
    x = synth.activation(1, cols, seed=121)
    a, q, d, s = quantize_both(x)
    Wd = dev(W)
    y = qx.qx_gemv(fmt, Wd, rows, cols, dev(x[0]), mode=qx.QX_MODE_W4A8_FUSED | qx.QX_FLAG_PDL)
    y2 = qx.qx_gemv(fmt, Wd, rows, cols, a, mode=qx.QX_MODE_W4A8)
    assert np.array_equal(host(y).view(np.uint32), host(y2).view(np.uint32))
    sel = np.unique(np.concatenate([np.random.default_rng(122).choice(rows, 64, replace=False), [0, rows - 1]]))
    ref, absdot = oracle.gemv_w4a8(fmt, np.ascontiguousarray(W[sel]), len(sel), cols, q[0], d[0])
    assert_close(host(y)[sel], ref, absdot, "wide merged-size Q6_K")
    del Wd, W
    # prefill: too wide for the small-batch lanes -> one GEMV per row of X
    for m, c in ((4, 32768), (8, 16384)):
        f, r = synth.Q4_K, 64
        Wq = dev(synth.weights(f, r, c, seed=123 + m))
        X = qx.qx_quantize_act_q8(dev(synth.activation(m, c, seed=124 + m)))
        y_auto = host(qx.qx_gemm_prefill(f, Wq, r, c, X))
        y_rows = host(qx.qx_gemm_prefill_ex(f, Wq, r, c, X, path=1))
        assert np.array_equal(y_auto.view(np.uint32), y_rows.view(np.uint32))
        with pytest.raises(qx.QxError) as ei:
            qx.qx_gemm_prefill_ex(f, Wq, r, c, X, path=4)
        assert ei.value.status == qx.QX_ERR_SHAPE
    # documented limits: f32 Q4_K up to 24576 columns, Q8_0 up to 8192
    for f, c_ok, c_bad, mode in ((synth.Q4_K, 24576, 24832, qx.QX_MODE_F32), (synth.Q8_0, 8192, 8224, qx.QX_MODE_F32),
                                 (synth.Q8_0, 8192, 8224, qx.QX_MODE_W4A8_FUSED)):
        for c, ok in ((c_ok, True), (c_bad, False)):
            Wc = dev(synth.weights(f, 3, c, seed=125))
            xc = dev(synth.activation(1, c, seed=126)[0])
            if ok:
                qx.qx_gemv(f, Wc, 3, c, xc, mode=mode)
            else:
                with pytest.raises(qx.QxError) as ei:
                    qx.qx_gemv(f, Wc, 3, c, xc, mode=mode)
                assert ei.value.status == qx.QX_ERR_SHAPE
    assert qx.qx_device_check() == qx.QX_OK
