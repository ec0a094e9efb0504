"""Pins of the CPU oracle against facts that do not come from the oracle itself.

* fp16 decode: every one of the 65,536 bit patterns against numpy's float16.
* Block layouts: hand-built blocks whose dequantised values were written by
  hand from the closed forms (tests/golden/*.txt), plus bijection properties
  (every quant field moves exactly one element, every element is reached once)
  and an exhaustive sweep of every 6-bit Q4_K scale and min field.
* Activation quantisation: zero block, one-hot block, exact multiples of a
  power-of-two scale, round-half-to-even ties, tiny scales, brute force.
* GEMV: unit-vector probes (y(e_i) is column i of the dequantised matrix),
  a dense f64 matmul of the dequantised matrix, the W4A8 result against the
  f64 dot with the dequantised activation, and integer partials against the
  dequantised unit-scale weights.
"""
import numpy as np
import pytest

import oracle
import synth
from tests.golden_blocks import load_cases

FMTS = [synth.Q4_K, synth.Q6_K, synth.Q8_0]


# ---------------------------------------------------------------- fp16 ----

def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    expect = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(h)) for h in bits])
    nan = np.isnan(expect)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], expect[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(expect[~nan]))


# ------------------------------------------------------ block layouts ----

@pytest.mark.parametrize("fname,fmt", [("q4_k_blocks.txt", synth.Q4_K),
                                       ("q6_k_blocks.txt", synth.Q6_K),
                                       ("q8_0_blocks.txt", synth.Q8_0)])
def test_dequant_hand_built_blocks(fname, fmt):
    cases = load_cases(fname, synth.BLOCK_BYTES[fmt], synth.BLOCK_WEIGHTS[fmt])
    assert len(cases) >= 5
    for name, row, exp, cols in cases:
        got = oracle.dequant(fmt, row, cols)[0]
        bad = np.nonzero(got != exp)[0]
        assert bad.size == 0, f"{fname}:{name}: elements {bad[:8]} got {got[bad[:8]]} want {exp[bad[:8]]}"


def _q4k_block(d=0x3C00, dmin=0, scales=None, qs=None):
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.array([d], dtype="<u2").view(np.uint8)
    b[2:4] = np.array([dmin], dtype="<u2").view(np.uint8)
    if scales is not None:
        b[4:16] = scales
    if qs is not None:
        b[16:144] = qs
    return b


def test_q4k_every_scale_and_min_value():
    """Every 6-bit value of every sc_j and m_j field decodes to itself.

    The fields are placed with the GGUF packing written out here from its
    prose description; each (j, value) is checked on its own, so a wrong shift
    or a swapped scale/min fails for some value."""
    ones = np.full(128, 0x11, dtype=np.uint8)  # every quant = 1
    for j in range(8):
        for v in range(64):
            for kind in ("sc", "m"):
                s = np.zeros(12, dtype=np.uint8)
                if j < 4:
                    s[j if kind == "sc" else j + 4] = v
                else:
                    lo, hi = v & 15, v >> 4
                    if kind == "sc":
                        s[j + 4] = lo
                        s[j - 4] = hi << 6
                    else:
                        s[j + 4] = lo << 4
                        s[j] = hi << 6
                if kind == "sc":
                    blk = _q4k_block(d=0x3C00, dmin=0, scales=s, qs=ones)
                    want = np.zeros(256)
                    want[32 * j:32 * j + 32] = v
                else:
                    blk = _q4k_block(d=0, dmin=0x3C00, scales=s, qs=ones)
                    want = np.zeros(256)
                    want[32 * j:32 * j + 32] = -v
                got = oracle.dequant(synth.Q4_K, blk, 256)[0]
                assert np.array_equal(got, want), (j, v, kind)


def test_q4k_quant_nibbles_are_a_bijection():
    """Each of the 256 nibbles of qs moves exactly one element; all 256 elements are hit."""
    s = np.array([1, 1, 1, 1, 0, 0, 0, 0, 0x01, 0x01, 0x01, 0x01], dtype=np.uint8)  # sc_j = 1, m_j = 0
    hit = []
    for byte in range(128):
        for shift in (0, 4):
            qs = np.zeros(128, dtype=np.uint8)
            qs[byte] = 5 << shift
            w = oracle.dequant(synth.Q4_K, _q4k_block(scales=s, qs=qs), 256)[0]
            nz = np.nonzero(w)[0]
            assert nz.size == 1 and w[nz[0]] == 5, (byte, shift, nz)
            hit.append(nz[0])
    assert sorted(hit) == list(range(256))


def _q6k_block(d=0x3C00, scales=1, ql=None, qh=None):
    b = np.zeros(210, dtype=np.uint8)
    if ql is not None:
        b[0:128] = ql
    if qh is not None:
        b[128:192] = qh
    b[192:208] = np.array(scales, dtype=np.int8).view(np.uint8) if np.ndim(scales) else np.uint8(scales)
    b[208:210] = np.array([d], dtype="<u2").view(np.uint8)
    return b


def test_q6k_fields_are_bijections_and_combine():
    """Each ql nibble and each 2-bit qh field moves exactly one element, and the
    element a qh field moves is the one whose low bits come from the matching
    ql nibble (together they make q = 63 -> w = 31)."""
    base = -32.0
    lo_map, hi_map = {}, {}
    for byte in range(128):
        for shift in (0, 4):
            ql = np.zeros(128, dtype=np.uint8)
            ql[byte] = 1 << shift
            w = oracle.dequant(synth.Q6_K, _q6k_block(ql=ql), 256)[0]
            nz = np.nonzero(w != base)[0]
            assert nz.size == 1 and w[nz[0]] == -31.0, (byte, shift, nz)
            lo_map[(byte, shift)] = nz[0]
    for byte in range(64):
        for shift in (0, 2, 4, 6):
            qh = np.zeros(64, dtype=np.uint8)
            qh[byte] = 1 << shift
            w = oracle.dequant(synth.Q6_K, _q6k_block(qh=qh), 256)[0]
            nz = np.nonzero(w != base)[0]
            assert nz.size == 1 and w[nz[0]] == -16.0, (byte, shift, nz)
            hi_map[(byte, shift)] = nz[0]
    assert sorted(lo_map.values()) == list(range(256))
    assert sorted(hi_map.values()) == list(range(256))
    inv_lo = {e: k for k, e in lo_map.items()}
    for (byte, shift), e in hi_map.items():
        lb, ls = inv_lo[e]
        ql = np.zeros(128, dtype=np.uint8)
        ql[lb] = 15 << ls
        qh = np.zeros(64, dtype=np.uint8)
        qh[byte] = 3 << shift
        w = oracle.dequant(synth.Q6_K, _q6k_block(ql=ql, qh=qh), 256)[0]
        assert w[e] == 31.0 and np.all(np.delete(w, e) == base)


def test_q6k_scale_groups_of_16():
    for g in range(16):
        sc = np.zeros(16, dtype=np.int8)
        sc[g] = -3
        w = oracle.dequant(synth.Q6_K, _q6k_block(scales=sc), 256)[0]
        want = np.zeros(256)
        want[16 * g:16 * g + 16] = 96.0  # (0 - 32) * -3
        assert np.array_equal(w, want), g


def test_zero_and_zero_scale_blocks():
    for fmt in FMTS:
        bb, bw = synth.BLOCK_BYTES[fmt], synth.BLOCK_WEIGHTS[fmt]
        assert np.all(oracle.dequant(fmt, np.zeros(bb, np.uint8), bw) == 0.0)
        # d = 0 (and dmin = 0) with random quants -> all zero
        W = synth.weights(fmt, 1, bw, seed=5)[0].copy()
        if fmt == synth.Q4_K:
            W[0:4] = 0
        elif fmt == synth.Q6_K:
            W[208:210] = 0
        else:
            W[0:2] = 0
        assert np.all(oracle.dequant(fmt, W, bw) == 0.0)


# ------------------------------------------------- activation quantise ----

def test_quant_zero_block():
    q, d, s = oracle.quantize_act_q8(np.zeros((1, 64), np.float32))
    assert np.all(q == 0) and np.all(d == 0) and np.all(s == 0)


def test_quant_one_hot():
    for v in (3.7, -0.001, 1e30, -7.0e-30):
        x = np.zeros((1, 32), np.float32)
        x[0, 11] = v
        q, d, s = oracle.quantize_act_q8(x)
        want = np.zeros(32, np.int8)
        want[11] = 127 if v > 0 else -127
        assert np.array_equal(q[0], want)
        assert d[0, 0] == np.float32(abs(np.float32(v))) / np.float32(127)
        assert s[0, 0] == want.sum()


def test_quant_exact_multiples_and_ties():
    # amax = 127/8 -> d = 1/8 exactly, so x = k/8 quantises to k.
    rng = np.random.default_rng(1)
    k = rng.integers(-127, 128, size=32)
    k[7] = 127
    x = (k / 8.0).astype(np.float32)[None]
    q, d, s = oracle.quantize_act_q8(x)
    assert d[0, 0] == np.float32(0.125)
    assert np.array_equal(q[0].astype(int), k) and s[0, 0] == k.sum()
    # ties go to even: x/d = 2.5 -> 2, 3.5 -> 4, -2.5 -> -2, 0.5 -> 0, 1.5 -> 2, -126.5 -> -126
    t = np.zeros(32, np.float32)
    t[0] = 127 / 8
    t[1:7] = np.array([2.5, 3.5, -2.5, 0.5, 1.5, -126.5]) / 8
    q, d, s = oracle.quantize_act_q8(t[None])
    assert list(q[0, :7]) == [127, 2, 4, -2, 0, 2, -126]


def test_quant_divides_by_the_scale():
    """q = rne(x / d) with a correctly rounded f32 quotient, not x * (1/d).

    Each pair (amax, x), given as f32 bit patterns, sits next to a rounding
    boundary where the two rules give different integers; the expected q is
    the division rule's (found by search with numpy float32 arithmetic)."""
    cases = [(1057935115, 1036675064, 22), (1064262554, 1010101904, 1),
             (1076999152, 1073012157, 88), (1064897509, 1052910458, 50)]
    for amax_bits, x_bits, want in cases:
        x = np.zeros((1, 32), np.float32)
        x[0, 0] = np.array([amax_bits], np.uint32).view(np.float32)[0]
        x[0, 1] = np.array([x_bits], np.uint32).view(np.float32)[0]
        q, d, s = oracle.quantize_act_q8(x)
        assert q[0, 0] == 127 and q[0, 1] == want, (amax_bits, x_bits, q[0, :2])


def test_quant_tiny_scale_underflows_to_zero():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = np.float32(1e-44)  # subnormal; amax/127 underflows to 0
    q, d, s = oracle.quantize_act_q8(x)
    assert d[0, 0] == 0 and np.all(q == 0) and s[0, 0] == 0


def test_quant_clamps_codes_of_subnormal_scales():
    """Where d = fl(amax / 127) is an f32 subnormal it can be far below amax / 127,
    so x / d exceeds 127 and the clamp to [-127, 127] decides the code.

    Values worked by hand in units of u = 2^-149 (the smallest subnormal):
      block 0: amax = 178u -> amax / 127 = 1.40u rounds to d = 1u;
               x = 178u, -178u, 50u, -3u -> 178, -178 clamp to 127, -127; 50, -3 stay.
      block 1: amax = 383u -> 3.016u rounds to d = 3u;
               x = 383u -> 127.67 -> 128 clamps to 127; 192u -> 64; 190u -> 63.33 -> 63;
               -383u -> -128 clamps to -127.
    """
    u = lambda k: np.array([k], np.uint32).view(np.float32)[0] if k >= 0 else -u(-k)
    x = np.zeros((1, 64), np.float32)
    x[0, 0:4] = [u(178), u(-178), u(50), u(-3)]
    x[0, 32:36] = [u(383), u(192), u(190), u(-383)]
    q, d, s = oracle.quantize_act_q8(x)
    assert list(d[0].view(np.uint32)) == [1, 3]
    assert list(q[0, 0:4]) == [127, -127, 50, -3] and np.all(q[0, 4:32] == 0)
    assert list(q[0, 32:36]) == [127, 64, 63, -127] and np.all(q[0, 36:] == 0)
    assert list(s[0]) == [47, 127]


def test_quant_rejects_non_finite():
    x = np.zeros((1, 32), np.float32)
    x[0, 3] = np.inf
    with pytest.raises(RuntimeError):
        oracle.quantize_act_q8(x)


def test_quant_brute_force():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((4, 1024)) * np.exp(rng.uniform(-20, 20, (4, 1)))).astype(np.float32)
    q, d, s = oracle.quantize_act_q8(x)
    xb = x.reshape(-1, 32)
    amax = np.abs(xb).max(axis=1)
    assert np.array_equal(d.reshape(-1), (amax / np.float32(127)).astype(np.float32))
    dd = d.reshape(-1, 1)
    qq = q.reshape(-1, 32).astype(np.float64)
    # nearest integer to the f32 quotient, ties to even
    assert np.array_equal(qq, np.rint((xb / dd).astype(np.float32)).astype(np.float64))
    assert np.all(np.abs(qq - xb.astype(np.float64) / dd.astype(np.float64)) <= 0.5 + 1e-5)
    assert np.all(np.abs(qq).max(axis=1) == 127)
    assert np.array_equal(s.reshape(-1), qq.sum(axis=1).astype(np.int32))


# -------------------------------------------------------------- GEMV ----

TINY = {synth.Q4_K: (3, 512), synth.Q6_K: (3, 512), synth.Q8_0: (4, 96)}


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_unit_vectors_give_dequantised_columns(fmt):
    rows, cols = TINY[fmt]
    W = synth.weights(fmt, rows, cols, seed=11)
    Wd = oracle.dequant(fmt, W, cols)
    for i in range(cols):
        e = np.zeros(cols, np.float32)
        e[i] = 1.0
        y, _ = oracle.gemv_f32(fmt, W, rows, cols, e, threads=1)
        assert np.array_equal(y, Wd[:, i]), i


@pytest.mark.parametrize("fmt", FMTS)
def test_gemv_f32_matches_dense_matmul(fmt):
    rows, cols = 37, 1024
    W = synth.weights(fmt, rows, cols, seed=12)
    x = synth.activation(1, cols, seed=13)[0]
    y, a = oracle.gemv_f32(fmt, W, rows, cols, x)
    Wd = oracle.dequant(fmt, W, cols)
    ref = Wd @ x.astype(np.float64)
    assert np.all(np.abs(y - ref) <= 1e-12 * np.abs(Wd * x).sum(axis=1))
    assert np.allclose(a, np.abs(Wd * x.astype(np.float64)).sum(axis=1), rtol=1e-12, atol=0)


@pytest.mark.parametrize("fmt", FMTS)
def test_w4a8_equals_dot_with_dequantised_activation(fmt):
    rows, cols = 29, 1024
    W = synth.weights(fmt, rows, cols, seed=14)
    x = synth.activation(1, cols, seed=15)
    q, d, _ = oracle.quantize_act_q8(x)
    y, a = oracle.gemv_w4a8(fmt, W, rows, cols, q[0], d[0])
    xprime = np.repeat(d[0].astype(np.float64), 32) * q[0].astype(np.float64)
    ref, aref = oracle.gemv_f64x(fmt, W, rows, cols, xprime)
    assert np.all(np.abs(y - ref) <= 1e-12 * aref)
    assert np.allclose(a, aref, rtol=1e-12, atol=0)


def _unit_scale(fmt, W):
    """Copy of W with every block's scales set so that w equals the integer quant."""
    W = W.copy()
    bb = synth.BLOCK_BYTES[fmt]
    B = W.reshape(-1, bb)
    if fmt == synth.Q4_K:
        B[:, 0:2] = (0x00, 0x3C)  # d = 1
        B[:, 2:4] = 0             # dmin = 0
        B[:, 4:16] = (1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1)  # sc_j = 1, m_j = 0
    elif fmt == synth.Q6_K:
        B[:, 192:208] = 1
        B[:, 208:210] = (0x00, 0x3C)
    else:
        B[:, 0:2] = (0x00, 0x3C)
    return W


@pytest.mark.parametrize("fmt", FMTS)
def test_partials_are_integer_dots_of_unit_scale_weights(fmt):
    rows, cols = 9, 768
    W = synth.weights(fmt, rows, cols, seed=16)
    x = synth.activation(1, cols, seed=17)
    q, _, _ = oracle.quantize_act_q8(x)
    P = oracle.partials(fmt, W, rows, cols, q[0])
    Wu = oracle.dequant(fmt, _unit_scale(fmt, W), cols).astype(np.int64)
    if fmt == synth.Q4_K:
        pass  # w = q in [0, 15]
    g = oracle.partial_group(fmt)
    ref = (Wu * q[0].astype(np.int64)).reshape(rows, cols // g, g).sum(axis=2)
    assert np.array_equal(P.astype(np.int64), ref)
    # partials do not depend on the scales
    assert np.array_equal(oracle.partials(fmt, _unit_scale(fmt, W), rows, cols, q[0]), P)


def test_zero_activation_padding_equals_truncation():
    """Q4_K rows of 1024 with activation columns 896.. zero give the 896-column product."""
    rows = 16
    W = synth.q4_k_weights(rows, 1024, seed=18)
    x = synth.activation(1, 1024, seed=19, valid_cols=896)[0]
    y, _ = oracle.gemv_f32(synth.Q4_K, W, rows, 1024, x)
    Wd = oracle.dequant(synth.Q4_K, W, 1024)
    ref = Wd[:, :896] @ x[:896].astype(np.float64)
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * np.abs(Wd).sum())
    q, d, _ = oracle.quantize_act_q8(x[None])
    assert np.all(q[0, 896:] == 0) and np.all(d[0, 28:] == 0)


def test_prefill_rows_are_independent_gemvs():
    rows, cols, m = 21, 512, 5
    W = synth.q4_k_weights(rows, cols, seed=20)
    X = synth.activation(m, cols, seed=21)
    q, d, _ = oracle.quantize_act_q8(X)
    Y, A = oracle.gemm_w4a8(synth.Q4_K, W, rows, cols, q, d)
    for i in range(m):
        y, a = oracle.gemv_w4a8(synth.Q4_K, W, rows, cols, q[i], d[i])
        assert np.array_equal(Y[i], y) and np.array_equal(A[i], a)


def test_row_bytes_and_shape_errors():
    assert oracle.row_bytes(synth.Q4_K, 4096) == 16 * 144
    assert oracle.row_bytes(synth.Q6_K, 14336) == 56 * 210
    assert oracle.row_bytes(synth.Q8_0, 896) == 28 * 34
    assert oracle.row_bytes(synth.Q4_K, 896) == -1
    assert oracle.row_bytes(99, 256) == -1
