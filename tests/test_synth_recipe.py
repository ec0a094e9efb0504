"""The seeded inputs follow the recipe they are documented with: field
offsets, value ranges and distributions of the block formats, activations,
determinism per seed.  (synth.py holds no arithmetic of the method; these
checks read only the bytes it lays out.)"""
import numpy as np

import synth

N_ROWS, COLS = 64, 4096


def _f16(col2: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(col2).view("<f2").astype(np.float64).ravel()


def test_row_sizes():
    for fmt, rows, cols in ((synth.Q4_K, 3, 512), (synth.Q6_K, 2, 768), (synth.Q8_0, 5, 96)):
        W = synth.weights(fmt, rows, cols, seed=1)
        assert W.dtype == np.uint8 and W.shape == (rows, synth.row_bytes(fmt, cols))


def test_q4_k_scales_are_half_normal_and_fields_uniform():
    blk = synth.weights(synth.Q4_K, N_ROWS, COLS, seed=3).reshape(-1, 144)
    for off in (0, 2):  # d, dmin: f16 of |N(0, 1e-3)|
        v = _f16(blk[:, off:off + 2])
        assert np.all(v >= 0) and np.all(np.isfinite(v))
        assert abs(np.median(v) / 1e-3 - 0.6745) < 0.05       # median of |N(0, 1)|
        sub = np.mean(v < 2.0 ** -14)                          # subnormal fp16 scales occur
        assert 0.02 < sub < 0.08                               # P(|N(0,1)| < 0.061) = 0.049
    body = blk[:, 4:144]
    counts = np.bincount(body.ravel(), minlength=256)
    assert counts.min() > 0.8 * body.size / 256 and counts.max() < 1.2 * body.size / 256


def test_q6_k_fields():
    blk = synth.weights(synth.Q6_K, N_ROWS, COLS, seed=4).reshape(-1, 210)
    sc = blk[:, 192:208].view(np.int8)
    assert sc.min() == -32 and sc.max() == 31 and len(np.unique(sc)) == 64
    d = _f16(blk[:, 208:210])
    assert np.all(d >= 0) and abs(np.median(d) / 1e-3 - 0.6745) < 0.05
    ql_qh = blk[:, :192]
    counts = np.bincount(ql_qh.ravel(), minlength=256)
    assert counts.min() > 0.8 * ql_qh.size / 256


def test_q8_0_fields():
    blk = synth.weights(synth.Q8_0, N_ROWS, 1024, seed=5).reshape(-1, 34)
    q = blk[:, 2:].view(np.int8)
    assert q.min() == -127 and q.max() == 127          # -128 never drawn
    d = _f16(blk[:, 0:2])
    assert np.all(d >= 0) and abs(np.median(d) / 2e-3 - 0.6745) < 0.05


def test_activation_and_padding():
    x = synth.activation(4, 1024, seed=6, valid_cols=896)
    assert x.dtype == np.float32 and x.shape == (4, 1024)
    assert np.all(x[:, 896:] == 0)
    v = x[:, :896].astype(np.float64)
    assert abs(v.mean()) < 0.1 and abs(v.std() - 1.0) < 0.05


def test_seeds_are_deterministic_and_distinct():
    a = synth.weights(synth.Q4_K, 4, 512, seed=7)
    assert np.array_equal(a, synth.weights(synth.Q4_K, 4, 512, seed=7))
    assert not np.array_equal(a, synth.weights(synth.Q4_K, 4, 512, seed=8))
    seeds = {synth.seed_for(w, layer, p) for w in range(5) for layer in range(32) for p in range(8)}
    assert len(seeds) == 5 * 32 * 8
