"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the bench.

This module holds no arithmetic of the quantised GEMV itself: it only lays
random bytes out at the field offsets of the GGUF block formats.  Neither the
oracle nor the CUDA path is imported here, and both consume exactly the bytes
produced here.

Value distributions (the decode workloads of the llambda.lisp README,
"Features & Architecture": Q4_K_M / Q6_K tensors; and of the llamay
"Backends and hardware" page, "Repacking is a per-device decision now": Q8_0):

* Q4_K super-block (256 weights, 144 bytes): fp16 ``d`` and ``dmin`` drawn as
  f16(|N(0, 1e-3)|), 12 bytes of packed 6-bit scales/mins, 128 bytes of 4-bit
  quants.  Under the GGUF packing every bit of the 12 scale bytes belongs to
  exactly one 6-bit scale or min, and every bit of the 128 quant bytes to one
  4-bit quant, so uniform random bytes are exactly "scales and mins uniform in
  [0, 63], quants uniform in [0, 15]" -- no packing step is needed.
* Q6_K super-block (256 weights, 210 bytes): ``ql[128]`` and ``qh[64]`` uniform
  random bytes (each 6-bit quant is 4 low bits from ``ql`` and 2 high bits from
  ``qh``, so the quants are uniform in [0, 63]), ``scales[16]`` int8 uniform in
  [-32, 31], fp16 ``d`` = f16(|N(0, 1e-3)|) stored last.
* Q8_0 block (32 weights, 34 bytes): fp16 ``d`` = f16(|N(0, 2e-3)|), then 32
  int8 uniform in [-127, 127].
* Activations: f32 N(0, 1).

fp16 values are produced by numpy's float64 -> float16 conversion (round to
nearest even); |N(0, sigma)| with sigma = 1e-3 falls below the smallest normal
fp16 (2**-14) a few percent of the time, so subnormal scales occur.
"""
from __future__ import annotations

import numpy as np

# GGML type ids, used as format tags throughout (a naming convention only).
Q8_0 = 8
Q4_K = 12
Q6_K = 14

BLOCK_WEIGHTS = {Q8_0: 32, Q4_K: 256, Q6_K: 256}
BLOCK_BYTES = {Q8_0: 34, Q4_K: 144, Q6_K: 210}
NAMES = {Q8_0: "q8_0", Q4_K: "q4_k", Q6_K: "q6_k"}


def row_bytes(fmt: int, cols: int) -> int:
    assert cols % BLOCK_WEIGHTS[fmt] == 0, (fmt, cols)
    return cols // BLOCK_WEIGHTS[fmt] * BLOCK_BYTES[fmt]


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _uniform_bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    return np.frombuffer(rng.bytes(n), dtype=np.uint8).copy()


def _f16_abs_normal(rng: np.random.Generator, n: int, sigma: float) -> np.ndarray:
    """Little-endian fp16 bit patterns of |N(0, sigma)|, as a [n, 2] uint8 array."""
    v = np.abs(rng.standard_normal(n)) * sigma
    return v.astype("<f2").view(np.uint8).reshape(n, 2)


def q4_k_weights(rows: int, cols: int, seed: int, sigma: float = 1e-3) -> np.ndarray:
    """[rows, cols/256*144] uint8: d(2) dmin(2) scales(12) qs(128) per block."""
    nb = rows * (cols // 256)
    rng = _rng(seed)
    blk = _uniform_bytes(rng, nb * 144).reshape(nb, 144)
    blk[:, 0:2] = _f16_abs_normal(rng, nb, sigma)
    blk[:, 2:4] = _f16_abs_normal(rng, nb, sigma)
    return blk.reshape(rows, row_bytes(Q4_K, cols))


def q6_k_weights(rows: int, cols: int, seed: int, sigma: float = 1e-3) -> np.ndarray:
    """[rows, cols/256*210] uint8: ql(128) qh(64) scales(16, int8) d(2) per block."""
    nb = rows * (cols // 256)
    rng = _rng(seed)
    blk = _uniform_bytes(rng, nb * 210).reshape(nb, 210)
    blk[:, 192:208] = rng.integers(-32, 32, size=(nb, 16), dtype=np.int8).view(np.uint8)
    blk[:, 208:210] = _f16_abs_normal(rng, nb, sigma)
    return blk.reshape(rows, row_bytes(Q6_K, cols))


def q8_0_weights(rows: int, cols: int, seed: int, sigma: float = 2e-3) -> np.ndarray:
    """[rows, cols/32*34] uint8: d(2) qs(32, int8) per block."""
    nb = rows * (cols // 32)
    rng = _rng(seed)
    blk = np.empty((nb, 34), dtype=np.uint8)
    blk[:, 2:34] = rng.integers(-127, 128, size=(nb, 32), dtype=np.int8).view(np.uint8)
    blk[:, 0:2] = _f16_abs_normal(rng, nb, sigma)
    return blk.reshape(rows, row_bytes(Q8_0, cols))


def weights(fmt: int, rows: int, cols: int, seed: int) -> np.ndarray:
    if fmt == Q4_K:
        return q4_k_weights(rows, cols, seed)
    if fmt == Q6_K:
        return q6_k_weights(rows, cols, seed)
    if fmt == Q8_0:
        return q8_0_weights(rows, cols, seed)
    raise ValueError(f"unknown format {fmt}")


def activation(m: int, cols: int, seed: int, valid_cols: int | None = None) -> np.ndarray:
    """f32 N(0, 1) activations [m, cols]; columns at and past ``valid_cols`` are 0.

    Zeroing the trailing columns is how a logical width that is not a whole
    number of super-blocks (Qwen2-0.5B's 896 for Q4_K) is carried in a padded
    row: a zero activation contributes exactly 0 in both modes.
    """
    x = _rng(seed).standard_normal((m, cols)).astype(np.float32)
    if valid_cols is not None:
        x[:, valid_cols:] = 0.0
    return x


# ---------------------------------------------------------------------------
# Workload shapes (sizes only).

# Llama-3.1-8B decode layer, Q4_K_M mix: (name, fmt, rows, cols).  q/k/v share
# one activation, gate/up share another.
LLAMA8B_LAYER = [
    ("q", Q4_K, 4096, 4096), ("k", Q4_K, 1024, 4096), ("v", Q4_K, 1024, 4096),
    ("o", Q4_K, 4096, 4096),
    ("gate", Q4_K, 14336, 4096), ("up", Q4_K, 14336, 4096),
    ("down", Q6_K, 4096, 14336),
]
LLAMA8B_GROUPS = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
LLAMA8B_LAYERS = 32

# Qwen2-0.5B decode step.  gate/up take 896 logical columns stored as 1024
# (four Q4_K super-blocks, the last half zero-activated).
QWEN05B_LAYER = [
    ("q", Q8_0, 896, 896), ("k", Q8_0, 128, 896), ("v", Q8_0, 128, 896),
    ("o", Q8_0, 896, 896),
    ("gate", Q4_K, 4864, 1024), ("up", Q4_K, 4864, 1024),
    ("down", Q4_K, 896, 4864),
]
QWEN05B_VALID_COLS = {"gate": 896, "up": 896}
QWEN05B_GROUPS = [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]]
QWEN05B_LAYERS = 24
QWEN05B_LM_HEAD = ("lm_head", Q8_0, 151936, 896)

LLAMA8B_LM_HEAD_Q6K = ("lm_head", Q6_K, 128256, 4096)
PREFILL = ("prefill", Q4_K, 14336, 4096)  # X[512, 4096]
PREFILL_M = 512
PREFILL_SWEEP_M = (1, 2, 4, 8, 16, 32, 64, 512)


def seed_for(workload: int, layer: int, proj: int) -> int:
    """Deterministic seed per (workload, layer, projection)."""
    return 1_000_003 * workload + 1009 * layer + 17 * proj + 1
