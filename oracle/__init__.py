"""ctypes loader for the plain-C oracle (``qx_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``.  The CUDA library never imports,
links or calls it, and it imports nothing from the CUDA side.

Every function returns numpy arrays computed by the C code; nothing here does
arithmetic of the method.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qx_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile qx_oracle.c to a shared library (gcc, OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    os.makedirs(_OUT_DIR, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        # QX_ORACLE_LIB lets the mutation tests load a deliberately broken copy.
        path = os.environ.get("QX_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.orc_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f64.restype = ctypes.c_double
        L.orc_row_bytes.argtypes = [I, I64]
        L.orc_row_bytes.restype = I64
        L.orc_dequant_row.argtypes = [I, P, I64, P]
        L.orc_quantize_act_q8.argtypes = [P, I64, I64, P, P, P]
        L.orc_gemv_f64x.argtypes = [I, P, I64, I64, P, P, P, I]
        L.orc_gemv_f32.argtypes = [I, P, I64, I64, P, P, P, I]
        L.orc_partials.argtypes = [I, P, I64, I64, P, P]
        L.orc_gemv_w4a8.argtypes = [I, P, I64, I64, P, P, P, P, I]
        L.orc_gemm_w4a8.argtypes = [I, P, I64, I64, I64, P, P, P, P, I]
        for name in ("orc_dequant_row", "orc_quantize_act_q8", "orc_gemv_f64x", "orc_gemv_f32",
                     "orc_partials", "orc_gemv_w4a8", "orc_gemm_w4a8", "orc_max_threads",
                     "orc_block_weights", "orc_block_bytes", "orc_partial_group"):
            getattr(L, name).restype = I
        for name in ("orc_block_weights", "orc_block_bytes", "orc_partial_group"):
            getattr(L, name).argtypes = [I]
        L.orc_max_threads.argtypes = []
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def f16_to_f64(h: int) -> float:
    return lib().orc_f16_to_f64(h)


def row_bytes(fmt: int, cols: int) -> int:
    return int(lib().orc_row_bytes(fmt, cols))


def partial_group(fmt: int) -> int:
    return int(lib().orc_partial_group(fmt))


def dequant(fmt: int, W: np.ndarray, cols: int) -> np.ndarray:
    """Dequantised weights [rows, cols] (float64)."""
    W = np.ascontiguousarray(W, dtype=np.uint8).reshape(-1, row_bytes(fmt, cols))
    out = np.empty((W.shape[0], cols), dtype=np.float64)
    for r in range(W.shape[0]):
        _check(lib().orc_dequant_row(fmt, _p(W[r]), cols, _p(out[r])), "dequant_row")
    return out


def quantize_act_q8(x: np.ndarray):
    """x f32 [m, cols] -> (q int8 [m, cols], d f32 [m, cols/32], sum int32 [m, cols/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    m, cols = x.shape
    q = np.empty((m, cols), dtype=np.int8)
    d = np.empty((m, cols // 32), dtype=np.float32)
    s = np.empty((m, cols // 32), dtype=np.int32)
    _check(lib().orc_quantize_act_q8(_p(x), m, cols, _p(q), _p(d), _p(s)), "quantize_act_q8")
    return q, d, s


def gemv_f32(fmt: int, W: np.ndarray, rows: int, cols: int, x: np.ndarray, threads: int | None = None,
             with_absdot: bool = True):
    """f32 mode: (y float64 [rows], absdot float64 [rows] or None)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(cols)
    y = np.empty(rows, dtype=np.float64)
    a = np.empty(rows, dtype=np.float64) if with_absdot else None
    _check(lib().orc_gemv_f32(fmt, _p(W), rows, cols, _p(x), _p(y), _p(a) if with_absdot else None,
                              threads or default_threads()), "gemv_f32")
    return y, a


def gemv_f64x(fmt: int, W: np.ndarray, rows: int, cols: int, x: np.ndarray, threads: int | None = None):
    W = np.ascontiguousarray(W, dtype=np.uint8)
    x = np.ascontiguousarray(x, dtype=np.float64).reshape(cols)
    y = np.empty(rows, dtype=np.float64)
    a = np.empty(rows, dtype=np.float64)
    _check(lib().orc_gemv_f64x(fmt, _p(W), rows, cols, _p(x), _p(y), _p(a),
                               threads or default_threads()), "gemv_f64x")
    return y, a


def partials(fmt: int, W: np.ndarray, rows: int, cols: int, qx: np.ndarray) -> np.ndarray:
    """int32 [rows, cols/group] integer partial sums."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    qx = np.ascontiguousarray(qx, dtype=np.int8).reshape(cols)
    P = np.empty((rows, cols // partial_group(fmt)), dtype=np.int32)
    _check(lib().orc_partials(fmt, _p(W), rows, cols, _p(qx), _p(P)), "partials")
    return P


def gemv_w4a8(fmt: int, W: np.ndarray, rows: int, cols: int, qx: np.ndarray, dx: np.ndarray,
              threads: int | None = None, with_absdot: bool = True):
    """W4A8 mode from an already quantised activation: (y, absdot) float64 [rows].

    with_absdot=False skips the tolerance scale (absdot is then None)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    qx = np.ascontiguousarray(qx, dtype=np.int8).reshape(cols)
    dx = np.ascontiguousarray(dx, dtype=np.float32).reshape(cols // 32)
    y = np.empty(rows, dtype=np.float64)
    a = np.empty(rows, dtype=np.float64) if with_absdot else None
    _check(lib().orc_gemv_w4a8(fmt, _p(W), rows, cols, _p(qx), _p(dx), _p(y), _p(a) if with_absdot else None,
                               threads or default_threads()), "gemv_w4a8")
    return y, a


def gemm_w4a8(fmt: int, W: np.ndarray, rows: int, cols: int, qx: np.ndarray, dx: np.ndarray,
              threads: int | None = None):
    """Prefill: Y [m, rows] float64 (and absdot) from quantised X [m, cols]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    qx = np.ascontiguousarray(qx, dtype=np.int8).reshape(-1, cols)
    m = qx.shape[0]
    dx = np.ascontiguousarray(dx, dtype=np.float32).reshape(m, cols // 32)
    Y = np.empty((m, rows), dtype=np.float64)
    A = np.empty((m, rows), dtype=np.float64)
    _check(lib().orc_gemm_w4a8(fmt, _p(W), rows, cols, m, _p(qx), _p(dx), _p(Y), _p(A),
                               threads or default_threads()), "gemm_w4a8")
    return Y, A


def max_threads() -> int:
    return int(lib().orc_max_threads())


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
