"""Python binding of libqx, the GB300 block-quantised GEMV library.

Argument marshalling only: every function here checks Python-side types,
allocates outputs with torch when the caller passes none, and calls the C ABI
of ``include/qx.h`` with raw device pointers and the current CUDA stream.  All
arithmetic runs in the CUDA kernels.  There is no fallback: if ``libqx.so`` is
missing or the device is not a GB300, calls raise ``QxError``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

QX_Q8_0, QX_Q4_K, QX_Q6_K = 8, 12, 14
QX_Q6_K_SOA = 142  # Q6_K repacked at load time (qx_repack)
QX_MODE_F32, QX_MODE_W4A8, QX_MODE_W4A8_FUSED = 0, 1, 2
QX_FLAG_PDL = 0x100
QX_OK = 0
QX_ERR_ARG, QX_ERR_FMT, QX_ERR_SHAPE, QX_ERR_ALIGN = -1, -2, -3, -4
QX_ERR_MODE, QX_ERR_CUDA, QX_ERR_DEVICE_TIMEOUT, QX_ERR_UNSUPPORTED_DEVICE = -5, -6, -7, -8
QX_MAX_MULTI = 8
QX_MAX_COLS = 32768
QX_CHAIN_MAX_JOBS = 128
QX_CHAIN_MAX_ENTRIES = 4

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libqx.so")

EXPORTS = ["qx_quantize_act_q8", "qx_gemv", "qx_gemv_multi", "qx_gemm_prefill", "qx_gemm_prefill_ex",
           "qx_gemv_partials", "qx_gemv_chain", "qx_gemv_chain_noalloc", "qx_gemv_chain_scratch_bytes", "qx_row_bytes", "qx_repack",
           "qx_device_check", "qx_debug_timeout_probe", "qx_debug_mma_rate", "qx_debug_noalloc_fill",
           "qx_debug_trace_read", "qx_status_string", "qx_last_error", "qx_version"]


class QxError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        detail = f" [{qx_last_error()}]" if status == QX_ERR_CUDA else ""
        super().__init__(f"{what}: {qx_status_string(status)} ({status}){detail}")


class _Act(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("d", ctypes.c_void_p), ("sum", ctypes.c_void_p),
                ("m", ctypes.c_int64), ("cols", ctypes.c_int64)]


class _Job(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("n", ctypes.c_int), ("W", ctypes.c_void_p * 4),
                ("rows", ctypes.c_int64 * 4), ("y", ctypes.c_void_p * 4), ("cols", ctypes.c_int64),
                ("x", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libqx.so (built by ``build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libqx.so not found at {LIB_PATH}: build it with "
                               "`python -m block_quantized_gemv_q8_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.qx_quantize_act_q8.argtypes = [P, I64, I64, ctypes.POINTER(_Act), P]
        L.qx_gemv.argtypes = [I, P, I64, I64, P, P, I, P]
        L.qx_gemv_multi.argtypes = [I, P, P, P, I64, P, P, I, P]
        L.qx_gemm_prefill.argtypes = [I, P, I64, I64, ctypes.POINTER(_Act), P, P]
        L.qx_gemm_prefill_ex.argtypes = [I, P, I64, I64, ctypes.POINTER(_Act), P, I, P]
        L.qx_gemv_partials.argtypes = [I, P, I64, I64, ctypes.POINTER(_Act), P, P]
        L.qx_gemv_chain.argtypes = [I, ctypes.POINTER(_Job), P, P]
        L.qx_gemv_chain_noalloc.argtypes = [I, ctypes.POINTER(_Job), P]
        L.qx_gemv_chain_scratch_bytes.argtypes = [I]
        L.qx_gemv_chain_scratch_bytes.restype = ctypes.c_size_t
        L.qx_row_bytes.argtypes = [I, I64]
        L.qx_row_bytes.restype = ctypes.c_size_t
        L.qx_device_check.argtypes = [P]
        L.qx_repack.argtypes = [I, I, P, I64, I64, P, P]
        L.qx_debug_mma_rate.argtypes = [I, ctypes.POINTER(ctypes.c_double), P]
        L.qx_debug_timeout_probe.argtypes = [ctypes.c_uint64, P]
        L.qx_debug_noalloc_fill.argtypes = [ctypes.c_uint32, P]
        L.qx_debug_trace_read.argtypes = [P, ctypes.c_size_t]
        L.qx_status_string.argtypes = [I]
        L.qx_status_string.restype = ctypes.c_char_p
        L.qx_last_error.argtypes = []
        L.qx_last_error.restype = ctypes.c_char_p
        L.qx_version.argtypes = []
        L.qx_version.restype = ctypes.c_char_p
        for n in ("qx_quantize_act_q8", "qx_gemv", "qx_gemv_multi", "qx_gemm_prefill", "qx_gemm_prefill_ex",
                  "qx_gemv_partials", "qx_gemv_chain", "qx_gemv_chain_noalloc",
                  "qx_device_check", "qx_debug_timeout_probe",
                  "qx_repack", "qx_debug_mma_rate", "qx_debug_noalloc_fill",
                  "qx_debug_trace_read"):
            getattr(L, n).restype = I
        _lib = L
    return _lib


def build_library(force: bool = False) -> str:
    """Compile libqx.so in-tree (nvcc, sm_103a)."""
    import importlib
    return importlib.import_module(__name__ + ".build").build(force=force)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t: torch.Tensor) -> ctypes.c_void_p:
    if not t.is_cuda:
        raise ValueError("qx operates on CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("qx needs contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _nbytes(t: torch.Tensor) -> int:
    return t.numel() * t.element_size()


def _need(t: torch.Tensor, nbytes: int, what: str) -> torch.Tensor:
    """A CUDA, contiguous tensor holding at least nbytes: the library writes and
    reads through raw pointers, so a short buffer is refused here."""
    _ptr(t)
    if nbytes > 0 and _nbytes(t) < nbytes:
        raise ValueError(f"{what}: {_nbytes(t)} bytes, need {nbytes}")
    return t


def _need_weights(W: torch.Tensor, fmt: int, rows: int, cols: int, what: str = "W") -> torch.Tensor:
    rb = qx_row_bytes(fmt, cols)
    return _need(W, rows * rb, what) if rb > 0 and rows > 0 else W  # invalid shapes: the library names them


def _served_cols(fmt: int, cols: int) -> int:
    """cols when the format serves that width, else 0: an invalid shape is left
    to the library, which names it (QX_ERR_SHAPE / QX_ERR_FMT)."""
    return cols if qx_row_bytes(fmt, cols) > 0 else 0


def _need_act(a: "ActQ8", m: int, cols: int, what: str):
    _need(a.q, m * cols, what + ".q")
    _need(a.d, m * (cols // 32) * 4, what + ".d")
    _need(a.sum, m * (cols // 32) * 4, what + ".sum")


def _check(st: int, what: str):
    if st != QX_OK:
        raise QxError(st, what)


@dataclass
class ActQ8:
    """An int8-quantised activation: q [m, cols] int8, d and sum [m, cols/32]."""
    q: torch.Tensor
    d: torch.Tensor
    sum: torch.Tensor

    @property
    def m(self) -> int:
        return self.q.shape[0]

    @property
    def cols(self) -> int:
        return self.q.shape[1]

    @staticmethod
    def empty(m: int, cols: int, device=None) -> "ActQ8":
        device = device or torch.device("cuda")
        return ActQ8(torch.empty((m, cols), dtype=torch.int8, device=device),
                     torch.empty((m, cols // 32), dtype=torch.float32, device=device),
                     torch.empty((m, cols // 32), dtype=torch.int32, device=device))

    def c_struct(self) -> _Act:
        return _Act(_ptr(self.q).value, _ptr(self.d).value, _ptr(self.sum).value, self.m, self.cols)

    def row(self, i: int) -> "ActQ8":
        return ActQ8(self.q[i:i + 1], self.d[i:i + 1], self.sum[i:i + 1])


def qx_row_bytes(fmt: int, cols: int) -> int:
    return int(lib().qx_row_bytes(fmt, cols))


def qx_repack(from_fmt: int, to_fmt: int, W: torch.Tensor, rows: int, cols: int, out: torch.Tensor | None = None,
              stream=None) -> torch.Tensor:
    """Repack rows x cols weights between QX_Q6_K and QX_Q6_K_SOA (device to device)."""
    nbytes = rows * qx_row_bytes(to_fmt, cols)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _need_weights(W, from_fmt, rows, cols)
    _need(out, nbytes, "out")
    _check(lib().qx_repack(from_fmt, to_fmt, _ptr(W), rows, cols, _ptr(out), _stream(stream)), "qx_repack")
    return out


def qx_status_string(st: int) -> str:
    return lib().qx_status_string(st).decode()


def qx_last_error() -> str:
    return lib().qx_last_error().decode()


def qx_version() -> str:
    return lib().qx_version().decode()


def qx_quantize_act_q8(x: torch.Tensor, out: ActQ8 | None = None, stream=None) -> ActQ8:
    """x f32 [m, cols] (or [cols]) -> ActQ8 (int8 per block of 32 with an f32 absmax scale)."""
    if x.dtype != torch.float32:
        raise TypeError("qx_quantize_act_q8 takes float32 activations")
    x2 = x.reshape(1, -1) if x.dim() == 1 else x
    m, cols = x2.shape
    out = out or ActQ8.empty(m, cols, x.device)
    _need_act(out, m, cols, "out")
    a = out.c_struct()
    _check(lib().qx_quantize_act_q8(_ptr(x2), m, cols, ctypes.byref(a), _stream(stream)), "qx_quantize_act_q8")
    return out


def _x_arg(x, mode, cols: int = 0):
    if (mode & 0xFF) in (QX_MODE_F32, QX_MODE_W4A8_FUSED):
        if not isinstance(x, torch.Tensor) or x.dtype != torch.float32:
            raise TypeError("f32 and fused-W4A8 modes take a float32 activation tensor")
        return _ptr(_need(x, cols * 4, "x")), None
    if not isinstance(x, ActQ8):
        raise TypeError("W4A8 mode takes an ActQ8 (from qx_quantize_act_q8)")
    _need_act(x, 1, cols, "x")
    a = x.c_struct()
    return ctypes.cast(ctypes.pointer(a), ctypes.c_void_p), a


def qx_gemv(fmt: int, W: torch.Tensor, rows: int, cols: int, x, y: torch.Tensor | None = None,
            mode: int = QX_MODE_W4A8, stream=None) -> torch.Tensor:
    """y[rows] = W . x for block-quantised W (uint8 bytes).

    mode: QX_MODE_F32 (x f32), QX_MODE_W4A8 (x an ActQ8) or QX_MODE_W4A8_FUSED
    (x f32, quantised inside the launch), optionally | QX_FLAG_PDL."""
    y = y if y is not None else torch.empty(rows, dtype=torch.float32, device=W.device)
    _need_weights(W, fmt, rows, cols)
    _need(y, rows * 4, "y")
    xp, keep = _x_arg(x, mode, _served_cols(fmt, cols))
    _check(lib().qx_gemv(fmt, _ptr(W), rows, cols, xp, _ptr(y), mode, _stream(stream)), "qx_gemv")
    return y


def qx_gemv_multi(fmts, Ws, rows, cols: int, x, ys=None, mode: int = QX_MODE_W4A8, stream=None):
    """Several GEMVs over one activation in one launch per format."""
    n = len(Ws)
    ys = ys if ys is not None else [torch.empty(r, dtype=torch.float32, device=Ws[0].device) for r in rows]
    if not (len(fmts) == len(rows) == len(ys) == n):
        raise ValueError("qx_gemv_multi: fmts, Ws, rows and ys differ in length")
    for f, w, r, y in zip(fmts, Ws, rows, ys):
        _need_weights(w, f, r, cols)
        _need(y, r * 4, "y")
    F = (ctypes.c_int * n)(*fmts)
    Wp = (ctypes.c_void_p * n)(*[_ptr(w).value for w in Ws])
    R = (ctypes.c_int64 * n)(*rows)
    Yp = (ctypes.c_void_p * n)(*[_ptr(t).value for t in ys])
    xp, keep = _x_arg(x, mode, min(_served_cols(f, cols) for f in fmts) if n else 0)
    _check(lib().qx_gemv_multi(n, F, Wp, R, cols, xp, Yp, mode, _stream(stream)), "qx_gemv_multi")
    return ys


def qx_gemv_partials(fmt: int, W: torch.Tensor, rows: int, cols: int, x: ActQ8, P: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Exact int32 partial sums [rows, cols/32] (Q4_K, Q8_0) or [rows, cols/16] (Q6_K, QX_Q6_K_SOA)."""
    g = 16 if fmt in (QX_Q6_K, QX_Q6_K_SOA) else 32
    P = P if P is not None else torch.empty((rows, cols // g), dtype=torch.int32, device=W.device)
    _need_weights(W, fmt, rows, cols)
    _need(P, rows * (cols // g) * 4, "P")
    _need_act(x, 1, _served_cols(fmt, cols), "x")
    a = x.c_struct()
    _check(lib().qx_gemv_partials(fmt, _ptr(W), rows, cols, ctypes.byref(a), _ptr(P), _stream(stream)),
           "qx_gemv_partials")
    return P


def qx_gemm_prefill(fmt: int, W: torch.Tensor, rows: int, cols: int, X: ActQ8, Y: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Y [X.m, rows] = X' . W^T for a quantised activation batch X."""
    return qx_gemm_prefill_ex(fmt, W, rows, cols, X, Y, 0, stream)


def qx_gemm_prefill_ex(fmt: int, W: torch.Tensor, rows: int, cols: int, X: ActQ8, Y: torch.Tensor | None = None,
                       path: int = 0, stream=None) -> torch.Tensor:
    Y = Y if Y is not None else torch.empty((X.m, rows), dtype=torch.float32, device=W.device)
    _need_weights(W, fmt, rows, cols)
    _need(Y, X.m * rows * 4, "Y")
    _need_act(X, X.m, _served_cols(fmt, cols), "X")
    a = X.c_struct()
    _check(lib().qx_gemm_prefill_ex(fmt, _ptr(W), rows, cols, ctypes.byref(a), _ptr(Y), path, _stream(stream)),
           "qx_gemm_prefill_ex")
    return Y


@dataclass
class GemvJob:
    """One job of a chain: y[k] = W[k] . x for its entries (W4A8, in-kernel quantisation)."""
    fmt: int
    W: list
    rows: list
    cols: int
    x: torch.Tensor
    y: list | None = None


def qx_gemv_chain_scratch_bytes(n_jobs: int) -> int:
    return int(lib().qx_gemv_chain_scratch_bytes(n_jobs))


def chain_scratch(n_jobs: int, device=None) -> torch.Tensor:
    """Zero-filled scratch for a chain of n_jobs (reusable across calls)."""
    return torch.zeros(qx_gemv_chain_scratch_bytes(n_jobs), dtype=torch.uint8, device=device or "cuda")


def make_chain(jobs) -> ctypes.Array:
    """Marshal a list of GemvJob into the C array (outputs allocated if missing)."""
    arr = (_Job * len(jobs))()
    for j, job in enumerate(jobs):
        if job.y is None:
            job.y = [torch.empty(r, dtype=torch.float32, device=job.W[0].device) for r in job.rows]
        c = arr[j]
        c.fmt, c.n, c.cols = job.fmt, len(job.W), job.cols
        for k, (W, r, y) in enumerate(zip(job.W, job.rows, job.y)):
            _need_weights(W, job.fmt, r, job.cols)
            _need(y, r * 4, "y")
            c.W[k] = _ptr(W).value
            c.rows[k] = r
            c.y[k] = _ptr(y).value
        c.x = _ptr(_need(job.x, _served_cols(job.fmt, job.cols) * 4, "x")).value
    return arr


def qx_gemv_chain(jobs, scratch: torch.Tensor, stream=None, marshalled=None):
    """Run a chain of dependent GEMVs in one launch; returns the jobs (with y)."""
    arr = marshalled if marshalled is not None else make_chain(jobs)
    _check(lib().qx_gemv_chain(len(arr), arr, _ptr(scratch), _stream(stream)), "qx_gemv_chain")
    return jobs


def qx_gemv_chain_noalloc(jobs, stream=None, marshalled=None):
    """qx_gemv_chain with the library's own arrival counters (no scratch; at
    most QX_CHAIN_MAX_JOBS jobs; calls on one device must not overlap)."""
    arr = marshalled if marshalled is not None else make_chain(jobs)
    _check(lib().qx_gemv_chain_noalloc(len(arr), arr, _stream(stream)), "qx_gemv_chain_noalloc")
    return jobs


def qx_debug_mma_rate(kind: int, stream=None) -> float:
    """Measured mma.sync rate (multiply-adds x 2 per second): kind 0 int8 m16n8k32, 1 f16 m16n8k16."""
    v = ctypes.c_double(0.0)
    _check(lib().qx_debug_mma_rate(kind, ctypes.byref(v), _stream(stream)), "qx_debug_mma_rate")
    return v.value


def qx_device_check(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error status."""
    return int(lib().qx_device_check(_stream(stream)))


def qx_debug_timeout_probe(limit_ns: int, stream=None):
    _check(lib().qx_debug_timeout_probe(limit_ns, _stream(stream)), "qx_debug_timeout_probe")


def qx_debug_noalloc_fill(value: int, stream=None):
    """Fill the library's no-alloc chain counter array with `value` (test hook)."""
    _check(lib().qx_debug_noalloc_fill(value, _stream(stream)), "qx_debug_noalloc_fill")
