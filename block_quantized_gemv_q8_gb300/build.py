"""Build libqx.so (the CUDA C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the shared library links the CUDA
runtime statically, so it needs nothing from PyTorch.  Usage:

    python -m block_quantized_gemv_q8_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqx.so")
SOURCES = ["qx_api.cu", "qx_actq8.cu", "qx_gemv.cu", "qx_f32mma.cu", "qx_chain.cu", "qx_prefill.cu", "qx_tc.cu", "qx_repack.cu", "qx_mma_rate.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"] + ARCH
# Extra defines for measurement sweeps of the launch geometry (e.g.
# QX_NVCC_DEFINES="QX_STAGE_KB=24 QX_INFLIGHT_KB=48"); empty in normal builds.
NVCC_FLAGS += ["-D" + d for d in os.environ.get("QX_NVCC_DEFINES", "").split()]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the qx CUDA library cannot be built")


def _deps() -> list[str]:
    inc_dir = os.path.join(os.path.dirname(HERE), "include")
    inc = [os.path.join(inc_dir, f) for f in os.listdir(inc_dir) if f.endswith(".h")]
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hdrs + inc


def _stale(target: str, sources: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(OUT_DIR, os.path.basename(src).replace(".cu", ".o"))
    if _stale(obj, [src] + _deps()):
        cmd = [nvcc(), "-c", src, "-o", obj] + NVCC_FLAGS
        r = subprocess.run(cmd, capture_output=True, text=True)
        log = obj + ".ptxas.txt"
        with open(log, "w") as f:
            f.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
        if verbose:
            sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    if force:
        for s in srcs:
            o = os.path.join(OUT_DIR, os.path.basename(s).replace(".cu", ".o"))
            if os.path.exists(o):
                os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
