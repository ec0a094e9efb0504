"""The C-ABI library loads, exports every entry point declared in include/*.h,
and rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

import block_quantized_gemv_q8_gb300 as qx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qx.build_library()
    return qx.lib()


def declared_functions(header=None):
    """qx_* functions declared in one header, or in every header of include/."""
    inc = os.path.join(ROOT, "include")
    names = [header] if header else sorted(f for f in os.listdir(inc) if f.endswith(".h"))
    found = set()
    for h in names:
        text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, h)).read(), flags=re.S)
        found |= set(re.findall(r"\b(qx_[a-z0-9_]+)\s*\(", text))
    return sorted(found)


def test_product_header_declares_no_debug_hooks():
    """Test and measurement hooks live in qx_debug.h, apart from the product calls."""
    product, debug = declared_functions("qx.h"), declared_functions("qx_debug.h")
    assert not [n for n in product if n.startswith("qx_debug")]
    assert debug and all(n.startswith("qx_debug") for n in debug)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["qx_quantize_act_q8", "qx_gemv", "qx_gemv_multi", "qx_gemm_prefill", "qx_gemv_partials",
              "qx_gemv_chain"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in include/ but not exported by libqx.so"
    assert set(qx.EXPORTS) <= set(declared_functions())


def test_row_bytes(lib):
    assert qx.qx_row_bytes(qx.QX_Q4_K, 4096) == 16 * 144
    assert qx.qx_row_bytes(qx.QX_Q6_K, 14336) == 56 * 210
    assert qx.qx_row_bytes(qx.QX_Q8_0, 896) == 28 * 34
    assert qx.qx_row_bytes(qx.QX_Q4_K, 896) == 0
    assert qx.qx_row_bytes(qx.QX_Q8_0, 0) == 0
    assert qx.qx_row_bytes(7, 256) == 0
    # the repacked Q6_K layout: 208 bytes per super-block, then the f16 d values padded to 16 bytes
    assert qx.qx_row_bytes(qx.QX_Q6_K_SOA, 4096) == 16 * 208 + 32 == qx.qx_row_bytes(qx.QX_Q6_K, 4096)
    assert qx.qx_row_bytes(qx.QX_Q6_K_SOA, 14336) == 56 * 208 + 112
    assert qx.qx_row_bytes(qx.QX_Q6_K_SOA, 2304) == 9 * 208 + 32
    assert qx.qx_row_bytes(qx.QX_Q6_K_SOA, 256) == 208 + 16
    assert qx.qx_row_bytes(qx.QX_Q6_K_SOA, 128) == 0


def test_status_strings_and_version(lib):
    for st in range(0, -9, -1):
        assert qx.qx_status_string(st).startswith("QX_")
    assert "sm_103a" in qx.qx_version()


A16 = 1 << 20  # a fake but 16-byte aligned address; never dereferenced


def test_host_validation_rejects_before_launch(lib):
    P, s = ctypes.c_void_p, None
    # unknown format / mode
    assert lib.qx_gemv(99, P(A16), 4, 256, P(A16), P(A16), 0, s) == qx.QX_ERR_FMT
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, P(A16), P(A16), 7, s) == qx.QX_ERR_MODE
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, P(A16), P(A16), 0x200 | 1, s) == qx.QX_ERR_MODE
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, P(A16 + 4), P(A16), qx.QX_MODE_W4A8_FUSED, s) == qx.QX_ERR_ALIGN
    # shape: cols not whole blocks, too wide, rows < 1
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 896, P(A16), P(A16), 0, s) == qx.QX_ERR_SHAPE
    assert lib.qx_gemv(qx.QX_Q8_0, P(A16), 4, 40, P(A16), P(A16), 0, s) == qx.QX_ERR_SHAPE
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 65536, P(A16), P(A16), 0, s) == qx.QX_ERR_SHAPE
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 0, 256, P(A16), P(A16), 0, s) == qx.QX_ERR_SHAPE
    # null pointers
    assert lib.qx_gemv(qx.QX_Q4_K, None, 4, 256, P(A16), P(A16), 0, s) == qx.QX_ERR_ARG
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, None, P(A16), 0, s) == qx.QX_ERR_ARG
    # misaligned pointers
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16 + 2), 4, 256, P(A16), P(A16), 0, s) == qx.QX_ERR_ALIGN
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, P(A16 + 4), P(A16), 0, s) == qx.QX_ERR_ALIGN
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, P(A16), P(A16 + 2), 0, s) == qx.QX_ERR_ALIGN
    # W4A8 activation descriptor checks
    act = qx._Act(A16, A16, A16, 1, 512)
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, ctypes.cast(ctypes.pointer(act), P), P(A16), 1, s) == \
        qx.QX_ERR_SHAPE
    act = qx._Act(A16, A16 + 4, A16, 1, 256)
    assert lib.qx_gemv(qx.QX_Q4_K, P(A16), 4, 256, ctypes.cast(ctypes.pointer(act), P), P(A16), 1, s) == \
        qx.QX_ERR_ALIGN
    act = qx._Act(A16, None, A16, 1, 256)
    assert lib.qx_gemv_partials(qx.QX_Q4_K, P(A16), 4, 256, ctypes.byref(act), P(A16), s) == qx.QX_ERR_ARG
    # multi: bad counts
    F = (ctypes.c_int * 9)(*([qx.QX_Q4_K] * 9))
    assert lib.qx_gemv_multi(0, F, None, None, 256, P(A16), None, 0, s) == qx.QX_ERR_ARG
    assert lib.qx_gemv_multi(9, F, None, None, 256, P(A16), None, 0, s) == qx.QX_ERR_ARG
    # quantise: cols not a multiple of 32
    act = qx._Act(A16, A16, A16, 0, 0)
    assert lib.qx_quantize_act_q8(P(A16), 1, 48, ctypes.byref(act), s) == qx.QX_ERR_SHAPE
    assert lib.qx_quantize_act_q8(P(A16 + 4), 1, 64, ctypes.byref(act), s) == qx.QX_ERR_ALIGN
    # prefill: bad path
    act = qx._Act(A16, A16, A16, 4, 256)
    assert lib.qx_gemm_prefill_ex(qx.QX_Q4_K, P(A16), 4, 256, ctypes.byref(act), P(A16), 5, s) == qx.QX_ERR_ARG
    # timeout probe limits
    assert lib.qx_debug_timeout_probe(10, s) == qx.QX_ERR_ARG
    # repack: only Q6_K <-> QX_Q6_K_SOA, aligned, not overlapping
    SOA, Q6 = qx.QX_Q6_K_SOA, qx.QX_Q6_K
    assert lib.qx_repack(qx.QX_Q4_K, SOA, P(A16), 4, 256, P(2 * A16), s) == qx.QX_ERR_FMT
    assert lib.qx_repack(Q6, Q6, P(A16), 4, 256, P(2 * A16), s) == qx.QX_ERR_FMT
    assert lib.qx_repack(Q6, SOA, P(A16), 4, 384, P(2 * A16), s) == qx.QX_ERR_SHAPE
    assert lib.qx_repack(Q6, SOA, P(A16 + 2), 4, 256, P(2 * A16), s) == qx.QX_ERR_ALIGN
    assert lib.qx_repack(SOA, Q6, P(A16), 4, 256, None, s) == qx.QX_ERR_ARG
    assert lib.qx_repack(Q6, SOA, P(A16), 4, 256, P(A16 + 256), s) == qx.QX_ERR_ARG  # overlap
    # the repacked layout is read by the GEMV only: the chain and the GEMM prefill paths refuse it
    act = qx._Act(A16, A16, A16, 4, 256)
    for path in (2, 3, 4):
        assert lib.qx_gemm_prefill_ex(SOA, P(A16), 4, 256, ctypes.byref(act), P(A16), path, s) == qx.QX_ERR_FMT
    job = qx._Job(SOA, 1, (ctypes.c_void_p * 4)(A16), (ctypes.c_int64 * 4)(4), (ctypes.c_void_p * 4)(A16), 256, A16)
    assert lib.qx_gemv_chain(1, ctypes.byref(job), P(A16), s) == qx.QX_ERR_FMT
    # the mma.sync rate probe: two kinds, an out pointer
    v = ctypes.c_double(0.0)
    assert lib.qx_debug_mma_rate(2, ctypes.byref(v), s) == qx.QX_ERR_ARG
    assert lib.qx_debug_mma_rate(0, None, s) == qx.QX_ERR_ARG


def test_python_binding_rejects_cpu_tensors(lib):
    import torch
    with pytest.raises((ValueError, TypeError)):
        qx.qx_gemv(qx.QX_Q4_K, torch.zeros(144, dtype=torch.uint8), 1, 256, torch.zeros(256), mode=qx.QX_MODE_F32)


def test_missing_library_fails_loudly(tmp_path):
    """Without libqx.so the binding raises; nothing falls back to another path."""
    import subprocess
    import sys
    code = ("import block_quantized_gemv_q8_gb300 as qx\n"
            f"qx.LIB_PATH = {str(tmp_path / 'missing' / 'libqx.so')!r}\n"
            "try:\n"
            "    qx.qx_row_bytes(qx.QX_Q4_K, 256)\n"
            "except RuntimeError as e:\n"
            "    print('raised:', e)\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert "raised:" in r.stdout and "libqx.so not found" in r.stdout



def test_python_binding_refuses_host_tensors_before_sizes(lib):
    """Every tensor goes through the same check (CUDA, contiguous, enough bytes);
    a host tensor is refused first."""
    import torch
    with pytest.raises(ValueError):
        qx._need(torch.zeros(4), 16, "t")


def test_header_compiles_as_c_and_links_from_c(lib, tmp_path):
    """include/qx.h is plain C: a C99 program built with -pedantic -Werror
    links libqx.so, loads it and gets the declared results from the calls
    that need no GPU."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    pkg = os.path.dirname(qx.LIB_PATH)
    exe = tmp_path / "abi_consumer"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "abi_consumer.c"), "-o", str(exe), "-L", pkg, "-lqx",
           f"-Wl,-rpath,{pkg}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"


def test_host_code_under_asan_and_ubsan(lib, tmp_path):
    """The library's host code (argument checks, shape arithmetic, status
    strings) compiled with -fsanitize=address,undefined, driven by the C
    consumer: no report, and a planted heap overread in the consumer is
    reported (the sanitizer is live in that process)."""
    import shutil
    import subprocess
    from block_quantized_gemv_q8_gb300 import build as qb
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    asan = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not os.path.isabs(asan) or not os.path.exists(asan):
        pytest.skip("no AddressSanitizer runtime")
    san = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer"]
    api_obj = tmp_path / "qx_api_san.o"
    subprocess.run([qb.nvcc(), "-c", os.path.join(qb.CSRC, "qx_api.cu"), "-o", str(api_obj), "-O1", "-g",
                    "-std=c++17", "-Xcompiler", ",".join(["-fPIC"] + san)] + qb.ARCH,
                   check=True, capture_output=True, text=True)
    objs = [os.path.join(qb.OUT_DIR, s.replace(".cu", ".o")) for s in qb.SOURCES if s != "qx_api.cu"]
    so = tmp_path / "libqx.so"
    subprocess.run([qb.nvcc(), "-shared", "-o", str(so), str(api_obj)] + objs + qb.ARCH +
                   ["-cudart", "static", "-Xcompiler", ",".join(san)], check=True, capture_output=True, text=True)
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1", UBSAN_OPTIONS="print_stacktrace=1")
    for plant, ok in ((False, True), (True, False)):
        exe = tmp_path / ("consumer_planted" if plant else "consumer")
        cmd = ["gcc", "-std=c99", "-g", "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_consumer.c"),
               "-o", str(exe), "-L", str(tmp_path), "-lqx", f"-Wl,-rpath,{tmp_path}"] + san
        if plant:
            cmd.append("-DQX_PLANT_OOB")
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120, env=env)
        if ok:
            assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr[-3000:]
            assert "runtime error" not in r.stderr and "AddressSanitizer" not in r.stderr, r.stderr[-3000:]
        else:
            assert r.returncode != 0 and "AddressSanitizer" in r.stderr, (r.stdout, r.stderr[-2000:])


def test_size_queries_need_no_gpu(lib):
    """Chain scratch sizes follow the header's formula; invalid counts give 0.
    The prefill needs no workspace: the header declares no size query for one."""
    assert not [n for n in declared_functions() if "workspace" in n]
    assert qx.qx_gemv_chain_scratch_bytes(1) == 8
    assert qx.qx_gemv_chain_scratch_bytes(qx.QX_CHAIN_MAX_JOBS) == 4 * (qx.QX_CHAIN_MAX_JOBS + 1)
    assert qx.qx_gemv_chain_scratch_bytes(0) == 0
    assert qx.qx_gemv_chain_scratch_bytes(qx.QX_CHAIN_MAX_JOBS + 1) == 0
