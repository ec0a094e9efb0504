"""The oracle under AddressSanitizer and UndefinedBehaviorSanitizer.

The oracle's C source is compiled with -fsanitize=address,undefined (UB
reports fatal) and the pin suite is run against it in a subprocess, the
sanitizer runtime preloaded into the interpreter.  A second build with an
out-of-bounds write planted in a copy of the source shows that the
sanitizer is live: that run must fail with an AddressSanitizer report.  The
committed oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qx_oracle.c")


def _asan_runtime():
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    p = subprocess.run(["gcc", "-print-file-name=libasan.so"], capture_output=True, text=True).stdout.strip()
    if not os.path.isabs(p) or not os.path.exists(p):
        pytest.skip("no AddressSanitizer runtime")
    return p


def _build(src_text: str, out_dir: str) -> str:
    c = os.path.join(out_dir, "oracle_san.c")
    so = os.path.join(out_dir, "liboracle_san.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-g", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer",
                    "-o", so, c, "-lm"], check=True, capture_output=True)
    return so


def _run_pins(so: str, runtime: str):
    env = dict(os.environ, QX_ORACLE_LIB=so, PYTHONPATH=ROOT, LD_PRELOAD=runtime,
               ASAN_OPTIONS="detect_leaks=0", UBSAN_OPTIONS="print_stacktrace=1")
    return subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                           "-x", "-q", "-s", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=600)


def test_pins_pass_under_asan_and_ubsan(tmp_path):
    runtime = _asan_runtime()
    r = _run_pins(_build(open(SRC).read(), str(tmp_path)), runtime)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-3000:]
    assert "AddressSanitizer" not in out and "runtime error" not in out, out[-3000:]


def test_planted_overflow_is_reported(tmp_path):
    """One weight past the end of the dequantised row: the sanitizer must stop the run."""
    runtime = _asan_runtime()
    src = open(SRC).read()
    old = "for (int64_t b = 0; b < cols / bw; b++) {"
    assert src.count(old) == 1
    r = _run_pins(_build(src.replace(old, "for (int64_t b = 0; b <= cols / bw; b++) {"), str(tmp_path)), runtime)
    assert r.returncode != 0
    assert "AddressSanitizer" in r.stdout + r.stderr
