"""Each plausible mistake planted in a copy of the oracle must fail a pin.

Every mutation below is a one-token slip of the kind the pins are meant to
catch (a dropped term, a wrong sign, shift, offset or index, another rounding
rule).  The mutated C source is compiled to a temporary library and the pin
suite is run against it in a subprocess; the test passes only if that run
fails.  The committed oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qx_oracle.c")

MUTATIONS = [
    ("f16 subnormal scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    ("f16 normal exponent bias", "e - 25);", "e - 24);"),
    ("q4_k scale high bits shift", "((s[j - 4] >> 6) << 4)", "((s[j - 4] >> 6) << 3)"),
    ("q4_k min high bits from the scale byte", "| ((s[j] >> 6) << 4)", "| ((s[j - 4] >> 6) << 4)"),
    ("q4_k low/high nibble swapped", "(e % 64) < 32 ? (b & 15) : (b >> 4)", "(e % 64) < 32 ? (b >> 4) : (b & 15)"),
    ("q4_k chunk stride", "blk[16 + 32 * (e / 64) + e % 32]", "blk[16 + 32 * (e / 32) % 128 + e % 32]"),
    ("q4_k min sign", "d * sc * q4k_quant(blk, e) - dmin * m", "d * sc * q4k_quant(blk, e) + dmin * m"),
    ("q6_k offset 31", "(q6k_quant(blk, e) - 32)", "(q6k_quant(blk, e) - 31)"),
    ("q6_k qh bit field", ">> (2 * t)) & 3", ">> (2 * h)) & 3"),
    ("q6_k ql half select", "blk[64 * h + 32 * (t & 1) + l]", "blk[64 * h + 32 * (t >> 1) + l]"),
    ("q6_k scale group of 32", "blk[192 + e / 16]", "blk[192 + e / 32]"),
    ("q8_0 quant offset", "(int8_t)blk[2 + e]", "(int8_t)blk[1 + e]"),
    ("act quant rounds half away from zero", "nearbyintf(xb[i] / db)", "roundf(xb[i] / db)"),
    ("act quant scale 1/128", "amax / 127.0f", "amax / 128.0f"),
    ("act quant multiplies by the reciprocal", "nearbyintf(xb[i] / db)", "nearbyintf(xb[i] * (1.0f / db))"),
    ("act quant block sum of magnitudes", "s += v;", "s += v < 0 ? -v : v;"),
    ("act quant clamp dropped", "v = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);", "v = (int)r;"),
    ("act quant clamp at 128", "v = r > 127.0f ? 127 : (r < -127.0f ? -127 : (int)r);",
     "v = r > 128.0f ? 128 : (r < -128.0f ? -128 : (int)r);"),
    ("gemv reversed activation index", "acc += w[i] * x[i];", "acc += w[i] * x[cols - 1 - i];"),
    ("w4a8 min term sign", "- f16_at(blk + 2) * m * dxg * (double)S", "+ f16_at(blk + 2) * m * dxg * (double)S"),
    ("w4a8 q6_k partial without -32", "qw = q6k_quant(blk, e0 + i) - 32;", "qw = q6k_quant(blk, e0 + i);"),
    ("partials activation index", "(int64_t)qw * qx[col0 + i]", "(int64_t)qw * qx[i]"),
    ("w4a8 activation scale of the wrong block", "(double)dx[col0 / 32]", "(double)dx[col0 / 64]"),
    ("w4a8 q4_k sub-block index", "(int)((col0 % 256) / 32)", "(int)((col0 % 256) / 64)"),
    ("q4_k d and dmin swapped", "double d = f16_at(blk), dmin = f16_at(blk + 2);",
     "double d = f16_at(blk + 2), dmin = f16_at(blk);"),
    ("q6_k d read from the front of the block", "double d = f16_at(blk + 208);", "double d = f16_at(blk);"),
    ("w4a8 q4_k min scaled by d", "- f16_at(blk + 2) * m * dxg", "- f16_at(blk) * m * dxg"),
    ("w4a8 q6_k scale of another group", "q6k_scale(blk, (int)(col0 % 256))", "q6k_scale(blk, (int)(col0 % 128))"),
    ("f32 gemv drops the last column", "for (int64_t i = 0; i < cols; i++) {\n                acc += w[i] * x[i];",
     "for (int64_t i = 0; i < cols - 1; i++) {\n                acc += w[i] * x[i];"),
    ("prefill activation scales of the wrong row", "dx + i * (cols / 32)", "dx + i * (cols / 64)"),
    ("act quant amax misses the last value", "for (int i = 0; i < 32; i++)\n            if (fabsf(xb[i]) > amax)",
     "for (int i = 0; i < 31; i++)\n            if (fabsf(xb[i]) > amax)"),
    ("q6_k low nibble for the upper quarters", "int low4 = t < 2 ? (lo & 15) : (lo >> 4);",
     "int low4 = t < 2 ? (lo >> 4) : (lo & 15);"),
    ("q6_k partial groups of 32", "if (fmt == ORC_Q6_K) return 16;", "if (fmt == ORC_Q6_K) return 32;"),
    ("w4a8 q4_k min term over half the block", "for (int i = 0; i < 32; i++) S += qx[col0 + i];",
     "for (int i = 0; i < 16; i++) S += qx[col0 + i];"),
    ("w4a8 q8_0 scale read past d", "acc += f16_at(blk) * dxg * (double)P[g];",
     "acc += f16_at(blk + 2) * dxg * (double)P[g];"),
    ("tolerance scale without the absolute value", "aacc += fabs(w[i] * ((double)dx[i / 32] * qx[i]));",
     "aacc += w[i] * ((double)dx[i / 32] * qx[i]);"),
]


def _compile(src_text: str, out_dir: str) -> str:
    c = os.path.join(out_dir, "mut.c")
    so = os.path.join(out_dir, "libmut.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", so, c, "-lm"], check=True, capture_output=True)
    return so


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    so = _compile(src.replace(old, new), str(tmp_path))
    env = dict(os.environ, QX_ORACLE_LIB=so, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutation '{name}' survived the pins:\n{r.stdout[-2000:]}"


def test_unmutated_copy_passes(tmp_path):
    so = _compile(open(SRC).read(), str(tmp_path))
    env = dict(os.environ, QX_ORACLE_LIB=so, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
