"""The oracle's pins catch plausible mistakes.

Each case copies oracle.c, plants one mistake (a dropped term, a wrong sign or
index, a swapped operand, a wrong rounding rule), compiles the copy, and runs
the oracle pin tests against it in a subprocess: they must fail.  CPU only; the
mistakes live only in temporary copies of the oracle.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PIN_TESTS = ["tests/test_oracle_codec.py", "tests/test_oracle_quantize.py", "tests/test_oracle_gemm.py",
             "tests/test_oracle_epilogue.py"]

MUTANTS = {
    "gemm drops the B scale": ("total += s_a * s_b * part;", "total += s_a * part;"),
    "gemm ignores the K offset": ("const uint8_t* pa = qa + i * lda + k0 + kb * 128;",
                                  "const uint8_t* pa = qa + i * lda + kb * 128;"),
    "gemm uses the wrong block scale": ("const double s_b = (double)sb[(kb0 + kb) * sb_ld + j];",
                                        "const double s_b = (double)sb[kb0 * sb_ld + j];"),
    "gemm transposes B": ("const uint8_t* pb = qb + j * ldb + k0 + kb * 128;",
                          "const uint8_t* pb = qb + (j % 3) * ldb + k0 + kb * 128;"),
    "encode ties away from even": ("else code = (lo & 1) ? hi : lo;", "else code = hi;"),
    "encode does not saturate": ("    if (a >= t[top]) {\n        code = top;",
                                 "    if (a >= t[top] * 1.1) {\n        code = 0x7F;"),
    "decode with a wrong exponent bias": ("const int bias = (fmt == ORACLE_E4M3) ? 7 : 15;",
                                          "const int bias = (fmt == ORACLE_E4M3) ? 8 : 15;"),
    "quantize scale inverted": ("scale = amax / fmax; /* binary32 division */",
                                "scale = fmax / amax; /* binary32 division */"),
    "quantize divides instead of multiplying": ("const float y = v[k] * inv; /* binary32 product */",
                                                "const float y = v[k] / inv; /* binary32 product */"),
    "transposed quantize reads rows": ("v[k] = oracle_bf16_to_f32(x[(b * 128 + k) * ldx + c]);",
                                       "v[k] = oracle_bf16_to_f32(x[(b * 128 + k) * ldx + (c % 2)]);"),
    "gelu wrong sign": ("return z / (1.0 + exp(-2.0 * u));", "return z / (1.0 + exp(2.0 * u));"),
    "gelu drops the cubic term": ("const double u = c * (z + 0.044715 * z * z * z);\n    return",
                                  "const double u = c * z;\n    return"),
    "dgelu drops a term": ("return sp + 2.0 * z * c * (1.0 + 3.0 * 0.044715 * z * z) * sp * sm;",
                           "return sp;"),
    "dgelu drops the cubic factor": ("return sp + 2.0 * z * c * (1.0 + 3.0 * 0.044715 * z * z) * sp * sm;",
                                     "return sp + 2.0 * z * c * sp * sm;"),
    "colsum over the wrong axis": ("for (int64_t i = 0; i < M; ++i) s += dz[i * N + j];",
                                   "for (int64_t i = 0; i < M; ++i) s += dz[j * M + i] * (j * M + i < M * N);"),
    "bf16 rounding truncates": ("const double r = nearbyint(a / spacing) * spacing;",
                                "const double r = floor(a / spacing) * spacing;"),
}


# per-tensor scaling: checked against its own pin file only
TENSOR_MUTANTS = {
    "tensor cast scale inverted": ("scale = amax_in / fmax; /* binary32 division */",
                                   "scale = fmax / amax_in; /* binary32 division */"),
    "tensor cast ignores the given amax": ("const float t = fmax / amax_in; /* binary32 division */",
                                           "const float t = fmax / 1.0f; /* binary32 division */"),
    "tensor cast records a signed maximum": ("const float a = fabsf(v);\n            if (a > amax) amax = a;",
                                             "const float a = v;\n            if (a > amax) amax = a;"),
    "tensor cast transposes wrongly": ("q[c * rows + r] = code;", "q[r * cols + c] = code;"),
    "history keeps the oldest instead of the newest": ("    hist[0] = amax_new;\n", "    hist[0] = hist[0];\n"),
    "history maximum skips the newest": ("for (int64_t i = 0; i < len; ++i)\n        if (hist[i] > m) m = hist[i];",
                                         "for (int64_t i = 1; i < len; ++i)\n        if (hist[i] > m) m = hist[i];"),
    "tensor gemm drops the B scale": ("const double s = (double)sa * (double)sb;", "const double s = (double)sa;"),
    "tensor gemm reads a wrong B row": ("const double p = ta[qa[i * lda + k]] * tb[qb[j * ldb + k]];",
                                        "const double p = ta[qa[i * lda + k]] * tb[qb[(j % 3) * ldb + k]];"),
}


# MXFP8: checked against its own pin file only
MX_MUTANTS = {
    "mx exponent one too small (the block saturates)": (
        "while (e > -127 && amax <= ldexp(fmax, e - 1)) --e;", "while (e > -127 && amax < ldexp(fmax, e)) --e;"),
    "mx codes scaled by 2^e instead of 2^-e": ("oracle_fp8_encode(fmt, (float)ldexp((double)v[k], -e));",
                                               "oracle_fp8_encode(fmt, (float)ldexp((double)v[k], e));"),
    "mx transposed cast reads rows": ("v[k] = oracle_bf16_to_f32(x[(b * 32 + k) * ldx + c]);",
                                      "v[k] = oracle_bf16_to_f32(x[(b * 32 + k) * ldx + (c % 2)]);"),
    "mx gemm drops the B exponent": ("const double b = ldexp(tb[qb[j * ldb + k]], eb[(k / 32) * eb_ld + j]);",
                                     "const double b = tb[qb[j * ldb + k]];"),
    "mx gemm uses the wrong 32-element group": ("const double a = ldexp(ta[qa[i * lda + k]], ea[(k / 32) * ea_ld + i]);",
                                                "const double a = ldexp(ta[qa[i * lda + k]], ea[(k / 128) * ea_ld + i]);"),
}


def run_pins_on_mutant(tmp_path, old, new, name, pin_tests):
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor not found: %s" % name
    src = tmp_path / "oracle.c"
    src.write_text(text.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(lib), str(src), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] + pin_tests,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch: %s\n%s" % (name, r.stdout[-2000:])


# bias gradient reduced from the fp8 operand: checked against its own pin file only
BGRADB_MUTANTS = {
    "operand row sum reads the scale of another row": (
        "const double v = (double)scale[(k / 128) * scale_ld + r] * t[q[r * ldq + k]];",
        "const double v = (double)scale[(k / 128) * scale_ld + r / 2] * t[q[r * ldq + k]];"),
    "operand row sum uses the first block's scale": (
        "const double v = (double)scale[(k / 128) * scale_ld + r] * t[q[r * ldq + k]];",
        "const double v = (double)scale[r] * t[q[r * ldq + k]];"),
    "operand row sum decodes with the wrong format": (
        "    const double* t = g_table[fmt ? 1 : 0];\n#pragma omp parallel for schedule(static)\n    for (int64_t r = 0;",
        "    const double* t = g_table[0];\n#pragma omp parallel for schedule(static)\n    for (int64_t r = 0;"),
}


@pytest.mark.parametrize("name", sorted(BGRADB_MUTANTS))
def test_bgradb_pins_catch_mutant(name, tmp_path):
    old, new = BGRADB_MUTANTS[name]
    run_pins_on_mutant(tmp_path, old, new, name, ["tests/test_oracle_bgrad_operand.py"])


@pytest.mark.parametrize("name", sorted(TENSOR_MUTANTS))
def test_tensor_pins_catch_mutant(name, tmp_path):
    old, new = TENSOR_MUTANTS[name]
    run_pins_on_mutant(tmp_path, old, new, name, ["tests/test_oracle_tensor.py"])


@pytest.mark.parametrize("name", sorted(MX_MUTANTS))
def test_mx_pins_catch_mutant(name, tmp_path):
    old, new = MX_MUTANTS[name]
    run_pins_on_mutant(tmp_path, old, new, name, ["tests/test_oracle_mx.py"])


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    run_pins_on_mutant(tmp_path, old, new, name, PIN_TESTS)
