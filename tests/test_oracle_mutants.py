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


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation anchor not found: %s" % name
    src = tmp_path / "oracle.c"
    src.write_text(text.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           "-o", str(lib), str(src), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] + PIN_TESTS,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch: %s\n%s" % (name, r.stdout[-2000:])
