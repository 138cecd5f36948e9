"""The boundary from plain C: include/fp8ll.h compiles as C11, and a C program
linked against the built library calls through it.  CPU only: every call
below is settled by the host-side argument checks (or needs no device)."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fp8ll.h"

#define CHECK(cond) do { if (!(cond)) { printf("failed: %s (line %d)\n", #cond, __LINE__); return 1; } } while (0)

int main(void) {
    /* sizes and strings need no device */
    CHECK(fp8_scale_ld(5) == 8 && fp8_scale_ld(8) == 8);
    CHECK(fp8_workspace_size(256, 100) == 4u * 2u * 4u * 100u);
    CHECK(strlen(fp8_status_string(FP8LL_ERR_INVALID_ARG)) > 0);
    CHECK(fp8_mx_sf_bytes(256, 128) == 2 * 512);
    /* invalid arguments are refused before any device call */
    void* p = (void*)0x10000;
    CHECK(fp8_quantize(p, 4, 100, 128, FP8LL_E4M3, 0, (uint8_t*)p, (float*)p, 4, NULL) == FP8LL_ERR_INVALID_ARG);
    CHECK(fp8_quantize(NULL, 0, 0, 0, FP8LL_E4M3, 0, NULL, NULL, 0, NULL) == FP8LL_OK);
    CHECK(fp8_quantize_dual(p, 100, 256, 256, FP8LL_E5M2, (uint8_t*)p, (float*)p, 100, (uint8_t*)p, (float*)p,
                            256, NULL) == FP8LL_ERR_INVALID_ARG);
    fp8ll_operand_t op = {(const uint8_t*)p, (const float*)p, 256, 8, FP8LL_E4M3, 0};
    CHECK(fp8_gemm_fprop(8, 8, 200, &op, &op, p, FP8LL_EPI_BIAS_GELU, FP8LL_ACC_FULL, p, NULL, NULL) ==
          FP8LL_ERR_INVALID_ARG);
    CHECK(fp8_gemm_dgrad(8, 8, 256, &op, &op, p, FP8LL_EPI_DGELU_BGRAD, FP8LL_ACC_FULL, p, (float*)p, p, 4, NULL) ==
          FP8LL_ERR_WORKSPACE);
    int64_t ks[2] = {128, 100};
    CHECK(fp8_grouped_wgrad(2, 8, 8, ks, &op, &op, (float*)p, 1, FP8LL_ACC_FULL, NULL) == FP8LL_ERR_INVALID_ARG);
    fp8ll_mx_operand_t mop = {(const uint8_t*)p, (const uint8_t*)p, 200, FP8LL_E4M3, 0};
    CHECK(fp8_mx_gemm_wgrad(8, 8, 256, &mop, &mop, (float*)p, 1, NULL) == FP8LL_ERR_INVALID_ARG);
    fp8ll_tensor_operand_t top = {(const uint8_t*)p, NULL, 256, FP8LL_E4M3, 0};
    CHECK(fp8_tensor_gemm_fprop(8, 8, 256, &top, &top, p, FP8LL_EPI_BIAS_GELU, p, NULL, NULL) ==
          FP8LL_ERR_INVALID_ARG);
    CHECK(fp8_amax_history_update((float*)p, 0, 4, (const float*)p, (float*)p, NULL) == FP8LL_ERR_INVALID_ARG);
    /* the bias-gradient entries: refused on the host, or nothing to do */
    CHECK(fp8_bgrad_from_operand(8, 200, &op, (float*)p, 0, NULL) == FP8LL_ERR_INVALID_ARG);
    CHECK(fp8_bgrad_from_operand(0, 256, &op, NULL, 0, NULL) == FP8LL_OK);
    CHECK(fp8_quantize_dbias(p, 256, 64, 64, FP8LL_E5M2, (uint8_t*)p, (float*)p, 64, NULL, NULL, 0,
                             (float*)((char*)p + 4096), (char*)p + 8192, 2 * 64 * 4 - 4, NULL) == FP8LL_ERR_WORKSPACE);
    CHECK(fp8_quantize_dbias(p, 200, 64, 64, FP8LL_E5M2, (uint8_t*)p, (float*)p, 64, NULL, NULL, 0,
                             (float*)p, p, 1 << 20, NULL) == FP8LL_ERR_INVALID_ARG);
    CHECK(fp8_mx_quantize_dbias(p, 256, 60, 64, FP8LL_E5M2, (uint8_t*)p, (uint8_t*)p, (float*)p, p, 1 << 20,
                                NULL) == FP8LL_ERR_INVALID_ARG);
    CHECK(fp8_mx_quantize_dbias(p, 256, 0, 64, FP8LL_E5M2, (uint8_t*)p, (uint8_t*)p, NULL, NULL, 0, NULL) ==
          FP8LL_OK);
    printf("ok\n");
    return 0;
}
"""


def test_header_is_c11():
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-pedantic", "-fsyntax-only", "-x", "c",
                        os.path.join(INCLUDE, "fp8ll.h")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_calls_the_library(tmp_path):
    import fp8_linear_layer_gb300.build as b
    lib = b.build()
    src = tmp_path / "abi.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "abi"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-o", str(exe), str(src), "-I", INCLUDE, lib,
                        "-Wl,-rpath," + os.path.dirname(lib)], capture_output=True, text=True)
    if r.returncode != 0 and "cannot find" in r.stderr:
        pytest.skip("linker cannot resolve the CUDA runtime here: " + r.stderr.strip().splitlines()[-1])
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stdout + out.stderr
