"""fp8_gemm_dgrad_noalloc: the data-gradient GEMM with bias-gradient sums for
callers that cannot allocate device memory (a runtime whose allocator owns
all device memory, a step replayed from a fixed memory plan, a C caller with
no allocator).  It uses the library's own fixed scratch array instead of a
caller workspace, so its results must match fp8_gemm_dgrad's, call after call
(the array keeps the previous call's contents), and sizes whose bias-gradient
partials do not fit the array must be refused before any launch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import FULL_C, assert_within, bf16_to_f64, bf16_ulp, dgelu_eval_bound

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
SCRATCH_BYTES = 16 << 20  # the built-in array: 4 Mi fp32 partial sums


def call_noalloc(fp8, A, B, z, out, bg, M, N, K):
    L = fp8.lib()
    oa, ob = A.operand(), B.operand()
    return L.fp8_gemm_dgrad_noalloc(M, N, K, ctypes.byref(oa), ctypes.byref(ob), ctypes.c_void_p(z.data_ptr()),
                                    fp8.EPI_DGELU_BGRAD, fp8.ACC_FULL, ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(bg.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_dgrad_matches_allocating_entry_point_twice(fp8):
    M, N, K = 1000, 1288, 512
    dy = workloads.normal_bf16((M, K), 91, "dy", std=1e-2)
    w = workloads.normal_bf16((N, K), 91, "w", std=0.02)
    z = workloads.normal_bf16((M, N), 91, "z", std=2.0).cuda()
    A = fp8.quantize(dy.cuda(), E5M2)
    B = fp8.quantize(w.cuda(), E4M3)
    ref_dz, ref_bg = fp8.gemm_dgrad(A, B, z, fp8.EPI_DGELU_BGRAD)
    torch.cuda.synchronize()
    # the oracle's dZ (float64, before bf16 rounding) and its column sums, with
    # the bound the other data-gradient tests use (from the oracle's sum |a b|)
    qa, sa = oracle.quantize(workloads.bits(dy), E5M2)
    qb, sb = oracle.quantize(workloads.bits(w), E4M3)
    acc, S = oracle.gemm(qa, sa, E5M2, qb, sb, E4M3)
    dzo = oracle.dgrad_epilogue(acc, workloads.bits(z))
    dbo = oracle.colsum(dzo)
    zf = bf16_to_f64(z)
    g = np.abs(oracle.dgelu(zf))
    ev = np.abs(acc) * dgelu_eval_bound(zf)
    elem = g * FULL_C * S + ev
    for _ in range(2):  # the second call finds the first call's partials in the array
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        bg = torch.full((N,), float("nan"), device="cuda")
        assert call_noalloc(fp8, A, B, z, out, bg, M, N, K) == 0
        torch.cuda.synchronize()
        assert fp8.device_status() == 0
        # the same kernels in the same order as fp8_gemm_dgrad: identical bits
        assert torch.equal(out.view(torch.int16), ref_dz.view(torch.int16)), "dZ differs from fp8_gemm_dgrad"
        assert torch.equal(bg.view(torch.int32), ref_bg.view(torch.int32)), "bgrad differs from fp8_gemm_dgrad"
        d = bf16_to_f64(out)
        assert_within(d, dzo, elem + bf16_ulp(np.maximum(np.abs(d), np.abs(dzo))), "dZ vs oracle")
        bb = bg.cpu().double().numpy()
        assert_within(bb, dbo, elem.sum(0) + 40 * 2.0 ** -24 * np.abs(dzo).sum(0) + 1e-30, "bgrad vs oracle")


def test_noalloc_refuses_sizes_beyond_its_scratch(fp8):
    # ceil(M/128) * 4 * N fp32 partials must fit in 16 MiB; 4096 x 65536 needs 32 MiB
    M, N, K = 4096, 65536, 128
    assert fp8.workspace_size(M, N) > SCRATCH_BYTES
    # operands of the full sizes (arguments are checked before the size is)
    A = fp8.quantize(torch.zeros(M, K, dtype=torch.bfloat16, device="cuda"), E5M2)
    B = fp8.quantize(torch.zeros(N, K, dtype=torch.bfloat16, device="cuda"), E4M3)
    z = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    bg = torch.zeros(4, device="cuda")
    assert call_noalloc(fp8, A, B, z, out, bg, M, N, K) == fp8.binding.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 0).all()) and bool((bg == 0).all())
