"""Bounded pipeline waits: a GEMM whose producer issues no loads (a flag that
nothing else sets) must time out, record FP8LL_ERR_TIMEOUT in the device
status word, write nothing, and leave the context usable."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


def test_starved_pipeline_times_out_and_context_survives(fp8):
    M, N, K = 256, 256, 256
    A = fp8.quantize(workloads.normal_bf16((M, K), 1, "a").cuda(), 0)
    B = fp8.quantize(workloads.normal_bf16((N, K), 1, "b").cuda(), 0)
    out = torch.zeros(M, N, device="cuda")
    assert fp8.device_status() == 0
    fp8.debug_starve_next_gemm(50)
    fp8.gemm_wgrad(A, B, out)
    assert fp8.device_status() == fp8.binding.ERR_TIMEOUT
    assert fp8.device_status() == 0  # reading clears it
    assert bool((out == 0).all())    # the starved launch wrote nothing
    fp8.gemm_wgrad(A, B, out)        # the next launch works normally
    assert fp8.device_status() == 0
    assert torch.isfinite(out).all() and out.abs().sum() > 0


def test_invalid_call_launches_nothing(fp8):
    M, N, K = 128, 256, 256
    A = fp8.quantize(workloads.normal_bf16((M, K), 2, "a").cuda(), 0)
    B = fp8.quantize(workloads.normal_bf16((N, K), 2, "b").cuda(), 0)
    out = torch.full((M, N), 7.0, device="cuda")
    with pytest.raises(fp8.Fp8Error):
        fp8.gemm_wgrad(A, B, out, K=200)
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())


def _starve_pair_kernel(fp8, gemm, A, B, M, N):
    # the CTA-pair kernels: the leader's MMA and scale-copy warps and both CTAs'
    # epilogue warps give up after the budget, meet at the final cluster
    # barrier and free tensor memory; nothing is written
    out = torch.full((M, N), 3.0, device="cuda")
    assert fp8.device_status() == 0
    fp8.debug_starve_next_gemm(50)
    gemm(A, B, out)
    assert fp8.device_status() == fp8.binding.ERR_TIMEOUT
    assert fp8.device_status() == 0
    assert bool((out == 3.0).all())
    gemm(A, B, out, accumulate=False)
    assert fp8.device_status() == 0
    assert torch.isfinite(out).all() and out.abs().sum() > 0


def test_starved_mx_pair_kernel_times_out_and_context_survives(fp8):
    M, N, K = 512, 256, 256
    A = fp8.mx_quantize(workloads.normal_bf16((M, K), 3, "a").cuda(), 0)
    B = fp8.mx_quantize(workloads.normal_bf16((N, K), 3, "b").cuda(), 0)
    _starve_pair_kernel(fp8, fp8.mx_gemm_wgrad, A, B, M, N)


def test_starved_per_tensor_pair_kernel_times_out_and_context_survives(fp8):
    M, N, K = 512, 256, 256
    a = workloads.normal_bf16((M, K), 4, "a").cuda()
    b = workloads.normal_bf16((N, K), 4, "b").cuda()
    A, _ = fp8.tensor_quantize(a, 0, fp8.tensor_amax(a))
    B, _ = fp8.tensor_quantize(b, 0, fp8.tensor_amax(b))
    _starve_pair_kernel(fp8, fp8.tensor_gemm_wgrad, A, B, M, N)
