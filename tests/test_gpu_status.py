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
