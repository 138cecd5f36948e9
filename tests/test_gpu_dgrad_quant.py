"""fp8_gemm_dgrad_quant: the data-gradient GEMM that also casts its bf16
output for the input-gradient GEMM ("Weight gradient kernels for dense and MoE
models": separate cast launches around the GEMMs cost end-to-end time).

The epilogue's dZ must be the bf16 dZ of fp8_gemm_dgrad (same kernel body),
and its e5m2 codes and 1x128 scales must be exactly the row cast of that
stored dZ: bit for bit against the library's own row cast and against the
oracle's cast of the same bf16 bytes.  Shapes are ragged in M, and N is a
multiple of 128 but not of the 256-column tile."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1


@pytest.mark.parametrize("M,N,K", [(300, 640, 384), (1000, 1024, 512), (129, 128, 128), (8192, 14336, 4096)])
def test_dgrad_quant_is_dgrad_then_row_cast(fp8, M, N, K):
    seed = 4000 + M + N
    dy = workloads.normal_bf16((M, K), seed, "dy", std=1e-2)
    w = workloads.normal_bf16((N, K), seed, "w", std=0.02)
    z = workloads.normal_bf16((M, N), seed, "z", std=2.0).cuda()
    A, B = fp8.quantize(dy.cuda(), E5M2), fp8.quantize(w.cuda(), E4M3)
    ref, _ = fp8.gemm_dgrad(A, B, z, fp8.EPI_DGELU)
    dz, Q = fp8.gemm_dgrad_quant(A, B, z)
    R = fp8.quantize(ref, E5M2)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    assert torch.equal(dz.view(torch.int16), ref.view(torch.int16)), "dZ differs from fp8_gemm_dgrad"
    assert torch.equal(Q.q, R.q), "codes differ from the row cast of the stored dZ"
    assert torch.equal(Q.scale[:, :M].contiguous().view(torch.int32), R.scale[:, :M].contiguous().view(torch.int32))
    # the oracle's cast of the same bf16 bytes (sampled rows at the full size)
    rows = np.arange(M) if M * N <= 2 ** 22 else np.unique(np.r_[0, M - 1, np.random.default_rng(seed).choice(M, 64)])
    qo, so = oracle.quantize(workloads.bits(dz[torch.from_numpy(rows).cuda()]), E5M2)
    assert np.array_equal(Q.q[torch.from_numpy(rows).cuda()].cpu().numpy(), qo)
    assert np.array_equal(Q.scale[:, torch.from_numpy(rows).cuda()].cpu().numpy(), so)


def test_dgrad_quant_rejects_unblocked_n(fp8):
    A = fp8.quantize(torch.zeros(256, 128, dtype=torch.bfloat16, device="cuda"), E5M2)
    B = fp8.quantize(torch.zeros(200, 128, dtype=torch.bfloat16, device="cuda"), E4M3)
    z = torch.zeros(256, 200, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error) as e:
        fp8.gemm_dgrad_quant(A, B, z, q_out=fp8.empty_fp8(256, 256, E5M2))
    assert e.value.code == fp8.binding.ERR_INVALID_ARG
