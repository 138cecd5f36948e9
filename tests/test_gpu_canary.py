"""No write outside the outputs: every output buffer is a window into a larger
allocation whose guard regions before and after hold a sentinel pattern; after
each call on ragged shapes (partial tiles in M, N and the casts' tails) the
guards must be unchanged.  Covers the casts (codes and scales, every recipe),
the three GEMMs with their epilogues, the bias gradient, the k-grouped weight
gradient, and the MXFP8 and per-tensor GEMMs."""
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
GUARD_BYTES = 256  # a multiple of 16, so that every window stays 16-byte aligned


class Guarded:
    """`shape` of `dtype` inside a byte buffer with GUARD_BYTES of sentinel on
    both sides."""

    def __init__(self, shape, dtype):
        n = 1
        for d in shape:
            n *= d
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((GUARD_BYTES * 2 + nbytes,), 0xA5, dtype=torch.uint8, device="cuda")
        self.view = self.buf[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype).view(*shape)
        self.nbytes = nbytes

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.buf[:GUARD_BYTES] == 0xA5).all()) and bool((self.buf[GUARD_BYTES + self.nbytes:] == 0xA5).all())


def guarded_fp8(fp8, rows, k, fmt):
    q, s = Guarded((rows, k), torch.uint8), Guarded((k // 128, fp8.scale_ld(rows)), torch.float32)
    return fp8.Fp8Tensor(q.view, s.view, fmt), (q, s)


@pytest.mark.parametrize("M,N,K", [(129, 257, 128), (300, 520, 384), (77, 13, 256)])
def test_gemm_outputs_stay_in_bounds(fp8, M, N, K):
    x = workloads.normal_bf16((M, K), 700, "x").cuda()
    w = workloads.normal_bf16((N, K), 700, "w", std=0.05).cuda()
    b = workloads.normal_bf16((N,), 700, "b", std=0.1).cuda()
    z = workloads.normal_bf16((M, N), 700, "z").cuda()
    X, gx = guarded_fp8(fp8, M, K, E4M3)
    W, gw = guarded_fp8(fp8, N, K, E4M3)
    fp8.quantize(x, E4M3, out=X)
    fp8.quantize(w, E4M3, out=W)
    assert all(g.intact() for g in gx + gw), "cast"
    Y, Z = Guarded((M, N), torch.bfloat16), Guarded((M, N), torch.bfloat16)
    fp8.gemm_fprop(X, W, b, fp8.EPI_BIAS_GELU, out=Y.view, aux=Z.view)
    assert Y.intact() and Z.intact(), "fprop"
    dZ, bg = Guarded((M, N), torch.bfloat16), Guarded((N,), torch.float32)
    fp8.gemm_dgrad(X, W, z, fp8.EPI_DGELU_BGRAD, out=dZ.view, bgrad=bg.view)
    assert dZ.intact() and bg.intact(), "dgrad"
    for accumulate in (False, True):
        out = Guarded((M, N), torch.float32)
        out.view.zero_()
        fp8.gemm_wgrad(X, W, out.view, accumulate=accumulate)
        assert out.intact(), "wgrad"
    G = Guarded((2, M, N), torch.float32)
    G.view.zero_()
    Xg, _ = guarded_fp8(fp8, M, 256, E4M3)
    Wg, _ = guarded_fp8(fp8, N, 256, E4M3)
    fp8.quantize(workloads.normal_bf16((M, 256), 701, "xg").cuda(), E4M3, out=Xg)
    fp8.quantize(workloads.normal_bf16((N, 256), 701, "wg").cuda(), E4M3, out=Wg)
    fp8.grouped_wgrad(Xg, Wg, [128, 128], G.view)
    assert G.intact(), "grouped wgrad"


@pytest.mark.parametrize("M,N,K", [(129, 384, 128), (300, 640, 256)])
def test_dgrad_quant_outputs_stay_in_bounds(fp8, M, N, K):
    # the data gradient that casts its own output: dZ, its codes and scales
    x = workloads.normal_bf16((M, K), 702, "x").cuda()
    w = workloads.normal_bf16((N, K), 702, "w", std=0.05).cuda()
    z = workloads.normal_bf16((M, N), 702, "z").cuda()
    X, W = fp8.quantize(x, E5M2), fp8.quantize(w, E4M3)
    dZ = Guarded((M, N), torch.bfloat16)
    Q, gq = guarded_fp8(fp8, M, N, E5M2)
    fp8.gemm_dgrad_quant(X, W, z, out=dZ.view, q_out=Q)
    assert dZ.intact() and all(g.intact() for g in gq), "dgrad with the row cast"


def test_casts_stay_in_bounds(fp8):
    x = workloads.normal_bf16((384, 136), 702, "c").cuda()
    T, gt = guarded_fp8(fp8, 136, 384, E5M2)
    fp8.quantize(x, E5M2, transpose=True, out=T)
    assert all(g.intact() for g in gt), "transposed cast"
    x2 = workloads.normal_bf16((256, 384), 703, "d").cuda()
    R, gr = guarded_fp8(fp8, 256, 384, E4M3)
    C, gc = guarded_fp8(fp8, 384, 256, E4M3)
    fp8.quantize_dual(x2, E4M3, out=R, out_t=C)
    assert all(g.intact() for g in gr + gc), "two-way cast"
    qm = Guarded((256, 384), torch.uint8)
    sf = Guarded((fp8.mx_sf_bytes(256, 384),), torch.uint8)
    fp8.mx_quantize(x2, E4M3, out=fp8.Fp8MxTensor(qm.view, sf.view, E4M3))
    assert qm.intact() and sf.intact(), "MXFP8 cast"
    qr, qc = Guarded((256, 384), torch.uint8), Guarded((384, 256), torch.uint8)
    sc, seen = Guarded((1,), torch.float32), Guarded((1,), torch.float32)
    am = fp8.tensor_amax(x2)
    fp8.tensor_quantize(x2, E4M3, am, rows=True, cols=True, amax_out=seen.view,
                        out=fp8.Fp8TensorScaled(qr.view, sc.view, E4M3),
                        out_t=fp8.Fp8TensorScaled(qc.view, sc.view, E4M3))
    assert qr.intact() and qc.intact() and sc.intact() and seen.intact(), "per-tensor cast"


@pytest.mark.parametrize("M,N,K", [(129, 257, 128), (300, 520, 384)])
def test_mx_and_per_tensor_gemm_outputs_stay_in_bounds(fp8, M, N, K):
    x = workloads.normal_bf16((M, K), 704, "x").cuda()
    w = workloads.normal_bf16((N, K), 704, "w", std=0.05).cuda()
    b = workloads.normal_bf16((N,), 704, "b", std=0.1).cuda()
    z = workloads.normal_bf16((M, N), 704, "z").cuda()
    operands = [(fp8.mx_quantize(x, E4M3), fp8.mx_quantize(w, E4M3), fp8.mx_gemm_fprop, fp8.mx_gemm_dgrad,
                 fp8.mx_gemm_wgrad)]
    Xt, _ = fp8.tensor_quantize(x, E4M3, fp8.tensor_amax(x))
    Wt, _ = fp8.tensor_quantize(w, E4M3, fp8.tensor_amax(w))
    operands.append((Xt, Wt, fp8.tensor_gemm_fprop, fp8.tensor_gemm_dgrad, fp8.tensor_gemm_wgrad))
    for A, B, fprop, dgrad, wgrad in operands:
        Y, Z = Guarded((M, N), torch.bfloat16), Guarded((M, N), torch.bfloat16)
        fprop(A, B, b, fp8.EPI_BIAS_GELU, out=Y.view, aux=Z.view)
        dZ, bg = Guarded((M, N), torch.bfloat16), Guarded((N,), torch.float32)
        dgrad(A, B, z, fp8.EPI_DGELU_BGRAD, out=dZ.view, bgrad=bg.view)
        out = Guarded((M, N), torch.float32)
        out.view.zero_()
        wgrad(A, B, out.view)
        assert all(g.intact() for g in (Y, Z, dZ, bg, out)), fprop.__name__
