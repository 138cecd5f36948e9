"""FAST accumulation ("FP8 GEMM for the fprop should use fast accumulation":
fast accumulation is the faster mode of unstated precision, selected per call)
on every 1x128 GEMM entry point, through the C ABI, against the CPU oracle.

The library's FAST runs the FULL promotion (every 128-deep K block meets its
own scale pair), so a FAST call must give the FULL call's bits, and both must
lie inside the FAST bound 8e-3 * S (S = sum_k |a_ik b_jk|) of the oracle.  The
long-K case follows the accumulation study's recipe at a reduced size: K =
16384, 1% of the rows of both operands scaled x64 (outliers), error measured
on sampled 256 x 256 output tiles that include outlier rows and columns.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (FAST_C, FULL_C, MAX_DGELU, assert_within, bf16_to_f64, bf16_ulp, dgelu_eval_bound, f32_ulp)

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
M, N, K = 300, 520, 384  # several 128 x 256 tiles, ragged in M and N


def operands(fp8, fa, fb, seed, std=1.0):
    a = workloads.normal_bf16((M, K), seed, "a", std=std)
    b = workloads.normal_bf16((N, K), seed, "b", std=std)
    A, B = fp8.quantize(a.cuda(), fa), fp8.quantize(b.cuda(), fb)
    qa, sa = oracle.quantize(workloads.bits(a), fa)
    qb, sb = oracle.quantize(workloads.bits(b), fb)
    acc, S = oracle.gemm(qa, sa, fa, qb, sb, fb)
    return A, B, acc, S


def same_bits(x, y):
    return torch.equal(x.contiguous().view(torch.uint8), y.contiguous().view(torch.uint8))


@pytest.mark.parametrize("epi", [0, 1, 2])
def test_fprop_fast(fp8, epi):
    A, B, acc, S = operands(fp8, E4M3, E4M3, 61)
    bias = workloads.normal_bf16((N,), 61, "bias", std=0.1)
    bc = bias.cuda() if epi else None
    Yf, Zf = fp8.gemm_fprop(A, B, bc, epi=epi, acc=fp8.ACC_FULL)
    Yq, Zq = fp8.gemm_fprop(A, B, bc, epi=epi, acc=fp8.ACC_FAST)
    torch.cuda.synchronize()
    assert same_bits(Yf, Yq)
    if epi == 2:
        assert same_bits(Zf, Zq)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(bias) if epi else None, gelu_on=(epi == 2))
    y = bf16_to_f64(Yq)
    gain = MAX_DGELU if epi == 2 else 1.0
    assert_within(y, Yo, gain * FAST_C * S + bf16_ulp(np.maximum(np.abs(y), np.abs(Yo))) + 1e-5 * np.abs(Zo), "Y")


@pytest.mark.parametrize("epi", [3, 4])
def test_dgrad_fast(fp8, epi):
    A, B, acc, S = operands(fp8, E5M2, E4M3, 62, std=0.05)
    z = workloads.normal_bf16((M, N), 62, "z", std=2.0).cuda()
    dZf, bgf = fp8.gemm_dgrad(A, B, z, epi=epi, acc=fp8.ACC_FULL)
    dZq, bgq = fp8.gemm_dgrad(A, B, z, epi=epi, acc=fp8.ACC_FAST)
    torch.cuda.synchronize()
    assert same_bits(dZf, dZq)
    if epi == 4:
        assert same_bits(bgf, bgq)
    dzo = oracle.dgrad_epilogue(acc, workloads.bits(z))
    zf = bf16_to_f64(z)
    elem = np.abs(oracle.dgelu(zf)) * FAST_C * S + np.abs(acc) * dgelu_eval_bound(zf)
    d = bf16_to_f64(dZq)
    assert_within(d, dzo, elem + bf16_ulp(np.maximum(np.abs(d), np.abs(dzo))), "dZ")
    if epi == 4:
        n_bands = 4 * ((M + 127) // 128)
        bound = elem.sum(0) + (8 + n_bands) * 2.0 ** -24 * np.abs(dzo).sum(0) + 1e-30
        assert_within(bgq.cpu().double().numpy(), oracle.colsum(dzo), bound, "bgrad")


@pytest.mark.parametrize("accumulate", [True, False])
def test_wgrad_fast(fp8, accumulate):
    A, B, acc, S = operands(fp8, E5M2, E4M3, 63, std=0.02)
    pre = workloads.normal_f32((M, N), 63, "pre", std=1e-3).cuda()
    outf, outq = pre.clone(), pre.clone()
    fp8.gemm_wgrad(A, B, outf, accumulate=accumulate, acc=fp8.ACC_FULL)
    fp8.gemm_wgrad(A, B, outq, accumulate=accumulate, acc=fp8.ACC_FAST)
    torch.cuda.synchronize()
    assert same_bits(outf, outq)
    want = oracle.wgrad(acc, pre.cpu().double().numpy() if accumulate else None)
    assert_within(outq.cpu().double().numpy(), want, FAST_C * S + f32_ulp(want), "out")


def test_grouped_wgrad_fast(fp8):
    ks = [128, 0, 256]
    a = workloads.normal_bf16((M, K), 64, "a", std=0.02)
    b = workloads.normal_bf16((N, K), 64, "b", std=0.02)
    A, B = fp8.quantize(a.cuda(), E4M3), fp8.quantize(b.cuda(), E4M3)
    pre = workloads.normal_f32((len(ks), M, N), 64, "pre", std=1e-3).cuda()
    outf, outq = pre.clone(), pre.clone()
    fp8.grouped_wgrad(A, B, ks, outf, acc=fp8.ACC_FULL)
    fp8.grouped_wgrad(A, B, ks, outq, acc=fp8.ACC_FAST)
    torch.cuda.synchronize()
    assert same_bits(outf, outq)
    qa, sa = oracle.quantize(workloads.bits(a), E4M3)
    qb, sb = oracle.quantize(workloads.bits(b), E4M3)
    want, S = oracle.grouped_wgrad(qa, sa, E4M3, qb, sb, E4M3, ks, prefill=pre.cpu().double().numpy())
    assert_within(outq.cpu().double().numpy(), want, FAST_C * S + f32_ulp(want), "grouped out")


def test_long_k_outlier_rows_full_and_fast(fp8):
    """Forward GEMM, bf16 out, K = 16384 with 1% outlier rows (x64) in both
    operands: max error normalized by S on 9 sampled 256 x 256 tiles (6 random,
    two through outlier rows of X and W, the last tile) within 2e-3 (FULL) and
    8e-3 (FAST), bf16 rounding of Y included."""
    Ms = Ns = 1024
    Kl = 16384
    x, xo = workloads.with_outlier_rows(workloads.normal_bf16((Ms, Kl), 65, "x"), 65, "x")
    w, wo = workloads.with_outlier_rows(workloads.normal_bf16((Ns, Kl), 65, "w"), 65, "w")
    X, W = fp8.quantize(x.cuda(), E4M3), fp8.quantize(w.cuda(), E4M3)
    Yf, _ = fp8.gemm_fprop(X, W, None, epi=0, acc=fp8.ACC_FULL)
    Yq, _ = fp8.gemm_fprop(X, W, None, epi=0, acc=fp8.ACC_FAST)
    torch.cuda.synchronize()
    assert same_bits(Yf, Yq)
    qx, sx = oracle.quantize(workloads.bits(x), E4M3)
    qw, sw = oracle.quantize(workloads.bits(w), E4M3)
    rng = np.random.default_rng(65)
    tiles = [(int(rng.integers(0, Ms // 256)), int(rng.integers(0, Ns // 256))) for _ in range(6)]
    tiles += [(int(xo[0]) // 256, int(wo[-1]) // 256), (int(xo[-1]) // 256, int(wo[0]) // 256),
              (Ms // 256 - 1, Ns // 256 - 1)]
    yf, yq = bf16_to_f64(Yf), bf16_to_f64(Yq)
    for (ti, tj) in tiles:
        rows = np.arange(256 * ti, 256 * ti + 256)
        cols = np.arange(256 * tj, 256 * tj + 256)
        acc, S = oracle.gemm(qx, sx, E4M3, qw, sw, E4M3, rows=rows, cols=cols)
        ulp = bf16_ulp(np.abs(acc))
        for name, y, c in (("full", yf, FULL_C), ("fast", yq, FAST_C)):
            got = y[np.ix_(rows, cols)]
            assert_within(got, acc, c * S + ulp, "%s tile (%d, %d)" % (name, ti, tj))
