"""MXFP8 path through the C ABI vs the oracle.

Casts: codes and scale exponents bit-exact against the oracle's MX cast
(scale bytes read back through the documented storage layout), padding bytes
127.  GEMMs: every epilogue on shapes with ragged M / N tails, within
2e-3 * S (S = sum_k |a_ik b_jk| of the dequantized operands) plus one bf16 ulp
for bf16 outputs -- the tensor core accumulates the scaled products in fp32
over the whole K range -- and bitwise repeatable.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import FULL_C, MAX_DGELU, assert_within, bf16_to_f64, bf16_ulp, dgelu_eval_bound, f32_ulp

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1


def sf_exponents(sf, rows, K):
    """Exponents [K/32][rows] from the scale bytes (layout of fp8ll.h)."""
    G = 2 * ((rows + 255) // 256)
    b = sf.cpu().numpy().astype(np.int16)
    kb, r, k = np.meshgrid(np.arange(K // 128), np.arange(rows), np.arange(4), indexing="ij")
    off = (kb * G + r // 128) * 512 + (r % 128 % 32) * 16 + (r % 128 // 32) * 4 + k
    e = (b[off] - 127).astype(np.int8)             # [K/128][rows][4]
    return np.ascontiguousarray(e.transpose(0, 2, 1).reshape(K // 32, rows))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rows,cols", [(300, 384), (256, 128), (1, 256), (513, 640)])
def test_mx_quantize_rows_bit_exact(fp8, fmt, rows, cols):
    x, _ = workloads.with_outlier_rows(workloads.normal_bf16((rows, cols), 91, "mxq", std=2.0), 91, "mxq")
    x[0, :32] = 0  # a zero block
    X = fp8.mx_quantize(x.cuda(), fmt)
    torch.cuda.synchronize()
    q, e = oracle.mx_quantize(workloads.bits(x), fmt)
    assert np.array_equal(X.q.cpu().numpy(), q)
    assert np.array_equal(sf_exponents(X.sf, rows, cols), e)
    G = 2 * ((rows + 255) // 256)
    b = X.sf.cpu().numpy().reshape(cols // 128, G, 512)
    for g in range(G):
        for rr in range(128):
            if 128 * g + rr >= rows:  # rows beyond the matrix: scale 1
                assert np.all(b[:, g, (rr % 32) * 16 + (rr // 32) * 4 + np.arange(4)] == 127)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rows,cols", [(256, 200), (128, 8), (384, 264)])
def test_mx_quantize_transposed_bit_exact(fp8, fmt, rows, cols):
    x = workloads.normal_bf16((rows, cols), 92, "mxt", std=0.5)
    X = fp8.mx_quantize(x.cuda(), fmt, transpose=True)
    torch.cuda.synchronize()
    q, e = oracle.mx_quantize(workloads.bits(x), fmt, transpose=True)
    assert X.q.shape == (cols, rows)
    assert np.array_equal(X.q.cpu().numpy(), q)
    assert np.array_equal(sf_exponents(X.sf, cols, rows), e)


def mx_both(fp8, a, b, fa, fb):
    A, B = fp8.mx_quantize(a.cuda(), fa), fp8.mx_quantize(b.cuda(), fb)
    qa, ea = oracle.mx_quantize(workloads.bits(a), fa)
    qb, eb = oracle.mx_quantize(workloads.bits(b), fb)
    return A, B, (qa, ea, fa), (qb, eb, fb)


SHAPES = [(256, 256, 256), (1, 1, 128), (300, 520, 384), (129, 257, 128), (513, 769, 640)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_mx_fprop_vs_oracle(fp8, M, N, K, epi):
    x = workloads.normal_bf16((M, K), 93, "x")
    w = workloads.normal_bf16((N, K), 93, "w", std=0.1)
    bias = workloads.normal_bf16((N,), 93, "b", std=0.1)
    A, B, oa, ob = mx_both(fp8, x, w, E4M3, E4M3)
    Y, Z = fp8.mx_gemm_fprop(A, B, bias.cuda() if epi else None, epi=epi)
    torch.cuda.synchronize()
    acc, S = oracle.mx_gemm(*oa, *ob)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(bias) if epi else None, gelu_on=(epi == 2))
    y = bf16_to_f64(Y)
    gain = MAX_DGELU if epi == 2 else 1.0
    assert_within(y, Yo, gain * FULL_C * S + bf16_ulp(np.maximum(np.abs(y), np.abs(Yo))) + 1e-5 * np.abs(Zo), "Y")
    if epi == 2:
        z = bf16_to_f64(Z)
        assert_within(z, Zo, FULL_C * S + bf16_ulp(np.maximum(np.abs(z), np.abs(Zo))), "Z")


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_mx_dgrad_vs_oracle(fp8, M, N, K):
    dy = workloads.normal_bf16((M, K), 94, "dy", std=1e-2)
    w = workloads.normal_bf16((N, K), 94, "w", std=0.02)
    z = workloads.normal_bf16((M, N), 94, "z", std=2.0)
    A, B, oa, ob = mx_both(fp8, dy, w, E5M2, E4M3)
    dZ, bg = fp8.mx_gemm_dgrad(A, B, z.cuda(), epi=4)
    torch.cuda.synchronize()
    acc, S = oracle.mx_gemm(*oa, *ob)
    dzo = oracle.dgrad_epilogue(acc, workloads.bits(z))
    zf = bf16_to_f64(z)
    g = np.abs(oracle.dgelu(zf))
    ev = np.abs(acc) * dgelu_eval_bound(zf)
    d = bf16_to_f64(dZ)
    assert_within(d, dzo, g * FULL_C * S + ev + bf16_ulp(np.maximum(np.abs(d), np.abs(dzo))), "dZ")
    n_tiles = (M + 127) // 128
    bbound = (g * FULL_C * S + ev).sum(axis=0) + (8 + 4 * n_tiles) * 2.0 ** -24 * np.abs(dzo).sum(axis=0) + 1e-30
    assert_within(bg.cpu().double().numpy(), oracle.colsum(dzo), bbound, "bgrad")


@pytest.mark.parametrize("M,N,K", SHAPES + [(1024, 768, 8192)])
@pytest.mark.parametrize("accumulate", [True, False])
def test_mx_wgrad_vs_oracle(fp8, M, N, K, accumulate):
    a = workloads.normal_bf16((M, K), 95, "a", std=0.02)
    b = workloads.normal_bf16((N, K), 95, "b", std=0.02)
    A, B, oa, ob = mx_both(fp8, a, b, E5M2, E4M3)
    pre = workloads.normal_f32((M, N), 95, "pre", std=1e-3)
    out = pre.clone().cuda() if accumulate else torch.full((M, N), float("nan"), device="cuda")
    fp8.mx_gemm_wgrad(A, B, out, accumulate=accumulate)
    torch.cuda.synchronize()
    rows = None if M * N <= 600 * 800 else np.arange(0, M, 7)
    acc, S = oracle.mx_gemm(*oa, *ob, rows=rows)
    p = pre.double().numpy() if rows is None else pre.double().numpy()[rows]
    want = oracle.wgrad(acc, p if accumulate else None)
    got = out.cpu().double().numpy() if rows is None else out.cpu().double().numpy()[rows]
    assert_within(got, want, FULL_C * S + f32_ulp(want), "out")


def test_mx_gemm_bitwise_repeatable(fp8):
    a = workloads.normal_bf16((2048, 4096), 96, "a", std=0.02).cuda()
    b = workloads.normal_bf16((6144, 4096), 96, "b", std=0.02).cuda()
    A, B = fp8.mx_quantize(a, E4M3), fp8.mx_quantize(b, E4M3)
    ref = torch.empty(2048, 6144, device="cuda")
    fp8.mx_gemm_wgrad(A, B, ref, accumulate=False)
    for _ in range(3):
        out = torch.empty_like(ref)
        fp8.mx_gemm_wgrad(A, B, out, accumulate=False)
        assert torch.equal(out, ref)
