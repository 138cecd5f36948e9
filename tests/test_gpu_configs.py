"""Parity at the full workload sizes, on sampled outputs the oracle computes one
by one (the oracle quantizes only the rows / columns it needs: the cast is
row-local, and column-local in its transposed form).

Workloads: the dense and grouped weight-gradient tables of "Weight gradient
kernels for dense and MoE models", the 256^3 case with bias + GELU, and the
GEMMs of one linear-layer training step (tokens 8192, in 4096, out 14336).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import (FULL_C, MAX_DGELU, assert_within, bf16_to_f64, bf16_ulp, dgelu_eval_bound, f32_ulp,
                     sample_indices)

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1


def oq_rows(x, idx, fmt):
    return oracle.quantize(workloads.bits(x[torch.from_numpy(idx)]), fmt)


def oq_cols(x, idx, fmt):
    return oracle.quantize(workloads.bits(x[:, torch.from_numpy(idx)].contiguous()), fmt, transpose=True)


def test_tiny_256_fprop_and_accumulate(fp8):
    n = 256
    x = workloads.normal_bf16((n, n), 1000, "x")
    w = workloads.normal_bf16((n, n), 1000, "w")
    b = workloads.normal_bf16((n,), 1000, "b", std=0.1)
    X, W = fp8.quantize(x.cuda(), E4M3), fp8.quantize(w.cuda(), E4M3)
    Y, Z = fp8.gemm_fprop(X, W, b.cuda(), fp8.EPI_BIAS_GELU)
    pre = workloads.normal_f32((n, n), 1000, "pre")
    out = pre.clone().cuda()
    fp8.gemm_wgrad(X, W, out)
    torch.cuda.synchronize()
    qx, sx = oracle.quantize(workloads.bits(x), E4M3)
    qw, sw = oracle.quantize(workloads.bits(w), E4M3)
    acc, S = oracle.gemm(qx, sx, E4M3, qw, sw, E4M3)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(b))
    y = bf16_to_f64(Y)
    assert_within(y, Yo, MAX_DGELU * FULL_C * S + bf16_ulp(np.maximum(abs(y), abs(Yo))) + 1e-6 * abs(Zo), "Y")
    o = out.cpu().double().numpy()
    want = oracle.wgrad(acc, pre.double().numpy())
    assert_within(o, want, FULL_C * S + f32_ulp(want), "out += X W^T")


@pytest.mark.parametrize("K", workloads.DENSE_WGRAD_K)
@pytest.mark.parametrize("M,N", workloads.DENSE_WGRAD_MN)
def test_dense_wgrad_table_shapes(fp8, M, N, K):
    seed = 2000 + M + N + K
    a = workloads.normal_bf16((M, K), seed, "a", std=0.02)
    b = workloads.normal_bf16((N, K), seed, "b", std=0.02)
    pre = workloads.normal_f32((M, N), seed, "pre", std=1e-3)
    A, B = fp8.quantize(a.cuda(), E4M3), fp8.quantize(b.cuda(), E4M3)
    out = pre.cuda()
    fp8.gemm_wgrad(A, B, out)
    ri = sample_indices(M, 40, seed)
    ci = sample_indices(N, 40, seed + 1)
    got = out[torch.from_numpy(ri).cuda()][:, torch.from_numpy(ci).cuda()].cpu().double().numpy()
    qa, sa = oq_rows(a, ri, E4M3)
    qb, sb = oq_rows(b, ci, E4M3)
    acc, S = oracle.gemm(qa, sa, E4M3, qb, sb, E4M3)
    want = oracle.wgrad(acc, pre.double().numpy()[np.ix_(ri, ci)])
    assert_within(got, want, FULL_C * S + f32_ulp(want), "dense wgrad %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("G,M,N,Kavg", workloads.GROUPED_WGRAD)
def test_grouped_wgrad_table_shapes(fp8, G, M, N, Kavg):
    seed = 3000 + G + M + Kavg
    ks = workloads.moe_group_sizes(G, G * Kavg, seed)
    tot = sum(ks)
    a = workloads.normal_bf16((M, tot), seed, "a", std=0.02)
    b = workloads.normal_bf16((N, tot), seed, "b", std=0.02)
    A, B = fp8.quantize(a.cuda(), E4M3), fp8.quantize(b.cuda(), E4M3)
    out = torch.zeros((G, M, N), device="cuda")
    fp8.grouped_wgrad(A, B, ks, out)
    ri = sample_indices(M, 24, seed)
    ci = sample_indices(N, 24, seed + 1)
    qa, sa = oq_rows(a, ri, E4M3)
    qb, sb = oq_rows(b, ci, E4M3)
    want, S = oracle.grouped_wgrad(qa, sa, E4M3, qb, sb, E4M3, ks)
    got = out[:, torch.from_numpy(ri).cuda()][:, :, torch.from_numpy(ci).cuda()].cpu().double().numpy()
    assert_within(got, want, FULL_C * S + f32_ulp(want), "grouped wgrad G=%d" % G)


# A skewed expert split of 16384 tokens (60%, none, 25%, 15%, in 128-token
# blocks), the largest group placed first and second-to-last in turn: the host
# schedules groups longest first, and results must not depend on the order.
SKEWED = [[9856, 0, 4096, 2432], [2432, 0, 4096, 9856]]


@pytest.mark.parametrize("ks", SKEWED)
def test_grouped_wgrad_skewed_split(fp8, ks):
    G, M, N = len(ks), 2048, 7168
    seed = 3500 + ks[0]
    tot = sum(ks)
    a = workloads.normal_bf16((M, tot), seed, "a", std=0.02)
    b = workloads.normal_bf16((N, tot), seed, "b", std=0.02)
    A, B = fp8.quantize(a.cuda(), E4M3), fp8.quantize(b.cuda(), E4M3)
    pre = workloads.normal_f32((G, M, N), seed, "pre", std=1e-3)
    out = pre.cuda()
    fp8.grouped_wgrad(A, B, ks, out)
    ri = sample_indices(M, 24, seed)
    ci = sample_indices(N, 24, seed + 1)
    qa, sa = oq_rows(a, ri, E4M3)
    qb, sb = oq_rows(b, ci, E4M3)
    p = pre.double().numpy()[:, ri][:, :, ci]
    want, S = oracle.grouped_wgrad(qa, sa, E4M3, qb, sb, E4M3, ks, prefill=p)
    got = out[:, torch.from_numpy(ri).cuda()][:, :, torch.from_numpy(ci).cuda()].cpu().double().numpy()
    assert_within(got, want, FULL_C * S + f32_ulp(want), "skewed grouped wgrad %s" % ks)
    assert np.array_equal(out[1].cpu().numpy(), pre[1].numpy())  # the empty group is untouched


TS = workloads.TRAIN_STEP


def test_train_step_fprop_full_size(fp8):
    m, k, n = TS["m"], TS["k"], TS["n"]
    x = workloads.normal_bf16((m, k), 1002, "X")
    w = workloads.normal_bf16((n, k), 1002, "W", std=0.02)
    b = workloads.normal_bf16((n,), 1002, "b", std=0.02)
    X, W = fp8.quantize(x.cuda(), E4M3), fp8.quantize(w.cuda(), E4M3)
    Y, Z = fp8.gemm_fprop(X, W, b.cuda(), fp8.EPI_BIAS_GELU)
    ri, ci = sample_indices(m, 48, 1), sample_indices(n, 48, 2)
    qa, sa = oq_rows(x, ri, E4M3)
    qb, sb = oq_rows(w, ci, E4M3)
    acc, S = oracle.gemm(qa, sa, E4M3, qb, sb, E4M3)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(b), cols=ci)
    sel = (torch.from_numpy(ri).cuda(), torch.from_numpy(ci).cuda())
    y = bf16_to_f64(Y[sel[0]][:, sel[1]])
    z = bf16_to_f64(Z[sel[0]][:, sel[1]])
    assert_within(y, Yo, MAX_DGELU * FULL_C * S + bf16_ulp(np.maximum(abs(y), abs(Yo))) + 1e-6 * abs(Zo), "Y")
    assert_within(z, Zo, FULL_C * S + bf16_ulp(np.maximum(abs(z), abs(Zo))), "Z")


def test_train_step_dgrad_full_size(fp8):
    m, k, n = TS["m"], TS["k"], TS["n"]
    dy = workloads.normal_bf16((m, k), 1002, "dY", std=1e-2)
    w = workloads.normal_bf16((n, k), 1002, "W", std=0.02)
    z = workloads.normal_bf16((m, n), 1002, "Zin", std=1.0)
    DY, W = fp8.quantize(dy.cuda(), E5M2), fp8.quantize(w.cuda(), E4M3)
    dZ, bg = fp8.gemm_dgrad(DY, W, z.cuda(), fp8.EPI_DGELU_BGRAD)
    ri, ci = sample_indices(m, 48, 3), sample_indices(n, 48, 4)
    qa, sa = oq_rows(dy, ri, E5M2)
    qb, sb = oq_rows(w, ci, E4M3)
    acc, S = oracle.gemm(qa, sa, E5M2, qb, sb, E4M3)
    zs = workloads.bits(z)[np.ix_(ri, ci)]
    dzo = oracle.dgrad_epilogue(acc, zs)
    zf = oracle.bf16_to_f64(zs)
    g = np.abs(oracle.dgelu(zf))
    d = bf16_to_f64(dZ[torch.from_numpy(ri).cuda()][:, torch.from_numpy(ci).cuda()])
    bound = g * FULL_C * S + np.abs(acc) * dgelu_eval_bound(zf) + bf16_ulp(np.maximum(abs(d), abs(dzo)))
    assert_within(d, dzo, bound, "dZ")
    # bias gradient of a few columns: all m rows by the oracle
    cb = ci[:6]
    qa_all, sa_all = oracle.quantize(workloads.bits(dy), E5M2)
    acc_c, S_c = oracle.gemm(qa_all, sa_all, E5M2, qb[:6], sb[:, :6], E4M3)
    zc = workloads.bits(z)[:, cb]
    dz_c = oracle.dgrad_epilogue(acc_c, zc)
    zcf = oracle.bf16_to_f64(zc)
    gc = np.abs(oracle.dgelu(zcf))
    bgo = oracle.colsum(dz_c)
    bound = ((gc * FULL_C * S_c + np.abs(acc_c) * dgelu_eval_bound(zcf)).sum(axis=0)
             + (8 + 4 * (m // 128)) * 2.0 ** -24 * np.abs(dz_c).sum(axis=0))
    assert_within(bg[torch.from_numpy(cb).cuda()].cpu().double().numpy(), bgo, bound, "bgrad")


def test_train_step_wgrad_full_size(fp8):
    m, k, n = TS["m"], TS["k"], TS["n"]
    dz = workloads.normal_bf16((m, n), 1002, "dZin", std=1e-2)
    x = workloads.normal_bf16((m, k), 1002, "X")
    DZT = fp8.quantize(dz.cuda(), E5M2, transpose=True)   # [n][m]
    XT = fp8.quantize(x.cuda(), E4M3, transpose=True)     # [k][m]
    pre = workloads.normal_f32((n, k), 1002, "dWpre", std=1e-3)
    dW = pre.cuda()
    fp8.gemm_wgrad(DZT, XT, dW)
    ri, ci = sample_indices(n, 40, 5), sample_indices(k, 40, 6)
    qa, sa = oq_cols(dz, ri, E5M2)
    qb, sb = oq_cols(x, ci, E4M3)
    acc, S = oracle.gemm(qa, sa, E5M2, qb, sb, E4M3)
    want = oracle.wgrad(acc, pre.double().numpy()[np.ix_(ri, ci)])
    got = dW[torch.from_numpy(ri).cuda()][:, torch.from_numpy(ci).cuda()].cpu().double().numpy()
    assert_within(got, want, FULL_C * S + f32_ulp(want), "dW")


def test_train_step_chain_small(fp8):
    """The whole step through LinearTrainStep at a small size, each output
    against the oracle run through the same step on its own intermediates.
    Where a GPU intermediate (bf16 Z, dZ) feeds the next GEMM, the bound adds
    the effect of a one-ulp difference in that intermediate."""
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    m, k, n = 512, 384, 640
    X = workloads.normal_bf16((m, k), 77, "X")
    W = workloads.normal_bf16((n, k), 77, "W", std=0.05)
    b = workloads.normal_bf16((n,), 77, "b", std=0.02)
    dY = workloads.normal_bf16((m, k), 77, "dY", std=1e-2)
    st = LinearTrainStep(m, k, n, bias_grad="dgrad")  # the epilogue's column sums
    st.step(X.cuda(), W.cuda(), b.cuda(), dY.cuda())
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    qx, sx = oracle.quantize(workloads.bits(X), E4M3)
    qw, sw = oracle.quantize(workloads.bits(W), E4M3)
    acc, S = oracle.gemm(qx, sx, E4M3, qw, sw, E4M3)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(b))
    y = bf16_to_f64(st.Y)
    assert_within(y, Yo, MAX_DGELU * FULL_C * S + bf16_ulp(np.maximum(abs(y), abs(Yo))) + 1e-6 * abs(Zo), "Y")
    zb = oracle.f64_to_bf16_array(Zo)  # the oracle's own rounding of its Z
    qd, sd = oracle.quantize(workloads.bits(dY), E5M2)
    acc2, S2 = oracle.gemm(qd, sd, E5M2, qw, sw, E4M3)
    dzo = oracle.dgrad_epilogue(acc2, zb)
    # |gelu''| <= 0.8: a Z differing by its bound + 1 ulp moves gelu' by at most 0.8 x that
    dz_z = 0.8 * (FULL_C * S + bf16_ulp(Zo)) * np.abs(acc2)
    zbf = oracle.bf16_to_f64(zb)
    g = np.abs(oracle.dgelu(zbf))
    d = bf16_to_f64(st.dZ)
    bound_dz = (g * FULL_C * S2 + dz_z + np.abs(acc2) * dgelu_eval_bound(zbf)
                + bf16_ulp(np.maximum(abs(d), abs(dzo))))
    assert_within(d, dzo, bound_dz, "dZ")
    assert_within(st.db.cpu().double().numpy(), oracle.colsum(dzo),
                  (g * FULL_C * S2 + dz_z).sum(0) + 24 * 2.0 ** -24 * np.abs(dzo).sum(0), "db")
    # dW: the oracle's weight-gradient operand is the transposed cast of the
    # GPU's stored bf16 dZ (the bytes the GPU's own cast read, as the data
    # gradient above reads the stored Z), so the element bound carries over
    # with no re-rounding of a neighbouring dZ into another e5m2 code
    qa, sa = oracle.quantize(workloads.bits(st.dZ), E5M2, transpose=True)
    qb, sb = oracle.quantize(workloads.bits(X), E4M3, transpose=True)
    acc3, S3 = oracle.gemm(qa, sa, E5M2, qb, sb, E4M3)
    got = st.dW.cpu().double().numpy()  # one step accumulated into zeros
    assert_within(got, acc3, FULL_C * S3 + f32_ulp(acc3), "dW")
