"""The CTA-pair GEMMs (MXFP8 and per-tensor scaling) at the training step's
full sizes (tokens 8192, in 4096, out 14336), in the launch configuration the
bench times: every pair walks many 256 x 256 tiles, so the accumulator
hand-off between tiles, the operand and scale-slot rings wrapping across tiles
and (MXFP8) the scale-copy warp all run many times per launch.  Outputs are
checked on sampled rows and columns (always the first and last, so the ragged
last tile is included) against the oracle, with the bounds of the small-shape
tests; the bias gradient on a few columns over all rows.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import FULL_C, MAX_DGELU, assert_within, bf16_to_f64, bf16_ulp, dgelu_eval_bound, f32_ulp, sample_indices

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
TS = workloads.TRAIN_STEP


def _sel(t, ri, ci):
    return t[torch.from_numpy(ri).cuda()][:, torch.from_numpy(ci).cuda()]


def _dz_bounds(acc, S, z_bits, d, dzo):
    zf = oracle.bf16_to_f64(z_bits)
    g = np.abs(oracle.dgelu(zf))
    ev = np.abs(acc) * dgelu_eval_bound(zf)
    return g * FULL_C * S + ev, g * FULL_C * S + ev + bf16_ulp(np.maximum(np.abs(d), np.abs(dzo)))


# ------------------------------------------------------------------- MXFP8 ----

def test_mx_fprop_full_size(fp8):
    m, k, n = TS["m"], TS["k"], TS["n"]
    x = workloads.normal_bf16((m, k), 1702, "X")
    w = workloads.normal_bf16((n, k), 1702, "W", std=0.02)
    b = workloads.normal_bf16((n,), 1702, "b", std=0.02)
    X, W = fp8.mx_quantize(x.cuda(), E4M3), fp8.mx_quantize(w.cuda(), E4M3)
    Y, Z = fp8.mx_gemm_fprop(X, W, b.cuda(), fp8.EPI_BIAS_GELU)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    ri, ci = sample_indices(m, 48, 11), sample_indices(n, 48, 12)
    qa, ea = oracle.mx_quantize(workloads.bits(x[ri]), E4M3)
    qb, eb = oracle.mx_quantize(workloads.bits(w[ci]), E4M3)
    acc, S = oracle.mx_gemm(qa, ea, E4M3, qb, eb, E4M3)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(b), cols=ci)
    y, z = bf16_to_f64(_sel(Y, ri, ci)), bf16_to_f64(_sel(Z, ri, ci))
    assert_within(y, Yo, MAX_DGELU * FULL_C * S + bf16_ulp(np.maximum(abs(y), abs(Yo))) + 1e-5 * abs(Zo), "Y")
    assert_within(z, Zo, FULL_C * S + bf16_ulp(np.maximum(abs(z), abs(Zo))), "Z")


def test_mx_dgrad_full_size(fp8):
    m, k, n = TS["m"], TS["k"], TS["n"]
    dy = workloads.normal_bf16((m, k), 1703, "dY", std=1e-2)
    w = workloads.normal_bf16((n, k), 1703, "W", std=0.02)
    z = workloads.normal_bf16((m, n), 1703, "Zin", std=1.0)
    DY, W = fp8.mx_quantize(dy.cuda(), E5M2), fp8.mx_quantize(w.cuda(), E4M3)
    dZ, bg = fp8.mx_gemm_dgrad(DY, W, z.cuda(), fp8.EPI_DGELU_BGRAD)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    # dZ on sampled columns over every row, so the same columns give the bias gradient
    ci = sample_indices(n, 8, 13)
    qa, ea = oracle.mx_quantize(workloads.bits(dy), E5M2)
    qb, eb = oracle.mx_quantize(workloads.bits(w[ci]), E4M3)
    acc, S = oracle.mx_gemm(qa, ea, E5M2, qb, eb, E4M3)
    zc = workloads.bits(z)[:, ci]
    dzo = oracle.dgrad_epilogue(acc, zc)
    d = bf16_to_f64(dZ[:, torch.from_numpy(ci).cuda()])
    per_elt, bound = _dz_bounds(acc, S, zc, d, dzo)
    assert_within(d, dzo, bound, "dZ")
    bbound = per_elt.sum(axis=0) + (8 + 4 * (m // 128)) * 2.0 ** -24 * np.abs(dzo).sum(axis=0)
    assert_within(bg[torch.from_numpy(ci).cuda()].cpu().double().numpy(), oracle.colsum(dzo), bbound, "bgrad")


def test_mx_wgrad_full_size(fp8):
    # dW [n][k] += dZ^T X with both operands cast down their token columns
    m, k, n = TS["m"], TS["k"], TS["n"]
    dz = workloads.normal_bf16((m, n), 1704, "dZin", std=1e-2)
    x = workloads.normal_bf16((m, k), 1704, "X")
    DZT = fp8.mx_quantize(dz.cuda(), E5M2, transpose=True)   # [n][m]
    XT = fp8.mx_quantize(x.cuda(), E4M3, transpose=True)     # [k][m]
    pre = workloads.normal_f32((n, k), 1704, "dWpre", std=1e-3)
    dW = pre.cuda()
    fp8.mx_gemm_wgrad(DZT, XT, dW)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    ri, ci = sample_indices(n, 40, 14), sample_indices(k, 40, 15)
    qa, ea = oracle.mx_quantize(workloads.bits(dz[:, ri]), E5M2, transpose=True)
    qb, eb = oracle.mx_quantize(workloads.bits(x[:, ci]), E4M3, transpose=True)
    acc, S = oracle.mx_gemm(qa, ea, E5M2, qb, eb, E4M3)
    want = oracle.wgrad(acc, pre.double().numpy()[np.ix_(ri, ci)])
    got = _sel(dW, ri, ci).cpu().double().numpy()
    assert_within(got, want, FULL_C * S + f32_ulp(want), "dW")


# -------------------------------------------------------------- per-tensor ----

def _tensor_cast(fp8, t, fmt):
    amax = float(np.abs(t.float().numpy()).max())
    dev_amax = torch.tensor([amax], dtype=torch.float32, device="cuda")
    q, _ = fp8.tensor_quantize(t.cuda(), fmt, dev_amax)
    return q, amax


def test_tensor_dgrad_full_size(fp8):
    m, k, n = TS["m"], TS["k"], TS["n"]
    dy = workloads.normal_bf16((m, k), 1705, "dY", std=1e-2)
    w = workloads.normal_bf16((n, k), 1705, "W", std=0.02)
    z = workloads.normal_bf16((m, n), 1705, "Zin", std=1.0)
    (DY, am_dy), (W, am_w) = _tensor_cast(fp8, dy, E5M2), _tensor_cast(fp8, w, E4M3)
    dZ, bg = fp8.tensor_gemm_dgrad(DY, W, z.cuda(), epi=fp8.EPI_DGELU_BGRAD)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    ci = sample_indices(n, 8, 16)
    qa, sa, _ = oracle.tensor_quantize(workloads.bits(dy), E5M2, am_dy)
    qb, sb, _ = oracle.tensor_quantize(workloads.bits(w[ci]), E4M3, am_w)
    acc, S = oracle.tensor_gemm(qa, sa, E5M2, qb, sb, E4M3)
    zc = workloads.bits(z)[:, ci]
    dzo = oracle.dgrad_epilogue(acc, zc)
    d = bf16_to_f64(dZ[:, torch.from_numpy(ci).cuda()])
    per_elt, bound = _dz_bounds(acc, S, zc, d, dzo)
    assert_within(d, dzo, bound, "dZ")
    bbound = per_elt.sum(axis=0) + (8 + 4 * (m // 128)) * 2.0 ** -24 * np.abs(dzo).sum(axis=0)
    assert_within(bg[torch.from_numpy(ci).cuda()].cpu().double().numpy(), oracle.colsum(dzo), bbound, "bgrad")


def test_tensor_wgrad_full_size(fp8):
    m, k, n = TS["m"], TS["k"], TS["n"]
    dz = workloads.normal_bf16((m, n), 1706, "dZin", std=1e-2)
    x = workloads.normal_bf16((m, k), 1706, "X")
    am_dz = float(np.abs(dz.float().numpy()).max())
    am_x = float(np.abs(x.float().numpy()).max())
    _, DZT = fp8.tensor_quantize(dz.cuda(), E5M2, torch.tensor([am_dz], device="cuda"), rows=False, cols=True)
    _, XT = fp8.tensor_quantize(x.cuda(), E4M3, torch.tensor([am_x], device="cuda"), rows=False, cols=True)
    pre = workloads.normal_f32((n, k), 1706, "dWpre", std=1e-3)
    dW = pre.cuda()
    fp8.tensor_gemm_wgrad(DZT, XT, dW)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    ri, ci = sample_indices(n, 40, 17), sample_indices(k, 40, 18)
    qa, sa, _ = oracle.tensor_quantize(workloads.bits(dz[:, ri]), E5M2, am_dz, transpose=True)
    qb, sb, _ = oracle.tensor_quantize(workloads.bits(x[:, ci]), E4M3, am_x, transpose=True)
    acc, S = oracle.tensor_gemm(qa, sa, E5M2, qb, sb, E4M3)
    want = oracle.wgrad(acc, pre.double().numpy()[np.ix_(ri, ci)])
    got = _sel(dW, ri, ci).cpu().double().numpy()
    assert_within(got, want, FULL_C * S + f32_ulp(want), "dW")


def test_mx_input_grad_full_size(fp8):
    # dX = dZ W on MXFP8 operands: dZ cast by rows, W down its columns
    m, k, n = TS["m"], TS["k"], TS["n"]
    dz = workloads.normal_bf16((m, n), 1707, "dz", std=1e-2)
    w = workloads.normal_bf16((n, k), 1707, "w", std=0.02)
    A = fp8.mx_quantize(dz.cuda(), E5M2)
    Bt = fp8.mx_quantize(w.cuda(), E4M3, transpose=True)
    dX, _ = fp8.mx_gemm_fprop(A, Bt, None, fp8.EPI_NONE, want_aux=False)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    ri, ci = sample_indices(m, 40, 19), sample_indices(k, 40, 20)
    qa, ea = oracle.mx_quantize(workloads.bits(dz[ri]), E5M2)
    qb, eb = oracle.mx_quantize(workloads.bits(w[:, ci]), E4M3, transpose=True)
    acc, S = oracle.mx_gemm(qa, ea, E5M2, qb, eb, E4M3)
    got = bf16_to_f64(_sel(dX, ri, ci))
    assert_within(got, acc, FULL_C * S + bf16_ulp(np.maximum(np.abs(got), np.abs(acc))), "dX")
