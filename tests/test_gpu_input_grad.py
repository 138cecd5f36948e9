"""The layer's input gradient dX = dZ W (bf16, m x k) through the C ABI vs the
oracle: dZ cast by rows (e5m2, blocks along the n output features), W cast
down its columns (e4m3, blocks along n) to the k x n operand, then the plain
NT GEMM without an epilogue -- the backward GEMM that contracts over the
output features ("How can we use te.Linear with weight parallel?").

Bound: |gpu - oracle| <= 2e-3 * S (S = sum_n |dz_in w_nk| of the dequantized
operands) + one bf16 ulp.  Shapes with ragged m and k.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import FULL_C, assert_within, bf16_to_f64, bf16_ulp

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1


@pytest.mark.parametrize("m,k,n", [(300, 264, 384), (129, 1000, 256), (1024, 520, 640)])
def test_input_grad_vs_oracle(fp8, m, k, n):
    dz = workloads.normal_bf16((m, n), 71, "dz", std=1e-2)
    w = workloads.normal_bf16((n, k), 71, "w", std=0.02)
    A = fp8.quantize(dz.cuda(), E5M2)
    Bt = fp8.quantize(w.cuda(), E4M3, transpose=True)
    assert Bt.q.shape == (k, n)
    dX, _ = fp8.gemm_fprop(A, Bt, None, fp8.EPI_NONE)
    torch.cuda.synchronize()
    assert dX.shape == (m, k)
    qa, sa = oracle.quantize(workloads.bits(dz), E5M2)
    qb, sb = oracle.quantize(workloads.bits(w), E4M3, transpose=True)
    acc, S = oracle.gemm(qa, sa, E5M2, qb, sb, E4M3)
    got = bf16_to_f64(dX)
    assert_within(got, acc, FULL_C * S + bf16_ulp(np.maximum(np.abs(got), np.abs(acc))), "dX")


def test_train_step_input_grad_matches_direct_call(fp8):
    # the training step's dX is the same GEMM on the same casts: bit-identical
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    m, k, n = 256, 384, 512
    X = workloads.normal_bf16((m, k), 72, "x").cuda()
    W = workloads.normal_bf16((n, k), 72, "w", std=0.02).cuda()
    b = workloads.normal_bf16((n,), 72, "b", std=0.02).cuda()
    dY = workloads.normal_bf16((m, k), 72, "dy", std=1e-2).cuda()
    step = LinearTrainStep(m, k, n)
    step.step(X, W, b, dY)
    dX = step.input_grad(W).clone()
    A = fp8.quantize(step.dZ, E5M2)
    Bt = fp8.quantize(W, E4M3, transpose=True)
    ref, _ = fp8.gemm_fprop(A, Bt, None, fp8.EPI_NONE)
    torch.cuda.synchronize()
    assert torch.equal(dX, ref)


def test_train_step_with_two_way_casts_is_bit_identical(fp8):
    # input_grad=True casts X, W and dZ both ways in one read each; every
    # output of the step and dX must equal the step built from single casts
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    m, k, n = 384, 256, 640
    X = workloads.normal_bf16((m, k), 73, "x").cuda()
    W = workloads.normal_bf16((n, k), 73, "w", std=0.02).cuda()
    b = workloads.normal_bf16((n,), 73, "b", std=0.02).cuda()
    dY = workloads.normal_bf16((m, k), 73, "dy", std=1e-2).cuda()
    plain, fused = LinearTrainStep(m, k, n), LinearTrainStep(m, k, n, input_grad=True)
    # and dZ's row codes for dX written by the data-gradient GEMM's epilogue instead
    by_epilogue = LinearTrainStep(m, k, n, input_grad=True, dz_rows="dgrad")
    operand = LinearTrainStep(m, k, n, input_grad=True, dz_rows="dgrad", bias_grad="operand")
    outs = []
    for st in (plain, fused, by_epilogue):
        st.step(X, W, b, dY)
        outs.append((st.Y.clone(), st.Z.clone(), st.dZ.clone(), st.db.clone(), st.dW.clone(),
                     st.input_grad(W).clone()))
    torch.cuda.synchronize()
    for o in outs[1:]:
        for a, c in zip(outs[0], o):
            assert torch.equal(a, c)
    # the operand-reduced db differs (it sums the fp8 values); every other output agrees
    operand.step(X, W, b, dY)
    dx = operand.input_grad(W)
    torch.cuda.synchronize()
    for a, c in zip(outs[0][:3] + outs[0][4:], (operand.Y, operand.Z, operand.dZ, operand.dW, dx)):
        assert torch.equal(a, c)


def test_cached_weight_steps_are_bit_identical(fp8):
    # two micro-batch steps with W cast once up front equal two steps that
    # cast W each time (every output, the accumulated dW and dX)
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    m, k, n = 256, 384, 512
    W = workloads.normal_bf16((n, k), 74, "w", std=0.02).cuda()
    b = workloads.normal_bf16((n,), 74, "b", std=0.02).cuda()
    batches = [(workloads.normal_bf16((m, k), 75 + i, "x").cuda(),
                workloads.normal_bf16((m, k), 75 + i, "dy", std=1e-2).cuda()) for i in range(2)]
    outs = []
    for cached in (False, True):
        st = LinearTrainStep(m, k, n, input_grad=True)
        if cached:
            st.cache_weight(W)
            assert st.KERNELS_PER_STEP == 7
        for X, dY in batches:
            st.step(X, W, b, dY)
        outs.append([t.clone() for t in (st.Y, st.Z, st.dZ, st.db, st.dW, st.input_grad(W))])
    torch.cuda.synchronize()
    for a, c in zip(*outs):
        assert torch.equal(a, c)


def test_mx_step_input_grad_vs_oracle(fp8):
    from fp8_linear_layer_gb300.linear import MxLinearTrainStep
    m, k, n = 256, 384, 512
    X = workloads.normal_bf16((m, k), 76, "x").cuda()
    W = workloads.normal_bf16((n, k), 76, "w", std=0.02)
    b = workloads.normal_bf16((n,), 76, "b", std=0.02).cuda()
    dY = workloads.normal_bf16((m, k), 76, "dy", std=1e-2).cuda()
    st = MxLinearTrainStep(m, k, n)
    st.step(X, W.cuda(), b, dY)
    dX = st.input_grad(W.cuda())
    torch.cuda.synchronize()
    qa, ea = oracle.mx_quantize(workloads.bits(st.dZ.cpu()), E5M2)
    qb, eb = oracle.mx_quantize(workloads.bits(W), E4M3, transpose=True)
    assert np.array_equal(st.dZq.q.cpu().numpy(), qa) and np.array_equal(st.WTq.q.cpu().numpy(), qb)
    acc, S = oracle.mx_gemm(qa, ea, E5M2, qb, eb, E4M3)
    got = bf16_to_f64(dX)
    assert_within(got, acc, FULL_C * S + bf16_ulp(np.maximum(np.abs(got), np.abs(acc))), "dX")


def test_per_tensor_step_input_grad_vs_oracle(fp8):
    from fp8_linear_layer_gb300.linear import TensorLinearTrainStep
    m, k, n = 256, 384, 512
    X = workloads.normal_bf16((m, k), 77, "x").cuda()
    W = workloads.normal_bf16((n, k), 77, "w", std=0.02)
    b = workloads.normal_bf16((n,), 77, "b", std=0.02).cuda()
    dY = workloads.normal_bf16((m, k), 77, "dy", std=1e-2).cuda()
    st = TensorLinearTrainStep(m, k, n)
    st.step(X, W.cuda(), b, dY)
    dX = st.input_grad(W.cuda())
    torch.cuda.synchronize()
    dz = st.dZ.cpu()
    qa, sa, _ = oracle.tensor_quantize(workloads.bits(dz), E5M2, float(dz.abs().max()))
    qb, sb, _ = oracle.tensor_quantize(workloads.bits(W), E4M3, float(W.abs().max()), transpose=True)
    assert np.array_equal(st.dZq.q.cpu().numpy(), qa) and np.array_equal(st.WTq.q.cpu().numpy(), qb)
    acc, S = oracle.tensor_gemm(qa, sa, E5M2, qb, sb, E4M3)
    got = bf16_to_f64(dX)
    assert_within(got, acc, FULL_C * S + bf16_ulp(np.maximum(np.abs(got), np.abs(acc))), "dX")


def test_input_grad_full_size(fp8):
    # dX = dZ W at the training step's sizes: 8192 x 4096, contracted over the
    # 14336 output features (112 K blocks per tile); sampled rows and columns
    from helpers import sample_indices
    m, k, n = workloads.TRAIN_STEP["m"], workloads.TRAIN_STEP["k"], workloads.TRAIN_STEP["n"]
    dz = workloads.normal_bf16((m, n), 72, "dz", std=1e-2)
    w = workloads.normal_bf16((n, k), 72, "w", std=0.02)
    A = fp8.quantize(dz.cuda(), E5M2)
    Bt = fp8.quantize(w.cuda(), E4M3, transpose=True)
    dX, _ = fp8.gemm_fprop(A, Bt, None, fp8.EPI_NONE)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    ri, ci = sample_indices(m, 40, 21), sample_indices(k, 40, 22)
    qa, sa = oracle.quantize(workloads.bits(dz[ri]), E5M2)
    qb, sb = oracle.quantize(workloads.bits(w[:, ci]), E4M3, transpose=True)
    acc, S = oracle.gemm(qa, sa, E5M2, qb, sb, E4M3)
    got = bf16_to_f64(dX[torch.from_numpy(ri).cuda()][:, torch.from_numpy(ci).cuda()])
    assert_within(got, acc, FULL_C * S + bf16_ulp(np.maximum(np.abs(got), np.abs(acc))), "dX")
