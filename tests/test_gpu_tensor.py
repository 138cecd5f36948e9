"""Per-tensor scaling through the C ABI vs the oracle.

Reading ("FP8 GEMM for the fprop should use fast accumulation": one scale per
operand tensor): the cast takes its amax from the caller -- the tensor's own
(current scaling) or the largest amax of earlier steps (delayed scaling,
values above it saturate) -- with inv = fl32(FMAX/amax), scale =
fl32(amax/FMAX), q = RNE-saturating fp8(fl32(x inv)); the GEMM accumulates
the raw fp8 products over all of K and multiplies once by sA sB.

Casts, amax and the history are compared bit for bit; the GEMMs within
2e-3 * S (S = sum_k |a_ik b_jk| of the dequantized operands) plus one ulp of
the output type, the epilogue terms as in test_gpu_gemm.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import FULL_C, MAX_DGELU, assert_within, bf16_to_f64, bf16_ulp, dgelu_eval_bound, f32_ulp

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
SHAPES = [(256, 256, 256), (1, 1, 128), (300, 520, 384), (129, 257, 128), (640, 1000, 1024), (513, 769, 640)]


def f32(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("shape", [(1, 8), (3, 200), (129, 1000), (1024, 4096)])
def test_amax_exact(fp8, shape):
    x = workloads.normal_bf16(shape, 500, "am", std=3.0)
    x[shape[0] - 1, shape[1] - 1] = -70.0  # the largest magnitude, negative, in the last element
    a = fp8.tensor_amax(x.cuda())
    torch.cuda.synchronize()
    assert a.item() == 70.0
    z = fp8.tensor_amax(torch.zeros(4, 16, dtype=torch.bfloat16, device="cuda"))
    e = fp8.tensor_amax(torch.zeros(0, 16, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert z.item() == 0.0 and e.item() == 0.0


def check_cast(fp8, x, fmt, amax, rows, cols, record):
    am_out = torch.full((1,), -1.0, device="cuda") if record else None
    qr, qc = fp8.tensor_quantize(x.cuda(), fmt, f32(amax), rows=rows, cols=cols, amax_out=am_out)
    torch.cuda.synchronize()
    xb = workloads.bits(x)
    for t, transpose in ((qr, False), (qc, True)):
        if t is None:
            continue
        qo, so, ao = oracle.tensor_quantize(xb, fmt, amax, transpose=transpose)
        q = t.q.cpu().numpy()
        assert np.array_equal(q, qo), "codes differ at %s" % (np.argwhere(q != qo)[:5].tolist(),)
        assert t.scale.cpu().numpy().view(np.uint32)[0] == np.float32(so).view(np.uint32)
        if record:
            assert am_out.item() == ao


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rows,cols", [(True, False), (False, True), (True, True)])
def test_cast_current_scaling(fp8, fmt, rows, cols):
    x = workloads.normal_bf16((384, 640), 510 + fmt, "cs", std=2.0)
    amax = float(np.abs(x.float().numpy()).max())
    check_cast(fp8, x, fmt, amax, rows, cols, record=True)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rows,cols", [(True, False), (False, True), (True, True)])
def test_cast_delayed_scaling_saturates(fp8, fmt, rows, cols):
    # an amax from the history below the tensor's own: codes saturate, the
    # recorded amax is the tensor's own
    x = workloads.normal_bf16((256, 384), 520 + fmt, "ds", std=1.0)
    amax = float(np.abs(x.float().numpy()).max()) / 3
    check_cast(fp8, x, fmt, amax, rows, cols, record=True)


@pytest.mark.parametrize("shape,rows,cols", [((128, 8), False, True), ((384, 136), False, True),
                                             ((7, 16), True, False), ((129, 1008), True, False)])
def test_cast_ragged_and_special(fp8, shape, rows, cols):
    x = workloads.normal_bf16(shape, 530, "rg", std=1.0).float()
    x[0, :] = 0.0
    x[1 % shape[0], : shape[1] // 2] = -0.0
    x[-1, -1] = 1e4
    xb = x.to(torch.bfloat16)
    check_cast(fp8, xb, E4M3, 8.0, rows, cols, record=True)  # 1e4 saturates
    check_cast(fp8, xb, E5M2, 0.0, rows, cols, record=False)  # amax 0: unit scale


def test_amax_history_matches_oracle(fp8):
    hist = torch.zeros(5, device="cuda")
    use = torch.empty(1, device="cuda")
    h_o = np.zeros(5, dtype=np.float32)
    for v in (3.0, 1.5, 7.25, 0.5, 0.25, 0.125, 0.0625, 2.0):
        fp8.amax_history_update(hist, f32(v), use)
        h_o, use_o = oracle.amax_history(h_o, v)
        torch.cuda.synchronize()
        assert np.array_equal(hist.cpu().numpy(), h_o) and use.item() == use_o


def quant_pair(fp8, a, b, fa, fb, shrink=1.0):
    """GPU operands cast with their own amax (times shrink, below 1 = saturating)
    and the oracle's operands from the same bf16 bytes."""
    am_a = float(np.abs(a.float().numpy()).max()) * shrink
    am_b = float(np.abs(b.float().numpy()).max()) * shrink
    A, _ = fp8.tensor_quantize(a.cuda(), fa, f32(am_a))
    B, _ = fp8.tensor_quantize(b.cuda(), fb, f32(am_b))
    qa, sa, _ = oracle.tensor_quantize(workloads.bits(a), fa, am_a)
    qb, sb, _ = oracle.tensor_quantize(workloads.bits(b), fb, am_b)
    return A, B, (qa, sa, fa), (qb, sb, fb)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("epi", [0, 1, 2])
def test_fprop_vs_oracle(fp8, M, N, K, epi):
    x = workloads.normal_bf16((M, K), 540, "x")
    w = workloads.normal_bf16((N, K), 540, "w", std=0.05)
    bias = workloads.normal_bf16((N,), 540, "b", std=0.1)
    A, B, oa, ob = quant_pair(fp8, x, w, E4M3, E4M3)
    Y, Z = fp8.tensor_gemm_fprop(A, B, bias.cuda() if epi else None, epi=epi)
    torch.cuda.synchronize()
    acc, S = oracle.tensor_gemm(*oa, *ob)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(bias) if epi else None, gelu_on=(epi == 2))
    y = bf16_to_f64(Y)
    gain = MAX_DGELU if epi == 2 else 1.0
    assert_within(y, Yo, gain * FULL_C * S + bf16_ulp(np.maximum(np.abs(y), np.abs(Yo))) + 1e-5 * np.abs(Zo), "Y")
    if epi == 2:
        z = bf16_to_f64(Z)
        assert_within(z, Zo, FULL_C * S + bf16_ulp(np.maximum(np.abs(z), np.abs(Zo))), "Z")


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("epi", [3, 4])
def test_dgrad_vs_oracle(fp8, M, N, K, epi):
    dy = workloads.normal_bf16((M, K), 550, "dy", std=1e-2)
    w = workloads.normal_bf16((N, K), 550, "w", std=0.02)
    z = workloads.normal_bf16((M, N), 550, "z", std=2.0)
    A, B, oa, ob = quant_pair(fp8, dy, w, E5M2, E4M3)
    dZ, bg = fp8.tensor_gemm_dgrad(A, B, z.cuda(), epi=epi)
    torch.cuda.synchronize()
    acc, S = oracle.tensor_gemm(*oa, *ob)
    dzo = oracle.dgrad_epilogue(acc, workloads.bits(z))
    zf = bf16_to_f64(z)
    g = np.abs(oracle.dgelu(zf))
    ev = np.abs(acc) * dgelu_eval_bound(zf)
    d = bf16_to_f64(dZ)
    assert_within(d, dzo, g * FULL_C * S + ev + bf16_ulp(np.maximum(np.abs(d), np.abs(dzo))), "dZ")
    if epi == 4:
        n_tiles = (M + 127) // 128
        bbound = (g * FULL_C * S + ev).sum(axis=0) + (8 + 4 * n_tiles) * 2.0 ** -24 * np.abs(dzo).sum(axis=0) + 1e-30
        assert_within(bg.cpu().double().numpy(), oracle.colsum(dzo), bbound, "bgrad")


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("accumulate", [True, False])
def test_wgrad_vs_oracle(fp8, M, N, K, accumulate):
    a = workloads.normal_bf16((M, K), 560, "a", std=0.02)
    b = workloads.normal_bf16((N, K), 560, "b", std=0.02)
    A, B, oa, ob = quant_pair(fp8, a, b, E5M2, E4M3)
    pre = workloads.normal_f32((M, N), 560, "pre", std=1e-3)
    out = pre.clone().cuda() if accumulate else torch.full((M, N), float("nan"), device="cuda")
    fp8.tensor_gemm_wgrad(A, B, out, accumulate=accumulate)
    torch.cuda.synchronize()
    acc, S = oracle.tensor_gemm(*oa, *ob)
    want = oracle.wgrad(acc, pre.double().numpy() if accumulate else None)
    got = out.cpu().double().numpy()
    assert np.all(np.isfinite(got))
    assert_within(got, want, FULL_C * S + f32_ulp(want), "out")


def test_saturated_operands_and_long_k(fp8):
    # delayed-scaling operands that saturate (amax from the history at half
    # the tensor's own) and K = 8192: the GEMM multiplies exactly what was cast
    M, N, K = 256, 512, 8192
    x = workloads.normal_bf16((M, K), 570, "x")
    w = workloads.normal_bf16((N, K), 570, "w", std=0.02)
    A, B, oa, ob = quant_pair(fp8, x, w, E4M3, E4M3, shrink=0.5)
    Y, _ = fp8.tensor_gemm_fprop(A, B, None, epi=0)
    torch.cuda.synchronize()
    acc, S = oracle.tensor_gemm(*oa, *ob)
    y = bf16_to_f64(Y)
    assert_within(y, acc, FULL_C * S + bf16_ulp(np.maximum(np.abs(y), np.abs(acc))), "Y")


def test_full_size_fprop_sampled(fp8):
    # the training step's forward GEMM, 8192 x 14336 x 4096, on sampled rows and columns
    m, k, n = 8192, 4096, 14336
    x = workloads.normal_bf16((m, k), 580, "x")
    w = workloads.normal_bf16((n, k), 580, "w", std=0.02)
    b = workloads.normal_bf16((n,), 580, "b", std=0.02)
    A, _ = fp8.tensor_quantize(x.cuda(), E4M3, fp8.tensor_amax(x.cuda()))
    B, _ = fp8.tensor_quantize(w.cuda(), E4M3, fp8.tensor_amax(w.cuda()))
    Y, Z = fp8.tensor_gemm_fprop(A, B, b.cuda(), epi=2)
    torch.cuda.synchronize()
    ri = np.array([0, 1, 127, 128, 4095, 5000, m - 1])
    ci = np.array([0, 255, 256, 7000, n - 2, n - 1])
    am_x = float(np.abs(x.float().numpy()).max())
    am_w = float(np.abs(w.float().numpy()).max())
    qa, sa, _ = oracle.tensor_quantize(workloads.bits(x[ri]), E4M3, am_x)
    qb, sb, _ = oracle.tensor_quantize(workloads.bits(w[ci]), E4M3, am_w)
    assert np.array_equal(A.q[torch.from_numpy(ri).cuda()].cpu().numpy(), qa)
    acc, S = oracle.tensor_gemm(qa, sa, E4M3, qb, sb, E4M3)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(b), cols=ci)
    y = bf16_to_f64(Y[torch.from_numpy(ri).cuda()][:, torch.from_numpy(ci).cuda()])
    assert_within(y, Yo, MAX_DGELU * FULL_C * S + bf16_ulp(np.maximum(np.abs(y), np.abs(Yo))) + 1e-5 * np.abs(Zo),
                  "Y")


def test_delayed_scaling_training_step(fp8):
    # step 1 casts with empty histories (unit scales) and records each tensor's
    # amax; step 2 casts with those: with the same inputs its forward equals
    # current scaling, and dZ^T is cast with the amax of step 1's dZ
    from fp8_linear_layer_gb300.linear import TensorLinearTrainStep
    m, k, n = 256, 384, 512
    X = workloads.normal_bf16((m, k), 590, "X")
    W = workloads.normal_bf16((n, k), 590, "W", std=0.05)
    b = workloads.normal_bf16((n,), 590, "b", std=0.02)
    dY = workloads.normal_bf16((m, k), 590, "dY", std=1e-2)
    st = TensorLinearTrainStep(m, k, n, scaling="delayed", history=4)
    Xd, Wd, bd, dYd = X.cuda(), W.cuda(), b.cuda(), dY.cuda()
    st.step(Xd, Wd, bd, dYd)
    torch.cuda.synchronize()
    dz1 = st.dZ.clone()
    own = [float(np.abs(t.float().numpy()).max()) for t in (X, W, dY)] + [float(dz1.abs().max())]
    assert np.array_equal(st.amax_seen.cpu().numpy().ravel(), np.float32(own))
    assert np.array_equal(st.hist[:, 0].cpu().numpy(), np.float32(own))
    assert np.array_equal(st.amax_use.cpu().numpy().ravel(), np.float32(own))
    dW1 = st.dW.clone()
    st.step(Xd, Wd, bd, dYd)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    qx, sx, _ = oracle.tensor_quantize(workloads.bits(X), E4M3, own[0])
    qw, sw, _ = oracle.tensor_quantize(workloads.bits(W), E4M3, own[1])
    assert np.array_equal(st.Xq.q.cpu().numpy(), qx) and np.array_equal(st.Wq.q.cpu().numpy(), qw)
    acc, S = oracle.tensor_gemm(qx, sx, E4M3, qw, sw, E4M3)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(b))
    y = bf16_to_f64(st.Y)
    assert_within(y, Yo, MAX_DGELU * FULL_C * S + bf16_ulp(np.maximum(np.abs(y), np.abs(Yo))) + 1e-5 * np.abs(Zo), "Y")
    # the transposed dZ codes of step 2 use step 1's dZ amax
    qdz, sdz, _ = oracle.tensor_quantize(workloads.bits(st.dZ.cpu()), E5M2, own[3], transpose=True)
    assert np.array_equal(st.dZTq.q.cpu().numpy(), qdz)
    assert st.dZTq.scale.item() == sdz
    # step 2's weight-gradient increment vs the oracle on the same codes
    qxt, sxt, _ = oracle.tensor_quantize(workloads.bits(X), E4M3, own[0], transpose=True)
    acc2, S2 = oracle.tensor_gemm(qdz, sdz, E5M2, qxt, sxt, E4M3)
    inc = (st.dW - dW1).cpu().double().numpy()
    assert_within(inc, acc2, FULL_C * S2 + 2 * f32_ulp(st.dW.cpu().double().numpy()), "dW increment")


def test_current_scaling_training_step(fp8):
    # current scaling: every cast takes its own tensor's amax first, so one
    # step's forward equals the oracle with per-tensor amaxes of its inputs
    from fp8_linear_layer_gb300.linear import TensorLinearTrainStep
    m, k, n = 384, 256, 640
    X = workloads.normal_bf16((m, k), 600, "X")
    W = workloads.normal_bf16((n, k), 600, "W", std=0.05)
    b = workloads.normal_bf16((n,), 600, "b", std=0.02)
    dY = workloads.normal_bf16((m, k), 600, "dY", std=1e-2)
    st = TensorLinearTrainStep(m, k, n, scaling="current")
    st.step(X.cuda(), W.cuda(), b.cuda(), dY.cuda())
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    am = [float(np.abs(t.float().numpy()).max()) for t in (X, W, dY)] + [float(st.dZ.abs().max())]
    assert np.array_equal(st.amax_use.cpu().numpy().ravel(), np.float32(am))
    qx, sx, _ = oracle.tensor_quantize(workloads.bits(X), E4M3, am[0])
    qw, sw, _ = oracle.tensor_quantize(workloads.bits(W), E4M3, am[1])
    acc, S = oracle.tensor_gemm(qx, sx, E4M3, qw, sw, E4M3)
    Zo, Yo = oracle.fprop_epilogue(acc, workloads.bits(b))
    y = bf16_to_f64(st.Y)
    assert_within(y, Yo, MAX_DGELU * FULL_C * S + bf16_ulp(np.maximum(np.abs(y), np.abs(Yo))) + 1e-5 * np.abs(Zo), "Y")
    qdz, sdz, _ = oracle.tensor_quantize(workloads.bits(st.dZ.cpu()), E5M2, am[3], transpose=True)
    assert np.array_equal(st.dZTq.q.cpu().numpy(), qdz)


def test_training_step_bitwise_repeatable(fp8):
    # the amax reductions are maxima (order-free) and every GEMM sum has a
    # fixed order: two fresh steps on the same inputs agree bit for bit
    from fp8_linear_layer_gb300.linear import TensorLinearTrainStep
    m, k, n = 512, 384, 768
    X = workloads.normal_bf16((m, k), 610, "X").cuda()
    W = workloads.normal_bf16((n, k), 610, "W", std=0.05).cuda()
    b = workloads.normal_bf16((n,), 610, "b", std=0.02).cuda()
    dY = workloads.normal_bf16((m, k), 610, "dY", std=1e-2).cuda()
    outs = []
    for _ in range(2):
        st = TensorLinearTrainStep(m, k, n, scaling="delayed", history=3)
        for _ in range(2):
            st.step(X, W, b, dY)
        outs.append([t.clone() for t in (st.Y, st.Z, st.dZ, st.db, st.dW, st.hist, st.amax_use)])
    torch.cuda.synchronize()
    for a, c in zip(*outs):
        assert torch.equal(a, c)


def test_amax_histories_batched(fp8):
    # three histories in one call: each row behaves as the oracle's single history
    hist = torch.zeros((3, 4), device="cuda")
    use = torch.empty((3, 1), device="cuda")
    h_o = [np.zeros(4, dtype=np.float32) for _ in range(3)]
    steps = [(1.0, 5.0, 0.25), (2.0, 0.5, 0.125), (0.5, 0.25, 8.0), (0.25, 0.125, 0.5), (0.125, 4.0, 0.25)]
    for vals in steps:
        new = torch.tensor(vals, dtype=torch.float32, device="cuda").reshape(3, 1)
        fp8.amax_history_update(hist, new, use)
        torch.cuda.synchronize()
        for h in range(3):
            h_o[h], u = oracle.amax_history(h_o[h], vals[h])
            assert np.array_equal(hist[h].cpu().numpy(), h_o[h]) and use[h].item() == u
