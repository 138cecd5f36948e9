"""fp8_bgrad_from_operand against the oracle: the bias gradient as row sums of
the weight-gradient GEMM's 1x128-scaled fp8 operand (BGRADB on "Replaced
cublasLt calls with rocblas gemm + 6 manually crafted epilogues").

Inputs are seeded: random codes and scales, and the oracle's own transposed
cast of seeded bf16 gradients.  Tolerance, from the kernel's arithmetic: every
term passes through at most 16 + K/2048 fp32 roundings (a chain of four codes
and a two-level tree per 16 codes, the scale product, a lane's chunks, the
butterfly over 32 lanes, the four warps of a row, the accumulate), so
|kernel - oracle| <= (48 + K/2048) 2^-24 S with S = sum of |terms|, plus one
rounding of the result when accumulating.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
U = 2.0 ** -24


def bound(K, S, result):
    return (48 + K // 2048) * U * S + U * np.abs(result) + 1e-30


def random_operand(fp8, rows, K, fmt, seed, ld_pad=0):
    """Random codes (no NaN / Inf) in [rows][K + ld_pad] and scales [K/128][scale_ld + 4]."""
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, (rows, K + ld_pad)).astype(np.uint8)
    if fmt == E4M3:
        q[(q & 0x7F) == 0x7F] = 0x5A
    else:
        q[(q & 0x7C) == 0x7C] = 0x3D
    sld = fp8.scale_ld(rows) + 4
    scale = rng.uniform(2.0 ** -12, 4.0, (K // 128, sld)).astype(np.float32)
    qd = torch.from_numpy(q).cuda()[:, :K]
    A = fp8.Fp8Tensor(qd, torch.from_numpy(scale).cuda(), fmt)
    return A, np.ascontiguousarray(q[:, :K]), scale


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rows,K", [(1, 128), (77, 384), (300, 2176), (1031, 4096)])
def test_random_codes_match_oracle(fp8, oracle_mod, fmt, rows, K):
    A, q, scale = random_operand(fp8, rows, K, fmt, 1000 + rows + fmt, ld_pad=48)
    assert A.q.stride(0) == K + 48
    ref, S = oracle_mod.operand_rowsum(q, scale[:, :rows], fmt)
    db = fp8.bgrad_from_operand(A).cpu().double().numpy()
    assert np.all(np.abs(db - ref) <= bound(K, S, ref)), np.abs(db - ref).max()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_accumulate(fp8, oracle_mod, fmt):
    rows, K = 333, 1152
    A, q, scale = random_operand(fp8, rows, K, fmt, 77 + fmt)
    ref, S = oracle_mod.operand_rowsum(q, scale[:, :rows], fmt)
    prefill = workloads.normal_f32((rows,), 78, "db0", std=50.0)
    out = prefill.clone().cuda()
    fp8.bgrad_from_operand(A, out=out, accumulate=True)
    want = prefill.double().numpy() + ref
    got = out.cpu().double().numpy()
    assert np.all(np.abs(got - want) <= bound(K, S, want) + U * np.abs(prefill.double().numpy()))
    # accumulate=False overwrites whatever was there
    fp8.bgrad_from_operand(A, out=out, accumulate=False)
    assert np.all(np.abs(out.cpu().double().numpy() - ref) <= bound(K, S, ref))


def test_transposed_cast_of_the_gradient(fp8, oracle_mod):
    # dZ [tokens][features], cast down its columns by the oracle: the weight
    # gradient's operand dZ^T; its row sums are the bias gradient
    tokens, features = 640, 264
    dz = workloads.normal_bf16((tokens, features), 91, "dz", std=0.01)
    qt, st = oracle_mod.quantize(workloads.bits(dz), E5M2, transpose=True)
    sld = fp8.scale_ld(features)
    sc = torch.zeros((tokens // 128, sld), dtype=torch.float32)
    sc[:, :features] = torch.from_numpy(st)
    A = fp8.Fp8Tensor(torch.from_numpy(qt).cuda(), sc.cuda(), E5M2)
    ref, S = oracle_mod.operand_rowsum(qt, st, E5M2)
    db = fp8.bgrad_from_operand(A).cpu().double().numpy()
    assert np.all(np.abs(db - ref) <= bound(tokens, S, ref))
    # and it is the column sum of dZ up to one e5m2 rounding per element
    x = dz.double().numpy()
    assert np.all(np.abs(db - x.sum(axis=0)) <= 2.0 ** -3 * np.abs(x).sum(axis=0) + tokens * 2.0 ** -16 * st.max()
                  + bound(tokens, S, ref))


def test_full_size_sampled_rows(fp8, oracle_mod):
    # the training step's operand: dZ of 8192 tokens x 14336 features, cast
    # down its columns on the GPU (e5m2), reduced over all 8192 tokens; 48
    # sampled features checked against the oracle's cast and row sums of those
    # columns (the cast down columns treats each column alone)
    tokens, features = 8192, 14336
    dz = workloads.normal_bf16((tokens, features), 92, "dzfull", std=0.01)
    A = fp8.quantize(dz.cuda(), E5M2, transpose=True)
    db = fp8.bgrad_from_operand(A).cpu().double().numpy()
    cols = np.sort(np.random.default_rng(93).choice(features, 48, replace=False))
    cols[0], cols[-1] = 0, features - 1
    sub = dz[:, torch.from_numpy(cols)].contiguous()
    qt, st = oracle_mod.quantize(workloads.bits(sub), E5M2, transpose=True)
    ref, S = oracle_mod.operand_rowsum(qt, st, E5M2)
    assert np.all(np.abs(db[cols] - ref) <= bound(tokens, S, ref))
    assert np.isfinite(db).all()


def test_deterministic_and_exact_cases(fp8):
    rows, K = 4099, 8192
    A, _, _ = random_operand(fp8, rows, K, E4M3, 5)
    a = fp8.bgrad_from_operand(A)
    b = fp8.bgrad_from_operand(A)
    assert torch.equal(a, b)
    # every code the largest e4m3 value (448), every scale 2^-10: the sum is exact
    q = torch.full((rows, K), 0x7E, dtype=torch.uint8, device="cuda")
    q[1] = 0xFE  # -448
    q[2] = 0x80  # -0
    s = torch.full((K // 128, fp8.scale_ld(rows)), 2.0 ** -10, dtype=torch.float32, device="cuda")
    db = fp8.bgrad_from_operand(fp8.Fp8Tensor(q, s, E4M3)).cpu()
    assert db[0] == 448.0 * K * 2.0 ** -10 and db[1] == -db[0] and db[2] == 0.0
    assert torch.all(db[3:] == db[0])
    # no rows: nothing launched, nothing written
    empty = fp8.Fp8Tensor(q[:0], s, E4M3)
    out = torch.full((0,), 1.0, device="cuda")
    fp8.bgrad_from_operand(empty, out=out)


def test_writes_stay_in_bounds(fp8):
    rows, K = 301, 640
    A, _, _ = random_operand(fp8, rows, K, E5M2, 6)
    G = 64
    buf = torch.full((rows + 2 * G,), 7.5, dtype=torch.float32, device="cuda")
    out = buf[G:G + rows]
    for accumulate in (False, True):
        fp8.bgrad_from_operand(A, out=out, accumulate=accumulate)
        torch.cuda.synchronize()
        assert torch.all(buf[:G] == 7.5) and torch.all(buf[G + rows:] == 7.5)


def test_train_step_with_the_operand_bias_gradient(fp8):
    """LinearTrainStep(bias_grad="operand"): the data-gradient GEMM drops its
    bias-gradient sums and db is reduced from dZ^T's codes.  dZ and dW are
    bit-identical to the step with the epilogue's sums; db is the oracle's column sum of its
    dZ within one e5m2 rounding per element (plus dZ's own bound)."""
    import oracle
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    from helpers import FULL_C, bf16_ulp, dgelu_eval_bound
    m, k, n = 512, 384, 640
    X = workloads.normal_bf16((m, k), 79, "X")
    W = workloads.normal_bf16((n, k), 79, "W", std=0.05)
    b = workloads.normal_bf16((n,), 79, "b", std=0.02)
    dY = workloads.normal_bf16((m, k), 79, "dY", std=1e-2)
    args = (X.cuda(), W.cuda(), b.cuda(), dY.cuda())
    ref = LinearTrainStep(m, k, n, bias_grad="dgrad")
    st = LinearTrainStep(m, k, n, bias_grad="operand")
    assert st.KERNELS_PER_STEP == ref.KERNELS_PER_STEP == 8
    assert [kind for kind, _ in st.launches(*args)].count("reduce") == 1
    ref.step(*args)
    st.step(*args)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    assert torch.equal(st.dZ, ref.dZ) and torch.equal(st.dW, ref.dW) and torch.equal(st.Y, ref.Y)
    qx, sx = oracle.quantize(workloads.bits(X), E4M3)
    qw, sw = oracle.quantize(workloads.bits(W), E4M3)
    acc, S = oracle.gemm(qx, sx, E4M3, qw, sw, E4M3)
    Zo, _ = oracle.fprop_epilogue(acc, workloads.bits(b))
    zb = oracle.f64_to_bf16_array(Zo)
    qd, sd = oracle.quantize(workloads.bits(dY), E5M2)
    acc2, S2 = oracle.gemm(qd, sd, E5M2, qw, sw, E4M3)
    dzo = oracle.dgrad_epilogue(acc2, zb)
    zbf = oracle.bf16_to_f64(zb)
    g = np.abs(oracle.dgelu(zbf))
    bound_dz = (g * FULL_C * S2 + 0.8 * (FULL_C * S + bf16_ulp(Zo)) * np.abs(acc2)
                + np.abs(acc2) * dgelu_eval_bound(zbf) + 2 * bf16_ulp(np.abs(dzo)))
    mag = np.abs(dzo) + bound_dz
    tol = 2.0 ** -3 * mag.sum(0) + bound_dz.sum(0) + m * 2.0 ** -16 * mag.max(0) / 57344 * 2 + 64 * U * mag.sum(0)
    db = st.db.cpu().double().numpy()
    assert np.all(np.abs(db - dzo.sum(0)) <= tol)
    # the two bias gradients agree to the e5m2 rounding of dZ
    assert np.all(np.abs(db - ref.db.cpu().double().numpy()) <= 2.0 ** -3 * mag.sum(0) + tol)
