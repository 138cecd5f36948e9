"""Pins for the oracle's per-tensor scaling (CPU only).

"FP8 GEMM for the fprop should use fast accumulation" works with one scale per
operand tensor.  The reading: a cast from a given amax A (the tensor's own amax
-- current scaling -- or the largest amax of earlier steps -- delayed scaling),
inv = fl32(FMAX/A), scale = fl32(A/FMAX), q = enc(fl32(x inv)) saturating at
+-FMAX; the amax history takes the new amax at its front and drops its oldest
entry; the GEMM is sa sb sum_k dec(qa) dec(qb).  The pins below are closed
forms, torch's float8 codec and exact invariants.
"""
import numpy as np
import pytest
import torch

import workloads

E4M3, E5M2 = 0, 1
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}
FMAX = {E4M3: 448.0, E5M2: 57344.0}
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def dec(q, fmt):
    return torch.from_numpy(np.ascontiguousarray(q)).view(TORCH_DT[fmt]).double().numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_all_ones_closed_form(oracle_mod, fmt):
    x = torch.ones(3, 256, dtype=torch.bfloat16)
    q, s, a = oracle_mod.tensor_quantize(workloads.bits(x), fmt, 1.0)
    assert np.all(q == MAXCODE[fmt])
    assert s == np.float32(1.0) / np.float32(FMAX[fmt])
    assert a == 1.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("transpose", [False, True])
def test_current_scaling_matches_torch_cast(oracle_mod, fmt, transpose):
    # with the tensor's own amax, every code is torch's saturating float8 cast
    # of the fp32 product x * fl32(FMAX/amax), and the largest |x| maps to FMAX
    x = workloads.normal_bf16((96, 320), 11 + fmt, "t", std=3.0)
    xf = x.float()
    amax = float(xf.abs().max())
    q, s, a = oracle_mod.tensor_quantize(workloads.bits(x), fmt, amax, transpose=transpose)
    assert a == np.float32(amax)
    inv = np.float32(FMAX[fmt]) / np.float32(amax)
    assert s == np.float32(amax) / np.float32(FMAX[fmt])
    ref = (xf * torch.tensor(inv, dtype=torch.float32)).clamp(-FMAX[fmt], FMAX[fmt]).to(TORCH_DT[fmt])
    ref = ref.view(torch.uint8).numpy()
    assert np.array_equal(q, ref.T if transpose else ref)
    assert (q & 0x7F).max() == MAXCODE[fmt]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_delayed_amax_saturates_above_it(oracle_mod, fmt):
    # a history amax below the tensor's own: everything beyond it saturates
    x = workloads.normal_bf16((64, 256), 13, "d", std=1.0)
    xf = x.float().numpy()
    own = float(np.abs(xf).max())
    hist = own / 4
    q, s, a = oracle_mod.tensor_quantize(workloads.bits(x), fmt, hist)
    assert a == np.float32(own)
    assert s == np.float32(hist) / np.float32(FMAX[fmt])
    big = np.abs(xf) >= hist
    assert big.any()
    assert np.all((q[big] & 0x7F) == MAXCODE[fmt])
    assert np.all((q[big] >> 7) == (xf[big] < 0))
    # below the history amax: the nearest code of x / scale (relative error of
    # one fp8 rounding, half a mantissa step, plus the subnormal spacing)
    d = dec(q, fmt) * float(s)
    small = ~big
    mant = 3 if fmt == E4M3 else 2
    sub = 2.0 ** (-9 if fmt == E4M3 else -16) * float(s)
    assert np.all(np.abs(d[small] - xf[small]) <= 2.0 ** -(mant + 1) * np.abs(xf[small]) * 1.001 + sub)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_zero_tensor_and_signed_zero(oracle_mod, fmt):
    x = torch.zeros(2, 128, dtype=torch.bfloat16)
    x[1] = -x[1]
    q, s, a = oracle_mod.tensor_quantize(workloads.bits(x), fmt, 0.0)
    assert s == 1.0 and a == 0.0
    assert np.all(q[0] == 0x00) and np.all(q[1] == 0x80)


def test_tiny_amax_takes_unit_scale(oracle_mod):
    # FMAX / amax overflows binary32: scale 1, the values encode as themselves
    x = torch.zeros(1, 128, dtype=torch.float32)
    x[0, 0] = 1e-38
    q, s, a = oracle_mod.tensor_quantize(workloads.bits(x.to(torch.bfloat16)), E4M3, 1e-38)
    assert s == 1.0
    assert np.all(q == 0)


def test_amax_history():
    import oracle
    h, use = oracle.amax_history(np.zeros(4, dtype=np.float32), 2.5)
    assert list(h) == [2.5, 0, 0, 0] and use == 2.5
    h, use = oracle.amax_history(h, 1.0)
    assert list(h) == [1.0, 2.5, 0, 0] and use == 2.5
    for v in (0.5, 0.25, 0.125):
        h, use = oracle.amax_history(h, v)
    # 2.5 has dropped out after four newer entries
    assert list(h) == [0.125, 0.25, 0.5, 1.0] and use == 1.0
    h1, use1 = oracle.amax_history(np.zeros(1, dtype=np.float32), 3.0)
    assert list(h1) == [3.0] and use1 == 3.0


def test_tensor_gemm_closed_form_and_float64_matmul(oracle_mod):
    # all-ones operands: every entry is K sa sb
    qa = np.full((3, 256), 0x38, dtype=np.uint8)  # e4m3 1.0
    qb = np.full((5, 256), 0x3C, dtype=np.uint8)  # e5m2 1.0
    acc, S = oracle_mod.tensor_gemm(qa, 0.5, E4M3, qb, 0.25, E5M2)
    assert np.all(acc == 256 * 0.125) and np.all(S == 256 * 0.125)
    # random codes (no NaN / Inf) against a float64 matmul of torch-decoded operands
    rng = np.random.default_rng(5)
    qa = rng.integers(0, 256, (7, 384)).astype(np.uint8)
    qb = rng.integers(0, 256, (9, 384)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x11
    qb[(qb & 0x7C) == 0x7C] = 0x22
    sa, sb = np.float32(0.37), np.float32(1.9)
    acc, S = oracle_mod.tensor_gemm(qa, sa, E4M3, qb, sb, E5M2)
    A, B = dec(qa, E4M3), dec(qb, E5M2)
    ref = float(sa) * float(sb) * (A @ B.T)
    assert np.allclose(acc, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.allclose(S, float(sa) * float(sb) * (np.abs(A) @ np.abs(B).T), rtol=1e-12)
    # a transposed operand gives the transposed result
    acc_t, _ = oracle_mod.tensor_gemm(qb, sb, E5M2, qa, sa, E4M3)
    assert np.allclose(acc_t, acc.T, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def test_recorded_amax_is_a_magnitude(oracle_mod):
    # the largest magnitude is negative: the recorded amax is its absolute value
    x = torch.full((2, 128), 0.5, dtype=torch.float32)
    x[1, 77] = -9.0
    x[0, 3] = 4.0
    q, s, a = oracle_mod.tensor_quantize(workloads.bits(x.to(torch.bfloat16)), E4M3, 9.0)
    assert a == 9.0
    assert q[1, 77] == 0xFE and s == np.float32(9.0) / np.float32(448.0)
