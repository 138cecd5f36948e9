"""Pins for the oracle's MXFP8 cast and GEMM (CPU only).

Reading (the MX block format is only named on "How can we use te.Linear with
weight parallel?"): one power-of-two scale 2^e per 32 consecutive elements of
a row (or of a column, transposed), stored as the UE8M0 byte e + 127; e is the
smallest integer in [-127, 127] with amax <= FMAX 2^e, so no element
saturates; an all-zero block takes e = 0; codes are enc(x 2^-e).  The pins are
closed forms, the defining inequalities, nearest-code optimality, exact
power-of-two round trips, exact-rational brute force and a float64 matmul of
torch-decoded operands.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads

E4M3, E5M2 = 0, 1
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
FMAX = {E4M3: 448.0, E5M2: 57344.0}


@pytest.mark.parametrize("fmt,e_ones", [(E4M3, -8), (E5M2, -15)])
def test_all_ones_closed_form(oracle_mod, fmt, e_ones):
    # 1 <= FMAX 2^e first holds at e = -8 (448/256 = 1.75) resp. -15 (57344/32768 = 1.75)
    x = torch.ones(3, 96, dtype=torch.bfloat16)
    q, e = oracle_mod.mx_quantize(workloads.bits(x), fmt)
    assert e.shape == (3, 3) and np.all(e == e_ones)
    assert np.all(oracle_mod.decode(fmt, q) == 2.0 ** -e_ones)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_exponent_is_the_smallest_that_avoids_saturation(oracle_mod, fmt):
    x = workloads.normal_bf16((48, 256), 81, "mx", std=3.0)
    x, _ = workloads.with_outlier_rows(x, 81, "mx")
    x[7, 64:96] = 0
    q, e = oracle_mod.mx_quantize(workloads.bits(x), fmt)
    xf = x.double().numpy()
    for r in range(48):
        for b in range(8):
            amax = np.abs(xf[r, 32 * b:32 * b + 32]).max()
            eb = int(e[b, r])
            if amax == 0:
                assert eb == 0
                continue
            assert amax <= FMAX[fmt] * 2.0 ** eb
            assert eb == -127 or amax > FMAX[fmt] * 2.0 ** (eb - 1)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_codes_are_nearest_to_the_scaled_values(oracle_mod, fmt):
    x = workloads.normal_bf16((16, 128), 82, "mxn", std=0.5)
    q, e = oracle_mod.mx_quantize(workloads.bits(x), fmt)
    t = oracle_mod.decode_table(fmt)
    fin = t[np.isfinite(t)]
    xf = x.double().numpy()
    for r in range(16):
        for b in range(4):
            y = xf[r, 32 * b:32 * b + 32] * 2.0 ** (-int(e[b, r]))
            d = np.abs(oracle_mod.decode(fmt, q[r, 32 * b:32 * b + 32]) - y)
            best = np.min(np.abs(fin[None, :] - y[:, None]), axis=1)
            assert np.all(d == best)
            assert np.all(np.abs(y) <= FMAX[fmt])  # nothing saturates


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_powers_of_two_round_trip_exactly(oracle_mod, fmt):
    # each block holds one power of two and its halves: exact after dequantization
    v = torch.zeros(4, 64, dtype=torch.float32)
    for r in range(4):
        for b in range(2):
            v[r, 32 * b:32 * b + 32] = 2.0 ** (3 * r - 5 * b) * torch.tensor([1.0, -0.5, 0.25] * 10 + [1.0, 0.0])
    q, e = oracle_mod.mx_quantize(workloads.bits(v.to(torch.bfloat16)), fmt)
    deq = oracle_mod.decode(fmt, q) * np.repeat(2.0 ** e.T.astype(np.float64), 32, axis=1)
    assert np.array_equal(deq, v.double().numpy())


def test_zero_and_tiny_blocks(oracle_mod):
    x = torch.zeros(2, 64, dtype=torch.float32)
    x[1] = -x[1]
    x[0, 32], x[0, 33] = 1e-38, -3e-39  # below 448 * 2^-127: the exponent clamps at -127
    q, e = oracle_mod.mx_quantize(workloads.bits(x.to(torch.bfloat16)), E4M3)
    assert e[0, 0] == 0 and e[0, 1] == 0 and e[1, 0] == -127
    assert np.all(q[0, :32] == 0x00) and np.all(q[1] == 0x80)
    assert q[0, 32] != 0 and q[0, 33] & 0x80  # still representable after scaling by 2^127


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_transposed_equals_rows_of_the_transpose(oracle_mod, fmt):
    x = workloads.normal_bf16((96, 40), 83, "mxt")
    qt, et = oracle_mod.mx_quantize(workloads.bits(x), fmt, transpose=True)
    qr, er = oracle_mod.mx_quantize(workloads.bits(x.t().contiguous()), fmt)
    assert qt.shape == (40, 96) and et.shape == (3, 40)
    assert np.array_equal(qt, qr) and np.array_equal(et, er)


@pytest.mark.parametrize("fmts", [(E4M3, E4M3), (E5M2, E4M3)])
def test_gemm_brute_force_exact_rationals(oracle_mod, fmts):
    fa, fb = fmts
    a = workloads.normal_bf16((3, 64), 84, "ga", std=2.0)
    b = workloads.normal_bf16((4, 64), 84, "gb", std=0.1)
    qa, ea = oracle_mod.mx_quantize(workloads.bits(a), fa)
    qb, eb = oracle_mod.mx_quantize(workloads.bits(b), fb)
    acc, S = oracle_mod.mx_gemm(qa, ea, fa, qb, eb, fb)
    da = torch.from_numpy(qa).view(TORCH_DT[fa]).double().numpy()
    db = torch.from_numpy(qb).view(TORCH_DT[fb]).double().numpy()
    for i in range(3):
        for j in range(4):
            exact = sum(Fraction(float(da[i, k])) * Fraction(2) ** int(ea[k // 32, i]) *
                        Fraction(float(db[j, k])) * Fraction(2) ** int(eb[k // 32, j]) for k in range(64))
            assert abs(Fraction(acc[i, j]) - exact) <= Fraction(1, 2 ** 50) * (Fraction(S[i, j]) + 1)


def test_gemm_matches_float64_matmul_of_torch_decoded_operands(oracle_mod):
    M, N, K = 33, 21, 256
    a = workloads.normal_bf16((M, K), 85, "a")
    b = workloads.normal_bf16((N, K), 85, "b", std=0.02)
    qa, ea = oracle_mod.mx_quantize(workloads.bits(a), E5M2)
    qb, eb = oracle_mod.mx_quantize(workloads.bits(b), E4M3)
    acc, S = oracle_mod.mx_gemm(qa, ea, E5M2, qb, eb, E4M3)
    A = torch.from_numpy(qa).view(torch.float8_e5m2).double().numpy() * np.repeat(2.0 ** ea.T.astype(np.float64), 32, 1)
    B = torch.from_numpy(qb).view(torch.float8_e4m3fn).double().numpy() * np.repeat(2.0 ** eb.T.astype(np.float64), 32, 1)
    assert np.all(np.abs(acc - A @ B.T) <= 1e-12 * S)
    assert np.allclose(S, np.abs(A) @ np.abs(B).T, rtol=1e-12)
    # and the MX-quantized product stays close to the unquantized one
    exact = a.double().numpy() @ b.double().numpy().T
    assert np.max(np.abs(acc - exact) / S) < 0.1


def test_gemm_all_ones_gives_K(oracle_mod):
    x = torch.ones(5, 320, dtype=torch.bfloat16)
    q, e = oracle_mod.mx_quantize(workloads.bits(x), E4M3)
    acc, S = oracle_mod.mx_gemm(q, e, E4M3, q, e, E4M3)
    assert np.all(acc == 320.0) and np.array_equal(acc, S)
