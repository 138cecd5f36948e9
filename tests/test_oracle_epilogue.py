"""Pins for the oracle's epilogue math (CPU only).

"Replaced cublasLt calls with rocblas gemm + 6 manually crafted epilogues":
Y = X W^T + b with b of length n (output features), db = sum of the output
gradient over the batch axis, and, with bias and GELU together, the GELU
derivative is applied before the bias-gradient reduction.  GELU is the tanh
form.  Pins: special values and limits, finite differences, torch's tanh GELU,
closed-form column sums.
"""
import numpy as np
import pytest
import torch

import workloads


def test_gelu_special_values(oracle_mod):
    assert oracle_mod.gelu([0.0])[0] == 0.0
    assert oracle_mod.dgelu([0.0])[0] == 0.5
    assert abs(oracle_mod.gelu([10.0])[0] - 10.0) < 1e-12
    assert abs(oracle_mod.gelu([-10.0])[0]) < 1e-12
    assert abs(oracle_mod.dgelu([10.0])[0] - 1.0) < 1e-12
    assert abs(oracle_mod.dgelu([-10.0])[0]) < 1e-12
    assert oracle_mod.dgelu([20.0])[0] == 1.0


def test_dgelu_finite_differences(oracle_mod):
    z = np.linspace(-8, 8, 4001)
    h = 1e-4
    fd = (oracle_mod.gelu(z + h) - oracle_mod.gelu(z - h)) / (2 * h)
    assert np.max(np.abs(fd - oracle_mod.dgelu(z))) < 1e-7


def test_gelu_matches_torch_tanh_gelu(oracle_mod):
    z = torch.linspace(-12, 12, 10001, dtype=torch.float64)
    ref = torch.nn.functional.gelu(z, approximate="tanh").numpy()
    assert np.max(np.abs(oracle_mod.gelu(z.numpy()) - ref)) < 1e-13
    zz = z.clone().requires_grad_(True)
    torch.nn.functional.gelu(zz, approximate="tanh").sum().backward()
    assert np.max(np.abs(oracle_mod.dgelu(z.numpy()) - zz.grad.numpy())) < 1e-13


def _tanh_form_decimal(z, deriv):
    """gelu / gelu' in the tanh form, 150 significant digits (decimal module)."""
    from decimal import Decimal, getcontext
    getcontext().prec = 150
    pi = Decimal("3.14159265358979323846264338327950288419716939937510582097494459230781640628620899862803482534211706798214808651328230664709384460955058223172535940812848111745")
    c = (Decimal(2) / pi).sqrt()
    a = Decimal("0.044715")
    zd = Decimal(repr(float(z)))
    u = c * (zd + a * zd ** 3)
    e2 = (2 * u).exp()
    t = (e2 - 1) / (e2 + 1)
    if not deriv:
        return float(Decimal("0.5") * zd * (1 + t))
    return float(Decimal("0.5") * (1 + t) + Decimal("0.5") * zd * (1 - t * t) * c * (1 + 3 * a * zd * zd))


def test_gelu_relative_accuracy_against_150_digit_tanh_form(oracle_mod):
    # includes large negative z, where 1 + tanh(u) cancels in binary64
    zs = np.concatenate([np.linspace(-12, 12, 241), [-9.7, -8.3, -7.1, -6.6, 7.3]])
    g = oracle_mod.gelu(zs)
    d = oracle_mod.dgelu(zs)
    for z, gv, dv in zip(zs, g, d):
        gr = _tanh_form_decimal(z, False)
        dr = _tanh_form_decimal(z, True)
        assert abs(gv - gr) <= 1e-13 * abs(gr) + 1e-300
        # gelu' crosses zero near z = -0.7518: relative there, absolute 1e-15 near it
        assert abs(dv - dr) <= 1e-12 * abs(dr) + 1e-15


def test_max_dgelu_bound(oracle_mod):
    # the error-propagation bound uses max |gelu'| < 1.13
    z = np.linspace(-10, 10, 200001)
    assert np.max(np.abs(oracle_mod.dgelu(z))) < 1.13


def test_bias_is_per_output_feature(oracle_mod):
    M, N = 3, 5
    acc = np.arange(M * N, dtype=np.float64).reshape(M, N)
    b = torch.tensor([1.0, 2.0, 4.0, 8.0, 16.0], dtype=torch.bfloat16)
    Z, Y = oracle_mod.fprop_epilogue(acc, workloads.bits(b), gelu_on=False)
    assert np.array_equal(Z, acc + np.array([1, 2, 4, 8, 16.0])[None, :])
    assert np.array_equal(Y, Z)
    Z2, Y2 = oracle_mod.fprop_epilogue(acc, workloads.bits(b))
    assert np.allclose(Y2, oracle_mod.gelu(Z2))
    with pytest.raises(ValueError):
        oracle_mod.fprop_epilogue(acc, workloads.bits(b[:3]))  # length m is not the fprop bias


def test_bgrad_closed_form(oracle_mod):
    # pre-activation far positive -> gelu' == 1; constant upstream c -> db[j] = M c
    M, N = 64, 10
    z = torch.full((M, N), 20.0, dtype=torch.bfloat16)
    acc = np.full((M, N), 0.25)
    dz = oracle_mod.dgrad_epilogue(acc, workloads.bits(z))
    assert np.all(dz == 0.25)
    db = oracle_mod.colsum(dz)
    assert db.shape == (N,) and np.all(db == M * 0.25)
    # order: derivative first, then the reduction (not gelu'(sum))
    z2 = torch.tensor([[0.0, 20.0], [20.0, 0.0]], dtype=torch.bfloat16)
    dz2 = oracle_mod.dgrad_epilogue(np.ones((2, 2)), workloads.bits(z2))
    assert np.allclose(oracle_mod.colsum(dz2), [1.5, 1.5])


def test_colsum_is_over_rows(oracle_mod):
    dz = np.arange(12, dtype=np.float64).reshape(3, 4)
    assert np.array_equal(oracle_mod.colsum(dz), dz.sum(axis=0))
