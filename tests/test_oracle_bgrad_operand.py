"""Pins for the oracle's bias gradient reduced from the weight-gradient GEMM's
fp8 operand (CPU only).

"Replaced cublasLt calls with rocblas gemm + 6 manually crafted epilogues"
takes db together with dW (BGRADB) by reducing the gradient operand of the
weight-gradient GEMM over that GEMM's k.  With the operand cast by 1x128
blocks the reduction is db[r] = sum_k scale[k/128][r] dec(q[r][k]).  Pins: a
closed form, torch's float8 decode with a float64 sum, and the bias gradient
it stands for (column sums of the unquantized gradient, within the cast's
rounding bound).
"""
import numpy as np
import pytest
import torch

import workloads

E4M3, E5M2 = 0, 1
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def dec(q, fmt):
    return torch.from_numpy(np.ascontiguousarray(q)).view(TORCH_DT[fmt]).double().numpy()


def test_ones_closed_form(oracle_mod):
    # every code is 1.0; block kb of row r has scale (r + 1) 2^-kb: db[r] = 128 (r + 1) (2 - 2^-(B-1))
    rows, B = 5, 3
    q = np.full((rows, 128 * B), 0x38, dtype=np.uint8)  # e4m3 1.0
    scale = np.zeros((B, 8), dtype=np.float32)
    for kb in range(B):
        scale[kb, :rows] = (np.arange(rows) + 1) * 2.0 ** -kb
    scale[:, rows:] = 1e30  # padding columns of the scale rows are never read
    out, S = oracle_mod.operand_rowsum(q, scale, E4M3)
    ref = 128 * (np.arange(rows) + 1) * (2 - 2.0 ** -(B - 1))
    assert np.array_equal(out, ref) and np.array_equal(S, ref)
    # the same codes read as e5m2 (0x38 = 0.5) halve every term
    q5 = np.full((rows, 128 * B), 0x38, dtype=np.uint8)
    out5, _ = oracle_mod.operand_rowsum(q5, scale, E5M2)
    assert np.array_equal(out5, ref / 2)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_random_codes_against_torch_decode(oracle_mod, fmt):
    rng = np.random.default_rng(31 + fmt)
    rows, K = 37, 640
    q = rng.integers(0, 256, (rows, K)).astype(np.uint8)
    if fmt == E4M3:
        q[(q & 0x7F) == 0x7F] = 0x21
    else:
        q[(q & 0x7C) == 0x7C] = 0x42
    scale = rng.uniform(0.01, 3.0, (K // 128, 40)).astype(np.float32)
    out, S = oracle_mod.operand_rowsum(q, scale, fmt)
    terms = dec(q, fmt) * np.repeat(scale[:, :rows].astype(np.float64).T, 128, axis=1)
    ref = terms.sum(axis=1)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(terms).sum(axis=1).max())
    assert np.allclose(S, np.abs(terms).sum(axis=1), rtol=1e-12)
    assert (out < 0).any() and (out > 0).any()


def test_is_the_bias_gradient_of_the_transposed_cast(oracle_mod):
    # dZ [tokens][features] cast down its columns (the weight-gradient operand
    # dZ^T, e5m2): its row sums are the bias gradient sum_t dZ[t][j] up to one
    # e5m2 rounding per element (half a mantissa step, plus the subnormal spacing)
    dz = workloads.normal_bf16((384, 256), 33, "g", std=0.02)
    qt, st = oracle_mod.quantize(workloads.bits(dz), E5M2, transpose=True)
    assert qt.shape == (256, 384)
    out, _ = oracle_mod.operand_rowsum(qt, st, E5M2)
    x = dz.double().numpy()
    exact = x.sum(axis=0)
    bound = 2.0 ** -3 * np.abs(x).sum(axis=0) + 384 * 2.0 ** -16 * st.max()
    err = np.abs(out - exact)
    assert np.all(err <= bound)
    assert err.max() > 0  # the cast rounds: this is not the plain column sum
    # and the untransposed cast's row sums are the sums over features instead
    q, s = oracle_mod.quantize(workloads.bits(dz), E5M2)
    out_r, _ = oracle_mod.operand_rowsum(q, s, E5M2)
    assert np.all(np.abs(out_r - x.sum(axis=1)) <= 2.0 ** -3 * np.abs(x).sum(axis=1) + 256 * 2.0 ** -16 * s.max())


def test_zero_rows_and_signed_zero(oracle_mod):
    q = np.zeros((3, 128), dtype=np.uint8)
    q[1] = 0x80  # -0
    q[2, 5] = 0xB8  # e4m3 -1.0
    scale = np.full((1, 4), 2.0, dtype=np.float32)
    out, S = oracle_mod.operand_rowsum(q, scale, E4M3)
    assert list(out) == [0.0, 0.0, -2.0] and list(S) == [0.0, 0.0, 2.0]
