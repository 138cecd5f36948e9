"""Pins for the oracle's block-scaled GEMM, weight-gradient accumulation and
k-grouped variant (CPU only).

Sources: "Weight gradient kernels for dense and MoE models" (DeepGEMM): the nt
weight-gradient GEMM accumulates (out += a b^T), its worked ones/rand example,
the k-grouped MoE form.  Pins: exact-rational brute force on tiny shapes, the
all-ones closed form, the page's printed ratios, the doubling property, and a
float64 matmul of operands decoded by torch's float8 dtypes.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads

E4M3, E5M2 = 0, 1
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def torch_dequant(q, s, fmt):
    """Independent dequantization: torch float8 decode times the block scale."""
    v = torch.from_numpy(np.ascontiguousarray(q)).view(TORCH_DT[fmt]).double().numpy()
    rows, K = q.shape
    return v * np.repeat(s[: K // 128].T.astype(np.float64), 128, axis=1)[:rows]


@pytest.mark.parametrize("K", [128, 256])
@pytest.mark.parametrize("fmts", [(E4M3, E4M3), (E5M2, E4M3)])
def test_brute_force_exact_rationals(oracle_mod, K, fmts):
    fa, fb = fmts
    a = workloads.normal_bf16((3, K), 21, "bfa", std=2.0)
    b = workloads.normal_bf16((4, K), 21, "bfb", std=0.5)
    qa, sa = oracle_mod.quantize(workloads.bits(a), fa)
    qb, sb = oracle_mod.quantize(workloads.bits(b), fb)
    acc, S = oracle_mod.gemm(qa, sa, fa, qb, sb, fb)
    da = torch.from_numpy(qa).view(TORCH_DT[fa]).double().numpy()
    db = torch.from_numpy(qb).view(TORCH_DT[fb]).double().numpy()
    for i in range(3):
        for j in range(4):
            exact = Fraction(0)
            absum = Fraction(0)
            for k in range(K):
                kb = k // 128
                t = Fraction(float(da[i, k])) * Fraction(float(sa[kb, i])) * \
                    Fraction(float(db[j, k])) * Fraction(float(sb[kb, j]))
                exact += t
                absum += abs(t)
            assert abs(Fraction(acc[i, j]) - exact) <= Fraction(1, 2 ** 50) * absum
            assert abs(Fraction(S[i, j]) - absum) <= Fraction(1, 2 ** 50) * absum
    # the GEMM is A B^T, not B A^T or A^T B: a transposed result would not match
    assert acc.shape == (3, 4)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_all_ones_gives_K(oracle_mod, fmt):
    K = 512
    x = torch.ones(5, K, dtype=torch.bfloat16)
    w = torch.ones(7, K, dtype=torch.bfloat16)
    qa, sa = oracle_mod.quantize(workloads.bits(x), fmt)
    qb, sb = oracle_mod.quantize(workloads.bits(w), E4M3)
    acc, S = oracle_mod.gemm(qa, sa, fmt, qb, sb, E4M3)
    assert np.all(np.abs(acc - K) <= K * 2.0 ** -21)
    assert np.array_equal(acc, S)


def test_matches_float64_matmul_of_torch_decoded_operands(oracle_mod):
    M, N, K = 37, 29, 640
    a = workloads.normal_bf16((M, K), 2, "a")
    b = workloads.normal_bf16((N, K), 2, "b", std=0.02)
    qa, sa = oracle_mod.quantize(workloads.bits(a), E5M2)
    qb, sb = oracle_mod.quantize(workloads.bits(b), E4M3)
    acc, S = oracle_mod.gemm(qa, sa, E5M2, qb, sb, E4M3)
    A = torch_dequant(qa, sa, E5M2)
    B = torch_dequant(qb, sb, E4M3)
    ref = A @ B.T
    assert np.all(np.abs(acc - ref) <= 1e-12 * S)
    assert np.allclose(S, np.abs(A) @ np.abs(B).T, rtol=1e-12)
    # quantized product stays close to the unquantized product (fp8 error scale)
    exact = a.double().numpy() @ b.double().numpy().T
    assert np.max(np.abs(acc - exact) / S) < 0.1


def test_row_col_selection_and_k_offset(oracle_mod):
    M, N, K = 20, 30, 512
    a = workloads.normal_bf16((M, K), 4, "a")
    b = workloads.normal_bf16((N, K), 4, "b")
    qa, sa = oracle_mod.quantize(workloads.bits(a), E4M3)
    qb, sb = oracle_mod.quantize(workloads.bits(b), E4M3)
    rows, cols = np.array([3, 0, 19]), np.array([29, 1, 7, 8])
    sub, _ = oracle_mod.gemm(qa, sa, E4M3, qb, sb, E4M3, K=256, k0=128, rows=rows, cols=cols)
    A = torch_dequant(qa, sa, E4M3)[:, 128:384]
    B = torch_dequant(qb, sb, E4M3)[:, 128:384]
    ref = (A @ B.T)[np.ix_(rows, cols)]
    assert np.allclose(sub, ref, rtol=1e-12, atol=1e-12)


def test_worked_example_out_plus_equals(oracle_mod):
    """The DeepGEMM page's example: out pre-filled with the fp32 reference, one
    accumulate call doubles it (printed ratios 1.9995 .. 2.0009); with a zero
    pre-fill the ratio is 1."""
    g = json.load(open(os.path.join(GOLDEN, "deepgemm_wgrad_ones_rand.json")))
    m, n, k = g["m"], g["n"], g["k"]
    x = torch.ones(m, k, dtype=torch.bfloat16)
    y = workloads.uniform_bf16((n, k), 1, "y")
    ref = (x.float() @ y.float().t()).numpy()
    qx, sx = oracle_mod.quantize(workloads.bits(x), E4M3)
    qy, sy = oracle_mod.quantize(workloads.bits(y), E4M3)
    # every row of x is identical, so a few rows suffice for all distinct values
    rows = np.array([0, 1, m - 1])
    acc, S = oracle_mod.gemm(qx, sx, E4M3, qy, sy, E4M3, rows=rows)
    out1 = oracle_mod.wgrad(acc, ref[rows])
    ratio = out1 / ref[rows]
    printed = np.array(g["printed_ratio_entries"])
    lo, hi = printed.min(), printed.max()
    # all ratios within the full-mode bound around 2 (S == ref here: all terms >= 0)
    assert np.all(np.abs(ratio - 2.0) <= 2e-3)
    # the printed spread is representative: most entries fall inside it
    inside = np.mean((ratio >= lo - 1e-4) & (ratio <= hi + 1e-4))
    assert inside > 0.5
    assert np.allclose(ratio[0], ratio[1]) and np.allclose(ratio[0], ratio[2])
    # the fix on the page: zero pre-fill gives ratio ~ 1
    out0 = oracle_mod.wgrad(acc, np.zeros_like(ref[rows]))
    assert np.all(np.abs(out0 / ref[rows] - g["with_zeros_prefill_ratio"]) <= 2e-3)


def test_second_accumulate_call_doubles(oracle_mod):
    a = workloads.normal_bf16((16, 256), 9, "a")
    b = workloads.normal_bf16((24, 256), 9, "b")
    qa, sa = oracle_mod.quantize(workloads.bits(a), E4M3)
    qb, sb = oracle_mod.quantize(workloads.bits(b), E4M3)
    acc, _ = oracle_mod.gemm(qa, sa, E4M3, qb, sb, E4M3)
    pre = workloads.normal_f32((16, 24), 9, "pre").double().numpy()
    once = oracle_mod.wgrad(acc, pre)
    twice = oracle_mod.wgrad(acc, once)
    assert np.allclose(twice - pre, 2 * acc, rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle_mod.wgrad(acc, None), acc)


def test_grouped_wgrad_slices_and_zero_groups(oracle_mod):
    M, N = 24, 40
    ks = [256, 0, 384, 128]
    tot = sum(ks)
    a = workloads.normal_bf16((M, tot), 13, "a", std=0.02)
    b = workloads.normal_bf16((N, tot), 13, "b", std=0.02)
    qa, sa = oracle_mod.quantize(workloads.bits(a), E4M3)
    qb, sb = oracle_mod.quantize(workloads.bits(b), E4M3)
    pre = workloads.normal_f32((len(ks), M, N), 13, "pre", std=1e-3).double().numpy()
    out, S = oracle_mod.grouped_wgrad(qa, sa, E4M3, qb, sb, E4M3, ks, prefill=pre)
    A = torch_dequant(qa, sa, E4M3)
    B = torch_dequant(qb, sb, E4M3)
    off = 0
    for g, kg in enumerate(ks):
        ref = pre[g] + A[:, off:off + kg] @ B[:, off:off + kg].T
        assert np.all(np.abs(out[g] - ref) <= 1e-12 * (S[g] + np.abs(pre[g])))
        off += kg
    assert np.array_equal(out[1], pre[1])  # zero-size group leaves out_g unchanged
    assert np.all(S[1] == 0)


def test_moe_group_sizes_recipe():
    for G in (4, 8):
        ks = workloads.moe_group_sizes(G, G * 4096, 1000 + G)
        assert len(ks) == G and sum(ks) == G * 4096 and all(k % 128 == 0 and k >= 0 for k in ks)
    assert workloads.moe_group_sizes(4, 4 * 4096, 5) == workloads.moe_group_sizes(4, 4 * 4096, 5)
