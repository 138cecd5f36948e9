"""Pins for the oracle's per-128-block cast (CPU only).

The per-token cast on the DeepGEMM page ("Weight gradient kernels for dense and
MoE models", worked example) is named but not defined; the reading is: per row
and 128-element block, amax = max|x|, inv = fl32(FMAX/amax),
scale = fl32(amax/FMAX), q = enc(fl32(x * inv)).  The pins below are closed
forms and invariants that any correct implementation of that reading meets.
"""
import numpy as np
import pytest
import torch

import workloads

E4M3, E5M2 = 0, 1
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}
FMAX = {E4M3: 448.0, E5M2: 57344.0}


def to_bits(t):
    return workloads.bits(t)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_all_ones_closed_form(oracle_mod, fmt):
    x = torch.ones(3, 256, dtype=torch.bfloat16)
    q, s = oracle_mod.quantize(to_bits(x), fmt)
    assert np.all(q == MAXCODE[fmt])
    assert np.all(s == np.float32(1.0) / np.float32(FMAX[fmt]))
    assert s.shape == (2, 3)


def test_hand_worked_block(oracle_mod):
    # amax = 4 -> inv = 448/4 = 112 exactly, scale = 4/448 in fp32.
    v = np.zeros(128, dtype=np.float32)
    v[:6] = [4.0, -2.0, 1.0, 0.5, 0.03125, -4.0]
    x = torch.from_numpy(v).to(torch.bfloat16)[None, :]
    q, s = oracle_mod.quantize(to_bits(x), E4M3)
    # 448 -> 0x7E; -224 = -1.75*2^7 -> 0xF6; 112 = 1.75*2^6 -> 0x6E; 56 -> 0x66;
    # 3.5 = 1.75*2^1 -> 0x46; -448 -> 0xFE; zeros stay +0.
    assert list(q[0, :6]) == [0x7E, 0xF6, 0x6E, 0x66, 0x46, 0xFE]
    assert np.all(q[0, 6:] == 0)
    assert s[0, 0] == np.float32(4.0) / np.float32(448.0)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_zero_block_and_signed_zero(oracle_mod, fmt):
    x = torch.zeros(2, 128, dtype=torch.bfloat16)
    x[1] = -x[1]  # the whole second row is -0
    q, s = oracle_mod.quantize(to_bits(x), fmt)
    assert np.all(s == 1.0)
    assert np.all(q[0] == 0x00) and np.all(q[1] == 0x80)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_tiny_block_takes_unit_scale(oracle_mod, fmt):
    # FMAX/amax overflows binary32 -> scale 1, values encode to signed zero
    x = torch.zeros(1, 128, dtype=torch.float32)
    x[0, 0], x[0, 1] = 1e-38, -5e-39
    q, s = oracle_mod.quantize(to_bits(x.to(torch.bfloat16)), fmt)
    assert s[0, 0] == 1.0 and q[0, 0] == 0x00 and q[0, 1] == 0x80


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_invariants_random(oracle_mod, fmt):
    x = workloads.normal_bf16((64, 512), 11, "q", std=3.0)
    x[5, 128:256] = 0  # a zero block
    q, s = oracle_mod.quantize(to_bits(x), fmt)
    xf = x.double().numpy()
    dec = oracle_mod.decode(fmt, q)
    t = oracle_mod.decode_table(fmt)
    for r in range(64):
        for b in range(4):
            blk = slice(128 * b, 128 * b + 128)
            amax = np.abs(xf[r, blk]).max()
            if amax == 0:
                assert s[b, r] == 1.0
                continue
            # scale definition and max code
            assert s[b, r] == np.float32(amax) / np.float32(FMAX[fmt])
            assert (q[r, blk] & 0x7F).max() == MAXCODE[fmt]
            # reconstruction: dec(q) is the nearest fp8 value to x*inv
            inv = np.float32(FMAX[fmt]) / np.float32(amax)
            y = (xf[r, blk].astype(np.float32) * inv).astype(np.float64)
            d = np.abs(dec[r, blk] - y)
            # distance to every finite code is no smaller than to the chosen one
            fin = t[np.isfinite(t)]
            best = np.min(np.abs(fin[None, :] - y[:, None]), axis=1)
            assert np.all(d == best)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_transposed_equals_rowwise_of_transpose(oracle_mod, fmt):
    x = workloads.normal_bf16((256, 200), 5, "t")
    qt, st = oracle_mod.quantize(to_bits(x), fmt, transpose=True)
    qr, sr = oracle_mod.quantize(to_bits(x.t().contiguous()), fmt, transpose=False)
    assert qt.shape == (200, 256) and st.shape == (2, 200)
    assert np.array_equal(qt, qr) and np.array_equal(st, sr)


def test_scale_layout_blocks_by_rows(oracle_mod):
    # block b of row r lands at scale[b][r]; blocks scaled differently per row
    x = torch.ones(3, 384, dtype=torch.float32)
    for r in range(3):
        for b in range(3):
            x[r, 128 * b:128 * (b + 1)] *= 2.0 ** (r + 4 * b)
    q, s = oracle_mod.quantize(to_bits(x.to(torch.bfloat16)), E4M3)
    for r in range(3):
        for b in range(3):
            assert s[b, r] == np.float32(2.0 ** (r + 4 * b)) / np.float32(448.0)
