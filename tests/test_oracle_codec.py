"""Pins for the oracle's fp8 / bf16 codec (CPU only).

The pages only name e4m3 (forward) and e5m2 (gradients) ("FP8 GEMM for the
fprop should use fast accumulation"); the bit layouts are the OCP FP8 ones.
The decode table is pinned against torch's float8 dtypes (a library routine),
the encoder against torch's float32 -> float8 casts inside the finite range,
and separately against ties-to-even and saturation special cases.
"""
import numpy as np
import pytest
import torch

E4M3, E5M2 = 0, 1
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
MAXCODE = {E4M3: 0x7E, E5M2: 0x7B}


def torch_decode(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_table_matches_torch(oracle_mod, fmt):
    ours = oracle_mod.decode_table(fmt)
    ref = torch_decode(fmt)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_decode_special_values(oracle_mod):
    t4 = oracle_mod.decode_table(E4M3)
    assert t4[0x7E] == 448.0 and t4[0x01] == 2.0 ** -9 and t4[0x08] == 2.0 ** -6 and t4[0x38] == 1.0
    assert np.isnan(t4[0x7F]) and np.isnan(t4[0xFF]) and t4[0x80] == 0.0 and np.signbit(t4[0x80])
    t5 = oracle_mod.decode_table(E5M2)
    assert t5[0x7B] == 57344.0 and t5[0x01] == 2.0 ** -16 and t5[0x3C] == 1.0
    assert np.isinf(t5[0x7C]) and all(np.isnan(t5[c]) for c in (0x7D, 0x7E, 0x7F))
    assert oracle_mod.fp8_max(E4M3) == 448.0 and oracle_mod.fp8_max(E5M2) == 57344.0


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_roundtrip_and_monotone(oracle_mod, fmt):
    t = oracle_mod.decode_table(fmt)
    finite = [c for c in range(256) if np.isfinite(t[c])]
    vals = t[finite].astype(np.float32)
    assert np.array_equal(oracle_mod.encode(fmt, vals), np.array(finite, dtype=np.uint8))
    pos = t[: MAXCODE[fmt] + 1]
    assert np.all(np.diff(pos) > 0)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_ties_to_even_at_every_midpoint(oracle_mod, fmt):
    t = oracle_mod.decode_table(fmt)
    lo = np.arange(0, MAXCODE[fmt])
    mid = ((t[lo] + t[lo + 1]) / 2).astype(np.float32)
    assert np.all(mid.astype(np.float64) == (t[lo] + t[lo + 1]) / 2)  # midpoints exact in fp32
    got = oracle_mod.encode(fmt, mid)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    got_neg = oracle_mod.encode(fmt, -mid)
    assert np.array_equal(got_neg, want | 0x80)
    # just off the midpoint goes to the nearer side
    up = np.nextafter(mid, np.float32(np.inf))
    dn = np.nextafter(mid, np.float32(0))
    assert np.array_equal(oracle_mod.encode(fmt, up), (lo + 1).astype(np.uint8))
    assert np.array_equal(oracle_mod.encode(fmt, dn), lo.astype(np.uint8))


def test_saturation_and_signed_zero(oracle_mod):
    assert list(oracle_mod.encode(E4M3, [448, 449, 463.9, 464, 480, 1e6, 3e38, -1e6])) == \
        [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE]
    assert list(oracle_mod.encode(E5M2, [57344, 61439, 61440, 1e9, -1e9])) == [0x7B, 0x7B, 0x7B, 0x7B, 0xFB]
    assert list(oracle_mod.encode(E4M3, [0.0, -0.0, 1e-30, -1e-30, 2.0 ** -10, 2.0 ** -10 * 1.0001])) == \
        [0x00, 0x80, 0x00, 0x80, 0x00, 0x01]
    assert list(oracle_mod.encode(E5M2, [2.0 ** -17, -(2.0 ** -17) * 1.0001])) == [0x00, 0x81]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_cast_in_range(oracle_mod, fmt):
    g = torch.Generator().manual_seed(7 + fmt)
    fmax = oracle_mod.fp8_max(fmt)
    # log-uniform magnitudes over the whole fp8 range and beyond its subnormals
    n = 400_000
    e = torch.rand(n, generator=g, dtype=torch.float64) * (np.log2(fmax) + 20) - 20
    s = torch.where(torch.rand(n, generator=g) < 0.5, -1.0, 1.0).double()
    x = (s * torch.exp2(e)).float()
    x = x[x.abs() <= fmax]  # torch's cast does not saturate: compare inside the range only
    ours = oracle_mod.encode(fmt, x.numpy())
    ref = x.to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_helpers(oracle_mod):
    # bf16 -> f64 is a bit shift; f64 -> bf16 rounds to nearest even
    x = torch.randn(10000, generator=torch.Generator().manual_seed(3)) * 100
    b = x.to(torch.bfloat16)
    bits = b.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle_mod.bf16_to_f64(bits), b.double().numpy())
    for v in x.numpy()[:2000]:  # fp32 inputs: torch's fp32 -> bf16 cast is single rounding
        want = int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)[0])
        assert oracle_mod.f64_to_bf16(float(v)) == want
    arr = oracle_mod.f64_to_bf16_array(x.numpy()[:2000].astype(np.float64))
    assert [int(a) for a in arr] == [oracle_mod.f64_to_bf16(float(v)) for v in x.numpy()[:2000]]
    # tie to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert oracle_mod.f64_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    assert oracle_mod.f64_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
