"""The device fp8 encoder against the oracle's, over every fp32 bit pattern.

fp8_cast_f32 runs the conversion the casts apply after scaling (round to
nearest even, saturating to +-FMAX, zero keeps its sign) on raw fp32 values.
The oracle encoder is exact rational rounding on the fp8 grid built from the
OCP bit fields.  Both formats ("FP8 GEMM for the fprop should use fast
accumulation": e4m3 forward, e5m2 backward) are compared code for code on all
2^32 patterns except NaNs, which must give a NaN code.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
CHUNK = 1 << 26


def nan_code(fmt, q):
    if fmt == 0:
        return (q & 0x7F) == 0x7F
    return ((q & 0x7C) == 0x7C) & ((q & 0x03) != 0)


@pytest.mark.parametrize("fmt", [0, 1])
def test_encoder_matches_oracle_on_every_fp32_pattern(fp8, fmt):
    xg = torch.empty(CHUNK, dtype=torch.float32, device="cuda")
    qg = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    checked = 0
    for start in range(0, 1 << 32, CHUNK):
        bits = np.arange(start, start + CHUNK, dtype=np.uint32)
        x = bits.view(np.float32)
        xg.copy_(torch.from_numpy(x))
        fp8.cast_f32(xg, fmt, out=qg)
        got = qg.cpu().numpy()
        want = oracle.encode(fmt, x)
        # NaN patterns: exponent all ones, mantissa not zero (either sign)
        nan = (bits & 0x7FFFFFFF) > 0x7F800000 if (start & 0x7FFFFFFF) + CHUNK > 0x7F800000 else None
        if nan is None:
            same = np.array_equal(got, want)
        else:
            same = np.array_equal(got[~nan], want[~nan])
            assert nan_code(fmt, got[nan]).all()
        if not same:
            bad = got != want if nan is None else (got != want) & ~nan
            i = int(np.argmax(bad))
            raise AssertionError("fmt %d: fp32 0x%08x (%r) -> 0x%02x, oracle 0x%02x"
                                 % (fmt, int(bits[i]), float(x[i]), int(got[i]), int(want[i])))
        checked += CHUNK - (0 if nan is None else int(nan.sum()))
    assert checked == (1 << 32) - 2 * ((1 << 23) - 1)
