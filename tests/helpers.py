"""Shared test utilities: GPU availability, error bounds, sampling.

The bounds follow the stated contract: |gpu - oracle| <= c * S (S = sum_k
|a_ik b_jk| of the dequantized operands), c = 2e-3 in full accumulation and
8e-3 in fast accumulation, plus one bf16 ulp where the output is bf16.
"""
import numpy as np
import torch

FULL_C = 2e-3
FAST_C = 8e-3
MAX_DGELU = 1.13  # max |gelu'(z)| of the tanh GELU, pinned in test_oracle_epilogue


def cuda_ok() -> bool:
    return torch.cuda.is_available()


def bf16_ulp(v) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (2^-133 below the normal range)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


def f32_ulp(v) -> np.ndarray:
    return np.spacing(np.abs(np.asarray(v, dtype=np.float32))).astype(np.float64)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def sample_indices(n: int, k: int, seed: int, tail: bool = True) -> np.ndarray:
    """k distinct sorted indices in [0, n), always including 0 and n-1."""
    rng = np.random.default_rng(seed)
    k = min(k, n)
    idx = set(rng.choice(n, size=k, replace=False).tolist())
    idx.add(0)
    if tail:
        idx.add(n - 1)
    return np.array(sorted(idx), dtype=np.int64)


def assert_within(got, want, bound, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bad = err > bound
    if np.any(bad):
        i = np.argwhere(bad)[0]
        ratio = float(np.max(err / np.maximum(bound, 1e-300)))
        raise AssertionError("%s: %d of %d outside bound; first at %s got %r want %r bound %r; max err/bound %.3f"
                             % (what, int(bad.sum()), bad.size, tuple(i), got[tuple(i)], want[tuple(i)],
                                bound[tuple(i)] if np.ndim(bound) else bound, ratio))
    return float(np.max(err / np.maximum(bound, 1e-300))) if err.size else 0.0


def dgelu_eval_bound(z) -> np.ndarray:
    """Bound on the fp32 evaluation error of gelu'(z) in the kernel (float64
    terms): the kernel forms gelu' = s(2u) + 2 z c (1 + 3a z^2) s(2u) s(-2u) with a
    handful of fp32 operations, the fast exponential intrinsic (documented error
    2 + 1.173|x| ulp, <= 96 ulp for the clamped |x| <= 80) and the approximate
    divide (2 ulp); 2^-16 (256 fp32 ulps) of the sum of the two terms'
    magnitudes bounds it."""
    z = np.asarray(z, dtype=np.float64)
    c = np.sqrt(2.0 / np.pi)
    x = np.clip(2.0 * c * (z + 0.044715 * z ** 3), -80.0, 80.0)
    sp = 1.0 / (1.0 + np.exp(-x))
    sm = 1.0 - sp
    t2 = np.abs(2.0 * z * c * (1.0 + 3 * 0.044715 * z * z) * sp * sm)
    return 2.0 ** -16 * (sp + t2) + 1e-30
