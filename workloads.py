"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module draws random numbers and rounds them to bf16; it holds none of the
method's arithmetic (no quantization, no GEMM, no epilogue).  Both the CUDA
path and the CPU oracle consume exactly the bf16 bytes produced here.

Every draw uses its own ``torch.Generator('cpu')`` seeded from a base seed and
a tensor tag, so a tensor never depends on which other tensors were drawn.

Workload shapes are those of the DeepGEMM weight-gradient tables ("Weight
gradient kernels for dense and MoE models", dense and grouped tables) and of
a transformer MLP linear layer (tokens 8192, in 4096, out 14336).
"""
import zlib

import numpy as np
import torch

# (M, N) pairs of the dense weight-gradient table; each is run at K = 4096 and 8192.
DENSE_WGRAD_MN = [(7168, 2112), (1536, 24576), (512, 32768), (16384, 7168), (7168, 4096), (2048, 7168)]
DENSE_WGRAD_K = [4096, 8192]
# (G, M, N, tokens per expert on average) rows of the grouped table.
GROUPED_WGRAD = [(4, 7168, 4096, 4096), (4, 2048, 7168, 4096), (4, 7168, 4096, 8192),
                 (4, 2048, 7168, 8192), (8, 7168, 4096, 4096), (8, 2048, 7168, 4096)]
# Linear-layer training step: tokens m, in-features k, out-features n.
TRAIN_STEP = dict(m=8192, k=4096, n=14336)


def _seed(base: int, tag: str) -> int:
    return (int(base) * 1000003 + zlib.crc32(tag.encode())) & 0x7FFFFFFFFFFF


def _gen(base: int, tag: str) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(_seed(base, tag))
    return g


def normal_bf16(shape, base: int, tag: str, std: float = 1.0) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws (drawn in fp32, rounded to nearest even)."""
    x = torch.randn(*shape, generator=_gen(base, tag), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def uniform_bf16(shape, base: int, tag: str) -> torch.Tensor:
    """bf16 tensor of U[0, 1) draws (as torch.rand)."""
    return torch.rand(*shape, generator=_gen(base, tag), dtype=torch.float32).to(torch.bfloat16)


def normal_f32(shape, base: int, tag: str, std: float = 1.0) -> torch.Tensor:
    x = torch.randn(*shape, generator=_gen(base, tag), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x


def with_outlier_rows(x: torch.Tensor, base: int, tag: str, frac: float = 0.01,
                      factor: float = 64.0):
    """Scale a seeded random ``frac`` of the rows of x by ``factor`` (in fp32,
    rounded back to bf16).  Returns (tensor, sorted row indices)."""
    rows = x.shape[0]
    n_out = max(1, int(round(rows * frac)))
    perm = torch.randperm(rows, generator=_gen(base, tag + "/rows"))
    idx = torch.sort(perm[:n_out]).values
    y = x.clone()
    y[idx] = (y[idx].float() * factor).to(torch.bfloat16)
    return y, idx.numpy()


def moe_group_sizes(G: int, total: int, base: int, tag: str = "moe", multiple: int = 128):
    """Per-expert token counts: a multinomial draw of ``total`` tokens over G
    equally likely experts, rounded to multiples of ``multiple`` by the
    largest-remainder rule so the sum stays ``total``.  Zero is allowed."""
    assert total % multiple == 0
    probs = torch.full((G,), 1.0 / G, dtype=torch.float64)
    draws = torch.multinomial(probs, total, replacement=True, generator=_gen(base, tag))
    counts = torch.bincount(draws, minlength=G).numpy().astype(np.int64)
    units = total // multiple
    exact = counts / multiple
    base_units = np.floor(exact).astype(np.int64)
    rem = exact - base_units
    short = units - int(base_units.sum())
    order = np.argsort(-rem, kind="stable")
    base_units[order[:short]] += 1
    return [int(u * multiple) for u in base_units]


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns, contiguous."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

