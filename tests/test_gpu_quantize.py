"""GPU quantize kernels vs the oracle: bytes and scale bits must match exactly.

Reading of the per-token cast ("Weight gradient kernels for dense and MoE
models"): per 128-block amax, inv = fl32(FMAX/amax), scale = fl32(amax/FMAX),
q = RNE-saturating fp8(fl32(x * inv)).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def gpu_quant(fp8, x, fmt, transpose):
    t = fp8.quantize(x.cuda(), fmt, transpose=transpose)
    torch.cuda.synchronize()
    return t.q.cpu().numpy(), t.scale.cpu().numpy()


def check_exact(fp8, x, fmt, transpose):
    q, s = gpu_quant(fp8, x, fmt, transpose)
    qo, so = oracle.quantize(workloads.bits(x), fmt, transpose=transpose)
    n = qo.shape[0]
    assert q.shape == qo.shape
    assert np.array_equal(q, qo), "codes differ at %s" % (np.argwhere(q != qo)[:5].tolist(),)
    assert np.array_equal(s[:, :n].view(np.uint32), so.view(np.uint32)), "scale bits differ"


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(1, 128), (3, 384), (77, 640), (256, 4096), (1000, 1152)])
def test_rowwise_exact(fp8, fmt, shape):
    x = workloads.normal_bf16(shape, 100 + fmt, "rq", std=2.0)
    check_exact(fp8, x, fmt, False)


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(128, 8), (128, 200), (384, 136), (1024, 1000), (256, 4096)])
def test_transposed_exact(fp8, fmt, shape):
    x = workloads.normal_bf16(shape, 200 + fmt, "tq", std=0.5)
    check_exact(fp8, x, fmt, True)


def check_dual(fp8, x, fmt):
    """Both outputs of the one-read cast: exact against the oracle's row and
    transposed casts, and bit-identical to the two separate kernels."""
    xd = x.cuda()
    tr, tc = fp8.quantize_dual(xd, fmt)
    sr, sc = fp8.quantize(xd, fmt), fp8.quantize(xd, fmt, transpose=True)
    torch.cuda.synchronize()
    rows, cols = x.shape
    for t, s, transpose, n in ((tr, sr, False, rows), (tc, sc, True, cols)):
        q, sb = t.q.cpu().numpy(), t.scale.cpu().numpy()[:, :n]
        qo, so = oracle.quantize(workloads.bits(x), fmt, transpose=transpose)
        assert np.array_equal(q, qo), "codes differ at %s" % (np.argwhere(q != qo)[:5].tolist(),)
        assert np.array_equal(sb.view(np.uint32), so.view(np.uint32)), "scale bits differ"
        assert torch.equal(t.q, s.q)
        assert np.array_equal(sb.view(np.uint32), s.scale.cpu().numpy()[:, :n].view(np.uint32))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("shape", [(128, 128), (256, 384), (640, 256), (1024, 1152)])
def test_dual_exact(fp8, fmt, shape):
    x = workloads.normal_bf16(shape, 400 + fmt, "dq", std=1.5)
    check_dual(fp8, x, fmt)


@pytest.mark.parametrize("fmt", [0, 1])
def test_dual_strided_and_special(fp8, fmt):
    # a row stride wider than the matrix, plus the special blocks of the test below
    x = workloads.normal_bf16((256, 640), 9, "dsp", std=1.0).float()
    x[0, :] = 0.0
    x[1, :128] = -0.0
    x[2, :128] = 1e-38
    x[3, 128:256] = 3e38
    x[:, 9] *= 64.0
    x[:128, 300] = 0.0
    wide = torch.zeros((256, 768), dtype=torch.bfloat16)
    wide[:, :640] = x.to(torch.bfloat16)
    xv = wide.cuda()[:, :640]
    tr, tc = fp8.quantize_dual(xv, fmt)
    torch.cuda.synchronize()
    xb = x.to(torch.bfloat16)
    for t, transpose, n in ((tr, False, 256), (tc, True, 640)):
        qo, so = oracle.quantize(workloads.bits(xb), fmt, transpose=transpose)
        assert np.array_equal(t.q.cpu().numpy(), qo)
        assert np.array_equal(t.scale.cpu().numpy()[:, :n].view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("fmt", [0, 1])
@pytest.mark.parametrize("transpose", [False, True])
def test_special_blocks(fp8, fmt, transpose):
    # zero blocks, signed zeros, tiny blocks (FMAX/amax overflows), huge values,
    # subnormal bf16, ties, outlier rows and columns
    x = workloads.normal_bf16((256, 512), 7, "sp", std=1.0).float()
    x[0, :] = 0.0
    x[1, :] = -0.0
    x[2, :128] = 1e-38
    x[2, 5] = -3e-39
    x[3, :] = 3e38
    x[3, 7] = -1.0
    x[4, :] = 2.0 ** -130
    x[5, :] *= 1e4
    x[:, 9] *= 64.0
    x[6, :] = torch.arange(512, dtype=torch.float32) / 7.0
    xb = x.to(torch.bfloat16)
    check_exact(fp8, xb, fmt, transpose)


@pytest.mark.parametrize("fmt", [0, 1])
def test_full_size_rowwise_sampled(fp8, fmt):
    # the widest operand of the dense weight-gradient table: 32768 x 8192
    rows, cols = 32768, 8192
    x = workloads.normal_bf16((rows, cols), 300 + fmt, "big", std=0.02)
    t = fp8.quantize(x.cuda(), fmt)
    torch.cuda.synchronize()
    idx = np.array([0, 1, 4095, 12345, 20000, rows - 1])
    qo, so = oracle.quantize(workloads.bits(x[idx]), fmt)
    q = t.q[torch.from_numpy(idx).cuda()].cpu().numpy()
    s = t.scale[:, torch.from_numpy(idx).cuda()].cpu().numpy()
    assert np.array_equal(q, qo)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))
    # invariant at any size: every non-zero block holds the maximum code
    maxcode = 0x7E if fmt == 0 else 0x7B
    blk = (t.q.view(rows, cols // 128, 128) & 0x7F).amax(dim=2)
    assert bool((blk == maxcode).all())


def test_full_size_transposed_sampled(fp8):
    # token-major operand of the training step's weight gradient: X^T of 8192 x 4096
    rows, cols = 8192, 4096
    x = workloads.normal_bf16((rows, cols), 301, "bigT")
    t = fp8.quantize(x.cuda(), 0, transpose=True)
    torch.cuda.synchronize()
    cidx = np.array([0, 1, 777, 2048, cols - 1])
    qo, so = oracle.quantize(workloads.bits(x[:, cidx]), 0, transpose=True)
    q = t.q[torch.from_numpy(cidx).cuda()].cpu().numpy()
    s = t.scale[:, torch.from_numpy(cidx).cuda()].cpu().numpy()
    assert np.array_equal(q, qo)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))


def test_strided_input(fp8):
    base = workloads.normal_bf16((64, 1024 + 64), 9, "ld")
    x = base[:, :1024]  # row stride 1088 elements
    assert x.stride(0) == 1088
    t = fp8.quantize(x.cuda(), 0)
    torch.cuda.synchronize()
    qo, so = oracle.quantize(workloads.bits(x.contiguous()), 0)
    assert np.array_equal(t.q.cpu().numpy(), qo)


@pytest.mark.parametrize("fmt", [0, 1])
def test_transposed_many_tiles_per_cta_ragged(fp8, fmt):
    # 64 row blocks x 33 column blocks (the last 8 columns wide) on a strided
    # input: more tiles than the persistent cast keeps resident CTAs, so each
    # CTA casts several tiles through both shared-memory stages and the ragged
    # column block lands on different CTAs at different iterations.  Every code
    # and scale is checked.
    rows, cols, pad = 8192, 4104, 24
    assert (rows // 128) * ((cols + 127) // 128) > 4 * 152 * 3
    base = workloads.normal_bf16((rows, cols + pad), 500 + fmt, "mt", std=0.7)
    x = base.cuda()[:, :cols]
    t = fp8.quantize(x, fmt, transpose=True)
    torch.cuda.synchronize()
    qo, so = oracle.quantize(workloads.bits(base[:, :cols].contiguous()), fmt, transpose=True)
    q, s = t.q.cpu().numpy(), t.scale.cpu().numpy()[:, :cols]
    assert np.array_equal(q, qo), "codes differ at %s" % (np.argwhere(q != qo)[:5].tolist(),)
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32)), "scale bits differ"
