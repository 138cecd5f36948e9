"""fp8_quantize_dbias against the oracle: the transposed cast of a gradient
(and optionally its row cast) together with its bias gradient, db = the column
sums of the bf16 gradient ("Replaced cublasLt calls with rocblas gemm + 6
manually crafted epilogues": db = sum(dY, axis=0), here taken while the
gradient is cast for the weight-gradient GEMM).

Codes and scales must be bit-identical to the plain casts.  Tolerance of db,
from the kernel's arithmetic: a thread adds its 32 values of a column in row
order (31 roundings), the quad combines four parts (2), the finalize adds the
rows/128 partials in eight slices and then the slices (rows/1024 + 7), so
|kernel - oracle| <= (41 + rows/1024) 2^-24 sum|x|.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
U = 2.0 ** -24


def db_bound(rows, x):
    return (41 + rows // 1024) * U * np.abs(x).sum(axis=0) + 1e-30


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rows,cols,pad,with_rows", [(128, 8, 0, False), (256, 264, 8, False),
                                                      (640, 1000, 24, False), (384, 256, 0, True),
                                                      (1024, 640, 64, True)])
def test_codes_identical_and_db_matches_oracle(fp8, fmt, rows, cols, pad, with_rows):
    full = workloads.normal_bf16((rows, cols + pad), 300 + rows + fmt, "g", std=0.02).cuda()
    x = full[:, :cols]
    out, out_t, db = fp8.quantize_dbias(x, fmt, rows=with_rows)
    ref_t = fp8.quantize(x, fmt, transpose=True)
    assert torch.equal(out_t.q, ref_t.q) and torch.equal(out_t.scale[:, :cols], ref_t.scale[:, :cols])
    if with_rows:
        ref = fp8.quantize(x, fmt)
        assert torch.equal(out.q, ref.q) and torch.equal(out.scale[:, :rows], ref.scale[:, :rows])
    else:
        assert out is None
    xd = oracle.bf16_to_f64(workloads.bits(x.cpu()))
    want = oracle.colsum(xd)
    got = db.cpu().double().numpy()
    assert np.all(np.abs(got - want) <= db_bound(rows, xd)), np.abs(got - want).max()


def test_full_size_sampled_columns(fp8):
    # the training step's dZ: 8192 tokens x 14336 features, e5m2
    rows, cols = 8192, 14336
    x = workloads.normal_bf16((rows, cols), 310, "dzfull", std=0.01).cuda()
    _, out_t, db = fp8.quantize_dbias(x, E5M2)
    ref_t = fp8.quantize(x, E5M2, transpose=True)
    assert torch.equal(out_t.q, ref_t.q) and torch.equal(out_t.scale, ref_t.scale)
    idx = np.sort(np.random.default_rng(311).choice(cols, 64, replace=False))
    idx[0], idx[-1] = 0, cols - 1
    xs = oracle.bf16_to_f64(workloads.bits(x[:, torch.from_numpy(idx).cuda()].cpu()))
    want = oracle.colsum(xs)
    got = db.cpu().double().numpy()[idx]
    assert np.all(np.abs(got - want) <= db_bound(rows, xs))


def test_deterministic_edges_and_errors(fp8):
    x = workloads.normal_bf16((1024, 392), 320, "e").cuda()
    _, _, a = fp8.quantize_dbias(x, E4M3)
    _, _, b = fp8.quantize_dbias(x, E4M3)
    assert torch.equal(a, b)
    # a column of equal values sums exactly; a zero column gives zero
    y = torch.zeros((1024, 16), dtype=torch.bfloat16, device="cuda")
    y[:, 3] = 0.375
    y[:, 5] = -2.0
    _, _, d = fp8.quantize_dbias(y, E5M2)
    d = d.cpu()
    assert d[3] == 384.0 and d[5] == -2048.0 and d[0] == 0.0
    # no rows: db is a sum over nothing
    db = torch.full((16,), 5.0, device="cuda")
    e = torch.empty((0, 16), dtype=torch.bfloat16, device="cuda")
    fp8.quantize_dbias(e, E5M2, out_t=fp8.empty_fp8(16, 0, E5M2), dbias=db, workspace=torch.empty(4, device="cuda"))
    assert torch.all(db.cpu() == 0.0)
    # a workspace smaller than (rows/128) x cols floats is refused before any launch
    with pytest.raises(fp8.Fp8Error) as err:
        fp8.quantize_dbias(x, E4M3, workspace=torch.empty(8 * 392 - 1, device="cuda"))
    assert err.value.code == fp8.binding.ERR_WORKSPACE


def test_writes_stay_in_bounds(fp8):
    rows, cols = 512, 200
    x = workloads.normal_bf16((rows, cols), 330, "w").cuda()
    G = 64
    buf = torch.full((cols + 2 * G,), 7.5, dtype=torch.float32, device="cuda")
    wbuf = torch.full(((rows // 128) * cols + 2 * G,), 7.5, dtype=torch.float32, device="cuda")
    fp8.quantize_dbias(x, E5M2, dbias=buf[G:G + cols], workspace=wbuf[G:G + (rows // 128) * cols])
    torch.cuda.synchronize()
    assert torch.all(buf[:G] == 7.5) and torch.all(buf[G + cols:] == 7.5)
    assert torch.all(wbuf[:G] == 7.5) and torch.all(wbuf[G + (rows // 128) * cols:] == 7.5)


@pytest.mark.parametrize("input_grad", [False, True])
def test_train_step_with_the_bias_gradient_in_the_cast(fp8, input_grad):
    """LinearTrainStep(bias_grad="cast"), the default: the data-gradient GEMM
    drops its column sums and the transposed cast of dZ takes db.  Y, dZ, dW
    (and dX) are bit-identical to the step with the epilogue's sums; db is the
    oracle's column sum of its dZ within dZ's bound, and the epilogue's db
    within the same."""
    from fp8_linear_layer_gb300.linear import LinearTrainStep
    from helpers import FULL_C, bf16_ulp, dgelu_eval_bound
    m, k, n = 512, 384, 640
    X = workloads.normal_bf16((m, k), 81, "X")
    W = workloads.normal_bf16((n, k), 81, "W", std=0.05)
    b = workloads.normal_bf16((n,), 81, "b", std=0.02)
    dY = workloads.normal_bf16((m, k), 81, "dY", std=1e-2)
    args = (X.cuda(), W.cuda(), b.cuda(), dY.cuda())
    ref = LinearTrainStep(m, k, n, input_grad=input_grad, bias_grad="dgrad")
    st = LinearTrainStep(m, k, n, input_grad=input_grad)
    assert st.bias_grad == "cast"
    assert st.KERNELS_PER_STEP == ref.KERNELS_PER_STEP == 8
    ref.step(*args)
    st.step(*args)
    if input_grad:
        ref.input_grad(args[1])
        st.input_grad(args[1])
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    assert torch.equal(st.dZ, ref.dZ) and torch.equal(st.dW, ref.dW) and torch.equal(st.Y, ref.Y)
    if input_grad:
        assert torch.equal(st.dX, ref.dX)
    qx, sx = oracle.quantize(workloads.bits(X), E4M3)
    qw, sw = oracle.quantize(workloads.bits(W), E4M3)
    acc, S = oracle.gemm(qx, sx, E4M3, qw, sw, E4M3)
    Zo, _ = oracle.fprop_epilogue(acc, workloads.bits(b))
    zb = oracle.f64_to_bf16_array(Zo)
    qd, sd = oracle.quantize(workloads.bits(dY), E5M2)
    acc2, S2 = oracle.gemm(qd, sd, E5M2, qw, sw, E4M3)
    dzo = oracle.dgrad_epilogue(acc2, zb)
    zbf = oracle.bf16_to_f64(zb)
    g = np.abs(oracle.dgelu(zbf))
    bound_dz = (g * FULL_C * S2 + 0.8 * (FULL_C * S + bf16_ulp(Zo)) * np.abs(acc2)
                + np.abs(acc2) * dgelu_eval_bound(zbf) + 2 * bf16_ulp(np.abs(dzo)))
    tol = bound_dz.sum(0) + (41 + m // 1024) * U * (np.abs(dzo) + bound_dz).sum(0)
    db = st.db.cpu().double().numpy()
    assert np.all(np.abs(db - dzo.sum(0)) <= tol)
    assert np.all(np.abs(db - ref.db.cpu().double().numpy()) <= 2 * tol)


def test_many_tiles_per_cta_ragged(fp8):
    # more tiles than the persistent cast keeps resident CTAs, a ragged last
    # column block and a strided input: codes and scales exact against the
    # oracle, db within the bound above in every column
    rows, cols, pad = 8192, 4104, 24
    base = workloads.normal_bf16((rows, cols + pad), 340, "mtd", std=0.02)
    x = base.cuda()[:, :cols]
    _, out_t, db = fp8.quantize_dbias(x, E5M2)
    torch.cuda.synchronize()
    xb = workloads.bits(base[:, :cols].contiguous())
    qo, so = oracle.quantize(xb, E5M2, transpose=True)
    assert np.array_equal(out_t.q.cpu().numpy(), qo)
    assert np.array_equal(out_t.scale.cpu().numpy()[:, :cols].view(np.uint32), so.view(np.uint32))
    xd = oracle.bf16_to_f64(xb)
    got = db.cpu().double().numpy()
    assert np.all(np.abs(got - oracle.colsum(xd)) <= db_bound(rows, xd))
