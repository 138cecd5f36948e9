"""fp8_mx_quantize_dbias: the MXFP8 transposed cast of a gradient together with
its bias gradient (db = the column sums of the bf16 gradient, "Replaced
cublasLt calls with rocblas gemm + 6 manually crafted epilogues").

Codes and scale bytes must be bit-identical to fp8_mx_quantize's; db is summed
in the same order as fp8_quantize_dbias's, so it must be bit-identical to that
one's, and within (41 + rows/1024) 2^-24 sum|x| of the oracle's column sums.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu
E4M3, E5M2 = 0, 1
U = 2.0 ** -24


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rows,cols,pad", [(128, 8, 0), (256, 264, 8), (640, 1000, 24), (1024, 512, 0)])
def test_codes_identical_and_db_matches(fp8, fmt, rows, cols, pad):
    full = workloads.normal_bf16((rows, cols + pad), 400 + rows + fmt, "g", std=0.02).cuda()
    x = full[:, :cols]
    out, db = fp8.mx_quantize_dbias(x, fmt)
    ref = fp8.mx_quantize(x, fmt, transpose=True)
    assert torch.equal(out.q, ref.q) and torch.equal(out.sf, ref.sf)
    _, _, db1 = fp8.quantize_dbias(x, fmt)
    assert torch.equal(db, db1)
    xd = oracle.bf16_to_f64(workloads.bits(x.cpu()))
    got = db.cpu().double().numpy()
    assert np.all(np.abs(got - oracle.colsum(xd)) <= (41 + rows // 1024) * U * np.abs(xd).sum(0) + 1e-30)


def test_no_rows_and_short_workspace(fp8):
    db = torch.full((16,), 5.0, device="cuda")
    e = torch.empty((0, 16), dtype=torch.bfloat16, device="cuda")
    fp8.mx_quantize_dbias(e, E5M2, out=fp8.empty_mx(16, 0, E5M2), dbias=db, workspace=torch.empty(4, device="cuda"))
    assert torch.all(db.cpu() == 0.0)
    x = workloads.normal_bf16((256, 64), 401, "s").cuda()
    with pytest.raises(fp8.Fp8Error) as err:
        fp8.mx_quantize_dbias(x, E5M2, workspace=torch.empty(2 * 64 - 1, device="cuda"))
    assert err.value.code == fp8.binding.ERR_WORKSPACE


def test_mx_step_with_the_bias_gradient_in_the_cast(fp8):
    """MxLinearTrainStep's default takes db in dZ's MXFP8 transposed cast: Y, dZ
    and dW bit-identical to the step with the epilogue's sums, db bit-identical
    to the 1x128 cast's sums of the same dZ and within the bf16 rounding of dZ
    of the epilogue's."""
    from fp8_linear_layer_gb300.linear import MxLinearTrainStep
    m, k, n = 512, 384, 640
    X = workloads.normal_bf16((m, k), 83, "X")
    W = workloads.normal_bf16((n, k), 83, "W", std=0.05)
    b = workloads.normal_bf16((n,), 83, "b", std=0.02)
    dY = workloads.normal_bf16((m, k), 83, "dY", std=1e-2)
    args = (X.cuda(), W.cuda(), b.cuda(), dY.cuda())
    ref = MxLinearTrainStep(m, k, n, bias_grad="dgrad")
    st = MxLinearTrainStep(m, k, n)
    assert st.bias_grad == "cast" and st.KERNELS_PER_STEP == ref.KERNELS_PER_STEP == 9
    ref.step(*args)
    st.step(*args)
    torch.cuda.synchronize()
    assert fp8.device_status() == 0
    assert torch.equal(st.dZ, ref.dZ) and torch.equal(st.dW, ref.dW) and torch.equal(st.Y, ref.Y)
    _, _, db1 = fp8.quantize_dbias(st.dZ, E5M2)
    assert torch.equal(st.db, db1)
    dz = st.dZ.double().cpu().numpy()
    mag = np.abs(dz).sum(0)
    assert np.all(np.abs(st.db.cpu().double().numpy() - ref.db.cpu().double().numpy()) <= 2.0 ** -8 * mag + 1e-30)
