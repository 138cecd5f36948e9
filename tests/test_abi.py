"""The C-ABI library builds, loads and exports every symbol include/fp8ll.h
declares; host-side validation rejects bad arguments before any device work.
CPU only: no call here reaches a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "fp8ll.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    import fp8_linear_layer_gb300.build as b
    b.build()
    import fp8_linear_layer_gb300 as f
    return f.lib()


def test_header_declares_the_expected_calls():
    names = header_functions()
    for n in ("fp8_quantize", "fp8_gemm_fprop", "fp8_gemm_dgrad", "fp8_gemm_wgrad", "fp8_grouped_wgrad"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    import fp8_linear_layer_gb300 as f
    names = header_functions()
    assert sorted(f.EXPORTS) == names
    for n in names:
        assert hasattr(L, n), n


def test_scale_ld_and_workspace(L):
    import fp8_linear_layer_gb300 as f
    assert [f.scale_ld(r) for r in (1, 4, 5, 101, 128)] == [4, 4, 8, 104, 128]
    assert f.workspace_size(8192, 14336) == 64 * 4 * 14336 * 4
    assert f.workspace_size(1, 1) == 4 * 4
    assert f.workspace_size(0, 5) == 0


def test_status_strings(L):
    import fp8_linear_layer_gb300 as f
    assert f.status_string(0) == "ok"
    assert "timed out" in f.status_string(-4)
    assert f.status_string(12345) == "unknown status"
    assert "scratch" in f.status_string(f.binding.ERR_SCRATCH)


def test_invalid_arguments_rejected_on_host(L):
    import fp8_linear_layer_gb300 as f
    E = f.binding.ERR_INVALID_ARG
    vp = ctypes.c_void_p
    fake = vp(0x10000)  # never dereferenced: validation fails first
    # quantize: bad format, misaligned pointer, cols not a multiple of 128
    assert L.fp8_quantize(fake, 4, 128, 128, 7, 0, fake, fake, 4, None) == E
    assert L.fp8_quantize(vp(0x10002), 4, 128, 128, 0, 0, fake, fake, 4, None) == E
    assert L.fp8_quantize(fake, 4, 100, 128, 0, 0, fake, fake, 4, None) == E
    assert L.fp8_quantize(fake, 100, 128, 128, 0, 1, fake, fake, 128, None) == E  # rows % 128 != 0
    assert L.fp8_quantize(fake, 4, 128, 128, 0, 0, fake, fake, 3, None) == E      # scale_ld too small
    assert L.fp8_quantize(None, 0, 0, 0, 0, 0, None, None, 0, None) == 0          # empty is a no-op
    # dual cast: both dimensions multiples of 128, both scale leading dimensions checked
    assert L.fp8_quantize_dual(fake, 128, 200, 200, 0, fake, fake, 128, fake, fake, 200, None) == E  # cols % 128
    assert L.fp8_quantize_dual(fake, 100, 256, 256, 0, fake, fake, 100, fake, fake, 256, None) == E  # rows % 128
    assert L.fp8_quantize_dual(fake, 128, 256, 256, 2, fake, fake, 128, fake, fake, 256, None) == E  # format
    assert L.fp8_quantize_dual(fake, 128, 256, 256, 0, fake, fake, 124, fake, fake, 256, None) == E  # row scales
    assert L.fp8_quantize_dual(fake, 128, 256, 256, 0, fake, fake, 128, fake, fake, 252, None) == E  # col scales
    assert L.fp8_quantize_dual(fake, 128, 256, 200, 0, fake, fake, 128, fake, fake, 256, None) == E  # ldx < cols
    assert L.fp8_quantize_dual(fake, 128, 256, 256, 0, vp(0x10008), fake, 128, fake, fake, 256, None) == E
    assert L.fp8_quantize_dual(fake, 128, 256, 256, 0, fake, fake, 128, None, fake, 256, None) == E
    assert L.fp8_quantize_dual(None, 0, 256, 256, 0, None, None, 0, None, None, 0, None) == 0        # empty
    op = f.binding.OperandStruct(0x10000, 0x20000, 256, 8, 0, 0)
    bad = f.binding.OperandStruct(0x10000, 0x20000, 200, 8, 0, 0)   # ld_q % 16 != 0
    ob, oo = ctypes.byref(op), ctypes.byref(bad)
    assert L.fp8_gemm_fprop(8, 8, 256, ob, oo, fake, 2, 0, fake, fake, None) == E
    assert L.fp8_gemm_fprop(8, 8, 200, ob, ob, fake, 2, 0, fake, fake, None) == E   # K % 128
    assert L.fp8_gemm_fprop(8, 8, 256, ob, ob, None, 2, 0, fake, fake, None) == E   # bias missing
    assert L.fp8_gemm_fprop(8, 8, 256, ob, ob, fake, 3, 0, fake, fake, None) == E   # dgrad epilogue
    assert L.fp8_gemm_fprop(8, 8, 256, ob, ob, fake, 2, 5, fake, fake, None) == E   # bad acc mode
    assert L.fp8_gemm_fprop(0, 8, 256, ob, ob, fake, 2, 0, fake, fake, None) == E   # M = 0
    assert L.fp8_gemm_fprop(8, 8, 256, ob, ob, fake, 2, 0, fake, fake, None) == E   # Y and Z share a buffer
    assert L.fp8_gemm_dgrad(8, 8, 256, ob, ob, fake, 4, 0, fake, fake, fake, 4, None) == f.binding.ERR_WORKSPACE
    assert L.fp8_gemm_dgrad(8, 8, 256, ob, ob, None, 3, 0, fake, None, None, 0, None) == E  # aux missing
    ks = (ctypes.c_int64 * 2)(128, 100)
    assert L.fp8_grouped_wgrad(2, 8, 8, ks, ob, ob, fake, 1, 0, None) == E              # K_g % 128
    ks0 = (ctypes.c_int64 * 1)(128)
    assert L.fp8_grouped_wgrad(0, 8, 8, ks0, ob, ob, fake, 1, 0, None) == E
    assert L.fp8_grouped_wgrad(1, 8, 8, ks0, ob, ob, fake, 2, 0, None) == E             # accumulate flag
    assert L.fp8_debug_starve_next_gemm(0) == E
    # the no-allocation data gradient checks arguments exactly as fp8_gemm_dgrad does, so a bad
    # call gets the same code from both even when M x N is beyond its built-in scratch
    nz = L.fp8_gemm_dgrad_noalloc
    assert nz(8, 8, 256, ob, oo, fake, 4, 0, fake, fake, None) == E                      # bad operand
    assert nz(8, 8, 200, ob, ob, fake, 4, 0, fake, fake, None) == E                      # K % 128
    big = ctypes.byref(f.binding.OperandStruct(0x10000, 0x20000, 256, 65536, 0, 0))  # scales for 65536 rows
    assert nz(4096, 65536, 256, big, oo, fake, 4, 0, fake, fake, None) == E              # bad operand, large
    assert nz(4096, 65536, 256, big, big, fake, 4, 0, fake, None, None) == E             # no bgrad, large
    assert nz(4096, 65536, 256, big, big, fake, 4, 0, fake, fake, None) == f.binding.ERR_WORKSPACE
    assert nz(8, 8, 256, ob, ob, fake, 9, 0, fake, fake, None) == E                      # epilogue
    # the data gradient that casts its own output: N % 128, scale_ld, overlapping outputs
    dq = L.fp8_gemm_dgrad_quant
    op8 = ctypes.byref(f.binding.OperandStruct(0x10000, 0x20000, 256, 8, 1, 0))
    wide = ctypes.byref(f.binding.OperandStruct(0x10000, 0x20000, 256, 256, 0, 0))
    outp, auxp, qp, sp = vp(0x1000000), vp(0x2000000), vp(0x3000000), vp(0x4000000)
    assert dq(8, 200, 256, op8, wide, auxp, 0, outp, qp, sp, 8, None) == E               # N % 128
    assert dq(8, 256, 256, op8, wide, auxp, 0, outp, qp, sp, 4, None) == E               # scale_ld < M
    assert dq(8, 256, 256, op8, wide, auxp, 0, outp, vp(0x1000000 + 64), sp, 8, None) == E   # q inside dZ
    assert dq(8, 256, 256, op8, wide, auxp, 0, outp, qp, vp(0x2000000 + 16), 8, None) == E   # scales inside Z
    assert dq(8, 256, 256, op8, wide, auxp, 3, outp, qp, sp, 8, None) == E               # accumulation mode


def test_tensor_scaling_validation(L):
    import fp8_linear_layer_gb300 as f
    E = f.binding.ERR_INVALID_ARG
    vp = ctypes.c_void_p
    fake, other, sc = vp(0x10000), vp(0x20000), vp(0x40000)
    # amax: misaligned result, cols % 8
    assert L.fp8_tensor_amax(fake, 4, 128, 128, vp(0x10002), None) == E
    assert L.fp8_tensor_amax(fake, 4, 100, 128, other, None) == E
    # cast: no output, amax_out aliasing amax_in, rows-layout cols % 16,
    # transposed rows % 128, both orientations with cols % 128
    assert L.fp8_tensor_quantize(fake, 128, 256, 256, 0, other, None, None, sc, None, None) == E
    assert L.fp8_tensor_quantize(fake, 128, 256, 256, 0, other, fake, None, fake, other, None) == E
    assert L.fp8_tensor_quantize(fake, 128, 256, 256, 0, other, fake, None, other, None, None) == E  # scale = amax_in
    assert L.fp8_tensor_quantize(fake, 128, 256, 256, 0, other, fake, None, vp(0x30000), vp(0x30000), None) == E
    assert L.fp8_tensor_quantize(fake, 128, 200, 200, 0, other, fake, None, sc, None, None) == E
    assert L.fp8_tensor_quantize(fake, 100, 256, 256, 0, other, None, fake, sc, None, None) == E
    assert L.fp8_tensor_quantize(fake, 128, 136, 136, 0, other, fake, fake, sc, None, None) == E
    assert L.fp8_tensor_quantize(fake, 128, 256, 256, 3, other, fake, None, sc, None, None) == E
    assert L.fp8_tensor_quantize(None, 0, 256, 256, 0, None, None, None, None, None, None) == 0  # empty
    # history: empty history
    assert L.fp8_amax_history_update(fake, 1, 0, other, other, None) == E
    assert L.fp8_amax_history_update(fake, 0, 4, other, other, None) == E
    # GEMMs: ld_q % 16, missing scale, K % 128, dgrad workspace
    op = f.binding.TensorOperandStruct(0x10000, 0x20000, 256, 0, 0)
    bad = f.binding.TensorOperandStruct(0x10000, 0x20000, 200, 0, 0)
    noscale = f.binding.TensorOperandStruct(0x10000, None, 256, 0, 0)
    ob = ctypes.byref(op)
    assert L.fp8_tensor_gemm_fprop(8, 8, 256, ob, ctypes.byref(bad), fake, 2, fake, fake, None) == E
    assert L.fp8_tensor_gemm_fprop(8, 8, 256, ob, ctypes.byref(noscale), fake, 2, fake, fake, None) == E
    assert L.fp8_tensor_gemm_fprop(8, 8, 200, ob, ob, fake, 2, fake, fake, None) == E
    assert L.fp8_tensor_gemm_dgrad(8, 8, 256, ob, ob, fake, 4, fake, fake, fake, 4, None) == f.binding.ERR_WORKSPACE
    assert L.fp8_tensor_gemm_wgrad(8, 8, 256, ob, ob, fake, 2, None) == E


def test_mx_sizes_and_validation(L):
    import fp8_linear_layer_gb300 as f
    # groups of 128 rows, rounded up to an even count, 512 bytes per group and K block
    assert f.mx_sf_bytes(256, 128) == 2 * 512
    assert f.mx_sf_bytes(300, 4096) == 32 * 4 * 512
    assert f.mx_sf_bytes(1, 256) == 2 * 2 * 512
    assert f.mx_sf_bytes(0, 128) == 0 and f.mx_sf_bytes(128, 100) == 0
    E = f.binding.ERR_INVALID_ARG
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    # rows cast needs cols % 128 == 0; transposed needs rows % 128 == 0
    assert L.fp8_mx_quantize(fake, 4, 100, 104, 0, 0, fake, fake, None) == E
    assert L.fp8_mx_quantize(fake, 100, 64, 64, 0, 1, fake, fake, None) == E
    assert L.fp8_mx_quantize(fake, 4, 128, 128, 7, 0, fake, fake, None) == E
    op = f.binding.MxOperandStruct(0x10000, 0x10000, 256, 0, 0)
    bad = f.binding.MxOperandStruct(0x10000, 0x10008, 256, 0, 0)  # misaligned scales
    out = vp(0x20000)
    assert L.fp8_mx_gemm_wgrad(128, 128, 100, ctypes.byref(op), ctypes.byref(op), out, 1, None) == E
    assert L.fp8_mx_gemm_wgrad(128, 128, 256, ctypes.byref(bad), ctypes.byref(op), out, 1, None) == E
    assert L.fp8_mx_gemm_fprop(128, 128, 256, ctypes.byref(op), ctypes.byref(op), None, 9, out, None, None) == E
    assert L.fp8_mx_gemm_dgrad(128, 128, 256, ctypes.byref(op), ctypes.byref(op), None, 4, out, None, None, 0,
                               None) == E



def test_bgrad_from_operand_validation(L):
    import fp8_linear_layer_gb300 as f
    E = f.binding.ERR_INVALID_ARG
    vp = ctypes.c_void_p
    q, s = 0x100000, 0x200000  # never dereferenced: validation fails first
    op = f.binding.OperandStruct(q, s, 256, 8, f.E4M3, 0)
    fn = L.fp8_bgrad_from_operand
    assert fn(8, 200, ctypes.byref(op), vp(0x300000), 0, None) == E  # K % 128
    assert fn(8, 256, ctypes.byref(op), vp(0x300002), 0, None) == E  # db misaligned
    assert fn(8, 256, ctypes.byref(op), None, 0, None) == E
    assert fn(9, 256, ctypes.byref(op), vp(0x300000), 0, None) == E  # scale_ld < rows
    assert fn(8, 256, ctypes.byref(op), vp(q + 7 * 256 + 200), 0, None) == E  # db inside the codes
    assert fn(8, 256, ctypes.byref(op), vp(s + 4 * 8 + 16), 0, None) == E  # db inside block 1's scales
    assert fn(8, 256, ctypes.byref(op), vp(q - 28), 0, None) == E  # db's last element on the first code
    assert fn(0, 256, ctypes.byref(op), None, 0, None) == f.binding.OK  # no rows: nothing to do
    assert fn(-1, 256, ctypes.byref(op), vp(0x300000), 0, None) == E


def test_quantize_dbias_validation(L):
    import fp8_linear_layer_gb300 as f
    E, WS = f.binding.ERR_INVALID_ARG, f.binding.ERR_WORKSPACE
    vp = ctypes.c_void_p
    x, q, s, db, ws = vp(0x100000), vp(0x200000), vp(0x300000), vp(0x400000), vp(0x500000)
    fn = L.fp8_quantize_dbias
    need = 2 * 64 * 4  # (256/128) x 64 floats
    assert fn(x, 200, 64, 64, 1, q, s, 64, None, None, 0, db, ws, need, None) == E  # rows % 128
    assert fn(x, 256, 60, 64, 1, q, s, 64, None, None, 0, db, ws, need, None) == E  # cols % 8
    assert fn(x, 256, 64, 64, 1, q, s, 60, None, None, 0, db, ws, need, None) == E  # scale_ld < cols
    assert fn(x, 256, 64, 64, 1, q, s, 64, q, s, 256, db, ws, need, None) == E  # row cast needs cols % 128
    assert fn(x, 256, 64, 64, 1, q, s, 64, None, None, 0, vp(0x400002), ws, need, None) == E  # db misaligned
    assert fn(x, 256, 64, 64, 1, q, s, 64, None, None, 0, db, ws, need - 4, None) == WS
    assert fn(x, 256, 64, 64, 1, q, s, 64, None, None, 0, db, None, need, None) == WS
    assert fn(x, 256, 64, 64, 1, q, s, 64, None, None, 0, vp(0x500000 + 64), ws, need, None) == E  # db in ws
    assert fn(x, 256, 0, 64, 1, q, s, 64, None, None, 0, db, ws, need, None) == f.binding.OK  # no columns
    assert fn(x, 256, 64, 64, 2, q, s, 64, None, None, 0, db, ws, need, None) == E  # format
    # the partials may not overlap what the cast reads (x) or writes (codes, scales)
    assert fn(x, 256, 64, 64, 1, q, s, 64, None, None, 0, db, vp(0x100000 + 256 * 128 - 16), need, None) == E
    assert fn(x, 256, 64, 64, 1, q, s, 64, None, None, 0, db, vp(0x200000 + 64 * 256 - 16), need, None) == E
    assert fn(x, 256, 64, 64, 1, q, s, 64, None, None, 0, db, vp(0x300000 - need + 16), need, None) == E
    q2, s2 = vp(0x600000), vp(0x700000)  # with the row cast: its codes and scales too
    assert fn(x, 256, 128, 128, 1, q, s, 128, q2, s2, 256, db, vp(0x600000 + 256 * 128 - 16), 2 * 128 * 4,
              None) == E
    assert fn(x, 256, 128, 128, 1, q, s, 128, q2, s2, 256, db, vp(0x700000 + 16), 2 * 128 * 4, None) == E


def test_binding_checks_every_status_with_its_call_name():
    # each _check(status, name) call passes exactly those two arguments
    import ast
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "fp8_linear_layer_gb300",
                        "binding.py")
    calls = [n for n in ast.walk(ast.parse(open(path).read()))
             if isinstance(n, ast.Call) and getattr(n.func, "id", "") == "_check"]
    assert len(calls) >= 20
    for c in calls:
        assert len(c.args) == 2 and isinstance(c.args[1], ast.Constant), c.lineno
        assert c.args[1].value.startswith("fp8_"), c.lineno


def test_mx_quantize_dbias_validation(L):
    import fp8_linear_layer_gb300 as f
    E, WS = f.binding.ERR_INVALID_ARG, f.binding.ERR_WORKSPACE
    vp = ctypes.c_void_p
    x, q, sf, db, ws = vp(0x100000), vp(0x200000), vp(0x300000), vp(0x400000), vp(0x500000)
    fn = L.fp8_mx_quantize_dbias
    need = 2 * 64 * 4
    assert fn(x, 200, 64, 64, 1, q, sf, db, ws, need, None) == E  # rows % 128
    assert fn(x, 256, 60, 64, 1, q, sf, db, ws, need, None) == E  # cols % 8
    assert fn(x, 256, 64, 56, 1, q, sf, db, ws, need, None) == E  # ldx < cols
    assert fn(x, 256, 64, 64, 1, q, sf, vp(0x400001), ws, need, None) == E
    assert fn(x, 256, 64, 64, 1, q, sf, db, ws, need - 4, None) == WS
    assert fn(x, 256, 64, 64, 1, q, sf, vp(0x500000 + 256), ws, need, None) == E  # db inside the partials
    assert fn(x, 256, 64, 64, 1, q, sf, db, vp(0x100000 + 256 * 128 - 16), need, None) == E  # ws over x's end
    assert fn(x, 256, 64, 64, 1, q, sf, db, vp(0x200000 + 64 * 256 - 16), need, None) == E  # ws over the codes
    assert fn(x, 256, 64, 64, 1, q, sf, db, vp(0x300000 + 16), need, None) == E  # ws over the scale bytes
    assert fn(x, 256, 0, 64, 1, q, sf, db, ws, need, None) == f.binding.OK
