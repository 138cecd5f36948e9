"""ctypes binding of libfp8ll.so (include/fp8ll.h): argument marshalling only.

Every computation happens in the CUDA library.  This module turns torch CUDA
tensors into device pointers, picks torch's current stream, allocates outputs
with torch when the caller does not pass them, and raises ``Fp8Error`` on a
non-zero status.  There is no fallback: if the library is missing or the
device is not supported, calls raise.
"""
import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence, Tuple

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp8ll.so")

E4M3, E5M2 = 0, 1
EPI_NONE, EPI_BIAS, EPI_BIAS_GELU, EPI_DGELU, EPI_DGELU_BGRAD = 0, 1, 2, 3, 4
ACC_FULL, ACC_FAST = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_DEVICE, ERR_LAUNCH, ERR_TIMEOUT, ERR_WORKSPACE, ERR_SCRATCH = 0, -1, -2, -3, -4, -5, -6

# every symbol include/fp8ll.h declares
EXPORTS = ("fp8_scale_ld", "fp8_quantize", "fp8_quantize_dual", "fp8_cast_f32", "fp8_gemm_fprop", "fp8_workspace_size",
           "fp8_gemm_dgrad", "fp8_gemm_dgrad_noalloc", "fp8_gemm_dgrad_quant", "fp8_gemm_wgrad", "fp8_grouped_wgrad", "fp8_get_device_status",
           "fp8_status_string", "fp8_debug_starve_next_gemm", "fp8_mx_sf_bytes", "fp8_mx_quantize",
           "fp8_mx_gemm_fprop", "fp8_mx_gemm_dgrad", "fp8_mx_gemm_wgrad", "fp8_tensor_amax", "fp8_tensor_quantize",
           "fp8_amax_history_update", "fp8_tensor_gemm_fprop", "fp8_tensor_gemm_dgrad", "fp8_tensor_gemm_wgrad",
           "fp8_bgrad_from_operand", "fp8_quantize_dbias", "fp8_mx_quantize_dbias")


class Fp8Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s failed: %s (%d)" % (what, status_string(code), code))


class OperandStruct(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("ld_q", ctypes.c_int64),
                ("scale_ld", ctypes.c_int64), ("fmt", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class MxOperandStruct(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("ld_q", ctypes.c_int64), ("fmt", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class TensorOperandStruct(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("ld_q", ctypes.c_int64),
                ("fmt", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libfp8ll.so is not built (run __graft_entry__.build() or "
                               "python fp8_linear_layer_gb300/build.py)")
        L = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        op = ctypes.POINTER(OperandStruct)
        L.fp8_scale_ld.argtypes = [i64]
        L.fp8_scale_ld.restype = i64
        L.fp8_quantize.argtypes = [vp, i64, i64, i64, i32, i32, vp, vp, i64, vp]
        L.fp8_quantize_dual.argtypes = [vp, i64, i64, i64, i32, vp, vp, i64, vp, vp, i64, vp]
        L.fp8_cast_f32.argtypes = [vp, i64, i32, vp, vp]
        L.fp8_gemm_fprop.argtypes = [i64, i64, i64, op, op, vp, i32, i32, vp, vp, vp]
        L.fp8_workspace_size.argtypes = [i64, i64]
        L.fp8_workspace_size.restype = sz
        L.fp8_gemm_dgrad.argtypes = [i64, i64, i64, op, op, vp, i32, i32, vp, vp, vp, sz, vp]
        L.fp8_gemm_dgrad_noalloc.argtypes = [i64, i64, i64, op, op, vp, i32, i32, vp, vp, vp]
        L.fp8_gemm_dgrad_quant.argtypes = [i64, i64, i64, op, op, vp, i32, vp, vp, vp, i64, vp]
        L.fp8_gemm_wgrad.argtypes = [i64, i64, i64, op, op, vp, i32, i32, vp]
        L.fp8_grouped_wgrad.argtypes = [i32, i64, i64, ctypes.POINTER(ctypes.c_int64), op, op, vp, i32, i32, vp]
        L.fp8_get_device_status.argtypes = [vp]
        L.fp8_status_string.argtypes = [i32]
        L.fp8_status_string.restype = ctypes.c_char_p
        L.fp8_debug_starve_next_gemm.argtypes = [i32]
        mop = ctypes.POINTER(MxOperandStruct)
        L.fp8_mx_sf_bytes.argtypes = [i64, i64]
        L.fp8_mx_sf_bytes.restype = sz
        L.fp8_mx_quantize.argtypes = [vp, i64, i64, i64, i32, i32, vp, vp, vp]
        L.fp8_mx_gemm_fprop.argtypes = [i64, i64, i64, mop, mop, vp, i32, vp, vp, vp]
        L.fp8_mx_gemm_dgrad.argtypes = [i64, i64, i64, mop, mop, vp, i32, vp, vp, vp, sz, vp]
        L.fp8_mx_gemm_wgrad.argtypes = [i64, i64, i64, mop, mop, vp, i32, vp]
        top = ctypes.POINTER(TensorOperandStruct)
        L.fp8_tensor_amax.argtypes = [vp, i64, i64, i64, vp, vp]
        L.fp8_tensor_quantize.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp]
        L.fp8_amax_history_update.argtypes = [vp, i64, i64, vp, vp, vp]
        L.fp8_tensor_gemm_fprop.argtypes = [i64, i64, i64, top, top, vp, i32, vp, vp, vp]
        L.fp8_tensor_gemm_dgrad.argtypes = [i64, i64, i64, top, top, vp, i32, vp, vp, vp, sz, vp]
        L.fp8_tensor_gemm_wgrad.argtypes = [i64, i64, i64, top, top, vp, i32, vp]
        L.fp8_bgrad_from_operand.argtypes = [i64, i64, op, vp, i32, vp]
        L.fp8_quantize_dbias.argtypes = [vp, i64, i64, i64, i32, vp, vp, i64, vp, vp, i64, vp, vp, sz, vp]
        L.fp8_mx_quantize_dbias.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, vp, sz, vp]
        for name in ("fp8_quantize", "fp8_quantize_dual", "fp8_cast_f32", "fp8_gemm_fprop", "fp8_gemm_dgrad",
                     "fp8_gemm_dgrad_noalloc", "fp8_gemm_dgrad_quant",
                     "fp8_gemm_wgrad", "fp8_mx_quantize", "fp8_mx_gemm_fprop", "fp8_mx_gemm_dgrad",
                     "fp8_mx_gemm_wgrad", "fp8_tensor_amax", "fp8_tensor_quantize", "fp8_amax_history_update",
                     "fp8_tensor_gemm_fprop", "fp8_tensor_gemm_dgrad", "fp8_tensor_gemm_wgrad",
                     "fp8_grouped_wgrad", "fp8_bgrad_from_operand", "fp8_quantize_dbias", "fp8_mx_quantize_dbias",
                     "fp8_get_device_status",
                     "fp8_debug_starve_next_gemm"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().fp8_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != OK:
        raise Fp8Error(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def scale_ld(rows: int) -> int:
    return int(lib().fp8_scale_ld(int(rows)))


@dataclass
class Fp8Tensor:
    """fp8 codes [rows][ld_q] (uint8) with block scales [K/128][scale_ld] (fp32)."""
    q: torch.Tensor
    scale: torch.Tensor
    fmt: int

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def k(self) -> int:
        return self.q.shape[1]

    def operand(self) -> OperandStruct:
        return OperandStruct(self.q.data_ptr(), self.scale.data_ptr(), self.q.stride(0),
                             self.scale.stride(0), int(self.fmt), 0)


def empty_fp8(rows: int, k: int, fmt: int, device="cuda") -> Fp8Tensor:
    q = torch.empty((rows, k), dtype=torch.uint8, device=device)
    s = torch.empty((k // 128, scale_ld(rows)), dtype=torch.float32, device=device)
    return Fp8Tensor(q, s, fmt)


def quantize(x: torch.Tensor, fmt: int, transpose: bool = False, out: Optional[Fp8Tensor] = None) -> Fp8Tensor:
    """bf16 [rows][cols] -> Fp8Tensor.  transpose=False: blocks along rows, codes
    [rows][cols]; transpose=True: blocks down columns, codes [cols][rows]."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if out is None:
        out = empty_fp8(cols, rows, fmt, x.device) if transpose else empty_fp8(rows, cols, fmt, x.device)
    _check(lib().fp8_quantize(_ptr(x), rows, cols, x.stride(0), int(fmt), int(bool(transpose)), _ptr(out.q),
                              _ptr(out.scale), out.scale.stride(0), _stream()), "fp8_quantize")
    return out


def quantize_dual(x: torch.Tensor, fmt: int, out: Optional[Fp8Tensor] = None,
                  out_t: Optional[Fp8Tensor] = None) -> Tuple[Fp8Tensor, Fp8Tensor]:
    """bf16 [rows][cols] -> (quantize(x, fmt), quantize(x, fmt, transpose=True))
    from one read of x; rows and cols multiples of 128."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if out is None:
        out = empty_fp8(rows, cols, fmt, x.device)
    if out_t is None:
        out_t = empty_fp8(cols, rows, fmt, x.device)
    _check(lib().fp8_quantize_dual(_ptr(x), rows, cols, x.stride(0), int(fmt), _ptr(out.q), _ptr(out.scale),
                                   out.scale.stride(0), _ptr(out_t.q), _ptr(out_t.scale), out_t.scale.stride(0),
                                   _stream()), "fp8_quantize_dual")
    return out, out_t


def cast_f32(x: torch.Tensor, fmt: int, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    assert x.dtype == torch.float32 and x.is_contiguous()
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(lib().fp8_cast_f32(_ptr(x), x.numel(), int(fmt), _ptr(out), _stream()), "fp8_cast_f32")
    return out


def gemm_fprop(A: Fp8Tensor, B: Fp8Tensor, bias: Optional[torch.Tensor] = None, epi: int = EPI_BIAS_GELU,
               acc: int = ACC_FULL, out: Optional[torch.Tensor] = None, aux: Optional[torch.Tensor] = None,
               want_aux: bool = True, K: Optional[int] = None):
    """Y (bf16 [M][N]) = epilogue(A B^T); returns (Y, Z-or-None)."""
    M, N = A.rows, B.rows
    K = A.k if K is None else K
    dev = A.q.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if aux is None and want_aux and epi == EPI_BIAS_GELU:
        aux = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_gemm_fprop(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(bias), int(epi), int(acc),
                                _ptr(out), _ptr(aux), _stream()), "fp8_gemm_fprop")
    return out, aux


def workspace_size(M: int, N: int) -> int:
    return int(lib().fp8_workspace_size(int(M), int(N)))


def gemm_dgrad(A: Fp8Tensor, B: Fp8Tensor, aux: torch.Tensor, epi: int = EPI_DGELU_BGRAD, acc: int = ACC_FULL,
               out: Optional[torch.Tensor] = None, bgrad: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, K: Optional[int] = None):
    """dZ (bf16 [M][N]) = (A B^T) * gelu'(aux); with DGELU_BGRAD also bgrad [N].
    Returns (dZ, bgrad-or-None)."""
    M, N = A.rows, B.rows
    K = A.k if K is None else K
    dev = A.q.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws_bytes = 0
    if epi == EPI_DGELU_BGRAD:
        if bgrad is None:
            bgrad = torch.empty((N,), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty((workspace_size(M, N) // 4,), dtype=torch.float32, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_gemm_dgrad(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(aux), int(epi), int(acc),
                                _ptr(out), _ptr(bgrad), _ptr(workspace), ws_bytes, _stream()), "fp8_gemm_dgrad")
    return out, bgrad


def gemm_dgrad_quant(A: Fp8Tensor, B: Fp8Tensor, aux: torch.Tensor, acc: int = ACC_FULL,
                     out: Optional[torch.Tensor] = None, q_out: Optional[Fp8Tensor] = None,
                     K: Optional[int] = None) -> Tuple[torch.Tensor, Fp8Tensor]:
    """dZ (bf16 [M][N]) = (A B^T) * gelu'(aux) and the e5m2 row cast of that
    dZ (exactly quantize(dZ, E5M2)) from the same epilogue; N % 128 == 0.
    Returns (dZ, Fp8Tensor of dZ)."""
    M, N = A.rows, B.rows
    K = A.k if K is None else K
    dev = A.q.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if q_out is None:
        q_out = empty_fp8(M, N, E5M2, dev)
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_gemm_dgrad_quant(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(aux), int(acc), _ptr(out),
                                      _ptr(q_out.q), _ptr(q_out.scale), q_out.scale.stride(0), _stream()),
           "fp8_gemm_dgrad_quant")
    return out, q_out


def gemm_wgrad(A: Fp8Tensor, B: Fp8Tensor, out: torch.Tensor, accumulate: bool = True, acc: int = ACC_FULL,
               K: Optional[int] = None) -> torch.Tensor:
    """fp32 out [M][N] (+)= A B^T (the weight-gradient accumulate)."""
    M, N = A.rows, B.rows
    K = A.k if K is None else K
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (M, N)
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_gemm_wgrad(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(out), int(bool(accumulate)),
                                int(acc), _stream()), "fp8_gemm_wgrad")
    return out


def grouped_wgrad(A: Fp8Tensor, B: Fp8Tensor, k_sizes: Sequence[int], out: torch.Tensor, accumulate: bool = True,
                  acc: int = ACC_FULL) -> torch.Tensor:
    """fp32 out [G][M][N]: out_g (+)= A[:, group g] B[:, group g]^T, groups contiguous along K."""
    G = len(k_sizes)
    M, N = A.rows, B.rows
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (G, M, N)
    ks = (ctypes.c_int64 * G)(*[int(k) for k in k_sizes])
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_grouped_wgrad(G, M, N, ks, ctypes.byref(oa), ctypes.byref(ob), _ptr(out),
                                   int(bool(accumulate)), int(acc), _stream()), "fp8_grouped_wgrad")
    return out


def bgrad_from_operand(A: Fp8Tensor, out: Optional[torch.Tensor] = None, accumulate: bool = False) -> torch.Tensor:
    """fp32 db [rows] (+)= the row sums of the dequantized operand A: the bias
    gradient reduced from the weight-gradient GEMM's gradient operand dZ^T."""
    if out is None:
        out = torch.empty(A.rows, dtype=torch.float32, device=A.q.device)
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (A.rows,)
    oa = A.operand()
    _check(lib().fp8_bgrad_from_operand(A.rows, A.k, ctypes.byref(oa), _ptr(out), int(bool(accumulate)), _stream()),
           "fp8_bgrad_from_operand")
    return out


def quantize_dbias(x: torch.Tensor, fmt: int, out_t: Optional[Fp8Tensor] = None, out: Optional[Fp8Tensor] = None,
                   rows: bool = False, dbias: Optional[torch.Tensor] = None,
                   workspace: Optional[torch.Tensor] = None) -> Tuple[Optional[Fp8Tensor], Fp8Tensor, torch.Tensor]:
    """bf16 gradient [rows][cols] -> (row cast or None, transposed cast, db):
    the transposed cast of quantize(x, fmt, transpose=True) (with rows=True
    or `out` given, also the row cast) and db [cols] fp32 = the column sums
    of x, from one read of x."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    if out_t is None:
        out_t = empty_fp8(C, R, fmt, x.device)
    if out is None and rows:
        out = empty_fp8(R, C, fmt, x.device)
    if dbias is None:
        dbias = torch.empty((C,), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty((max(R // 128, 1) * C,), dtype=torch.float32, device=x.device)
    assert dbias.dtype == torch.float32 and dbias.is_contiguous() and tuple(dbias.shape) == (C,)
    _check(lib().fp8_quantize_dbias(_ptr(x), R, C, x.stride(0), int(fmt), _ptr(out_t.q), _ptr(out_t.scale),
                                    out_t.scale.stride(0), _ptr(out.q) if out is not None else None,
                                    _ptr(out.scale) if out is not None else None,
                                    out.scale.stride(0) if out is not None else 0, _ptr(dbias), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream()), "fp8_quantize_dbias")
    return out, out_t, dbias


def device_status() -> int:
    """Synchronizes the current stream; returns and clears the device status word."""
    return int(lib().fp8_get_device_status(_stream()))


def debug_starve_next_gemm(budget_ms: int):
    _check(lib().fp8_debug_starve_next_gemm(int(budget_ms)), "fp8_debug_starve_next_gemm")


# ----------------------------------------------------------------- MXFP8 ----

@dataclass
class Fp8MxTensor:
    """MXFP8 codes [rows][ld_q] (uint8) with UE8M0 scale bytes in the layout the
    GEMM copies into tensor memory (see fp8ll.h)."""
    q: torch.Tensor
    sf: torch.Tensor
    fmt: int

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def k(self) -> int:
        return self.q.shape[1]

    def operand(self) -> MxOperandStruct:
        return MxOperandStruct(self.q.data_ptr(), self.sf.data_ptr(), self.q.stride(0), int(self.fmt), 0)


def mx_sf_bytes(rows: int, k: int) -> int:
    return int(lib().fp8_mx_sf_bytes(int(rows), int(k)))


def empty_mx(rows: int, k: int, fmt: int, device="cuda") -> Fp8MxTensor:
    q = torch.empty((rows, k), dtype=torch.uint8, device=device)
    sf = torch.empty((mx_sf_bytes(rows, k),), dtype=torch.uint8, device=device)
    return Fp8MxTensor(q, sf, fmt)


def mx_quantize(x: torch.Tensor, fmt: int, transpose: bool = False, out: Optional[Fp8MxTensor] = None) -> Fp8MxTensor:
    """bf16 [rows][cols] -> Fp8MxTensor (one power-of-two scale per 32 elements).
    transpose=False: blocks along rows, codes [rows][cols]; transpose=True:
    blocks down columns, codes [cols][rows]."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    if out is None:
        out = empty_mx(cols, rows, fmt, x.device) if transpose else empty_mx(rows, cols, fmt, x.device)
    _check(lib().fp8_mx_quantize(_ptr(x), rows, cols, x.stride(0), int(fmt), int(bool(transpose)), _ptr(out.q),
                                 _ptr(out.sf), _stream()), "fp8_mx_quantize")
    return out


def mx_quantize_dbias(x: torch.Tensor, fmt: int, out: Optional[Fp8MxTensor] = None,
                      dbias: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None) -> Tuple[Fp8MxTensor, torch.Tensor]:
    """bf16 gradient [rows][cols] -> (mx_quantize(x, fmt, transpose=True), db):
    db [cols] fp32 = the column sums of x, from the same read."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    R, C = x.shape
    if out is None:
        out = empty_mx(C, R, fmt, x.device)
    if dbias is None:
        dbias = torch.empty((C,), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty((max(R // 128, 1) * C,), dtype=torch.float32, device=x.device)
    assert dbias.dtype == torch.float32 and dbias.is_contiguous() and tuple(dbias.shape) == (C,)
    _check(lib().fp8_mx_quantize_dbias(_ptr(x), R, C, x.stride(0), int(fmt), _ptr(out.q), _ptr(out.sf), _ptr(dbias),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(), _stream()),
           "fp8_mx_quantize_dbias")
    return out, dbias


def mx_gemm_fprop(A: Fp8MxTensor, B: Fp8MxTensor, bias: Optional[torch.Tensor] = None, epi: int = EPI_BIAS_GELU,
                  out: Optional[torch.Tensor] = None, aux: Optional[torch.Tensor] = None, want_aux: bool = True):
    """Y (bf16 [M][N]) = epilogue(A B^T) with MX operands; returns (Y, Z-or-None)."""
    M, N, K = A.rows, B.rows, A.k
    dev = A.q.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if aux is None and want_aux and epi == EPI_BIAS_GELU:
        aux = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_mx_gemm_fprop(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(bias), int(epi), _ptr(out),
                                   _ptr(aux), _stream()), "fp8_mx_gemm_fprop")
    return out, aux


def mx_gemm_dgrad(A: Fp8MxTensor, B: Fp8MxTensor, aux: torch.Tensor, epi: int = EPI_DGELU_BGRAD,
                  out: Optional[torch.Tensor] = None, bgrad: Optional[torch.Tensor] = None,
                  workspace: Optional[torch.Tensor] = None):
    """dZ (bf16 [M][N]) = (A B^T) * gelu'(aux) with MX operands (+ bias gradient [N])."""
    M, N, K = A.rows, B.rows, A.k
    dev = A.q.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws_bytes = 0
    if epi == EPI_DGELU_BGRAD:
        if bgrad is None:
            bgrad = torch.empty((N,), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty((workspace_size(M, N) // 4,), dtype=torch.float32, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_mx_gemm_dgrad(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(aux), int(epi), _ptr(out),
                                   _ptr(bgrad), _ptr(workspace), ws_bytes, _stream()), "fp8_mx_gemm_dgrad")
    return out, bgrad


def mx_gemm_wgrad(A: Fp8MxTensor, B: Fp8MxTensor, out: torch.Tensor, accumulate: bool = True) -> torch.Tensor:
    """fp32 out [M][N] (+)= A B^T with MX operands."""
    M, N, K = A.rows, B.rows, A.k
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (M, N)
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_mx_gemm_wgrad(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(out), int(bool(accumulate)),
                                   _stream()), "fp8_mx_gemm_wgrad")
    return out


# ------------------------------------------------------ per-tensor scaling ----

@dataclass
class Fp8TensorScaled:
    """fp8 codes [rows][ld_q] (uint8) with the tensor's one fp32 scale (a
    1-element device tensor)."""
    q: torch.Tensor
    scale: torch.Tensor
    fmt: int

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def k(self) -> int:
        return self.q.shape[1]

    def operand(self) -> TensorOperandStruct:
        return TensorOperandStruct(self.q.data_ptr(), self.scale.data_ptr(), self.q.stride(0), int(self.fmt), 0)


def empty_tensor_scaled(rows: int, k: int, fmt: int, device="cuda") -> Fp8TensorScaled:
    return Fp8TensorScaled(torch.empty((rows, k), dtype=torch.uint8, device=device),
                           torch.empty((1,), dtype=torch.float32, device=device), fmt)


def tensor_amax(x: torch.Tensor, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """max|x| of a bf16 matrix into a 1-element fp32 device tensor."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    if out is None:
        out = torch.empty((1,), dtype=torch.float32, device=x.device)
    _check(lib().fp8_tensor_amax(_ptr(x), x.shape[0], x.shape[1], x.stride(0), _ptr(out), _stream()),
           "fp8_tensor_amax")
    return out


def tensor_quantize(x: torch.Tensor, fmt: int, amax_in: torch.Tensor, rows: bool = True, cols: bool = False,
                    amax_out: Optional[torch.Tensor] = None, out: Optional[Fp8TensorScaled] = None,
                    out_t: Optional[Fp8TensorScaled] = None):
    """Per-tensor cast of bf16 x [r][c] with the amax in amax_in (1-element
    device tensor).  rows: codes [r][c]; cols: transposed codes [c][r]; both
    share the one scale.  Returns (rows operand or None, cols operand or None)."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1 and (rows or cols)
    r, c = x.shape
    scale = out.scale if out is not None else (out_t.scale if out_t is not None else None)
    if scale is None:
        scale = torch.empty((1,), dtype=torch.float32, device=x.device)
    if rows and out is None:
        out = Fp8TensorScaled(torch.empty((r, c), dtype=torch.uint8, device=x.device), scale, fmt)
    if cols and out_t is None:
        out_t = Fp8TensorScaled(torch.empty((c, r), dtype=torch.uint8, device=x.device), scale, fmt)
    if rows and cols:
        assert out.scale.data_ptr() == out_t.scale.data_ptr(), "both orientations share one scale"
    _check(lib().fp8_tensor_quantize(_ptr(x), r, c, x.stride(0), int(fmt), _ptr(amax_in),
                                     _ptr(out.q) if rows else None, _ptr(out_t.q) if cols else None, _ptr(scale),
                                     _ptr(amax_out), _stream()), "fp8_tensor_quantize")
    return (out if rows else None), (out_t if cols else None)


def amax_history_update(history: torch.Tensor, amax_new: torch.Tensor, amax_use: torch.Tensor) -> torch.Tensor:
    """Delayed scaling: push amax_new into history and write the largest entry
    to amax_use (fp32 device tensors).  history [len] for one tensor, or
    [count][len] with amax_new and amax_use holding count values."""
    assert history.dtype == torch.float32 and history.is_contiguous()
    count = 1 if history.dim() == 1 else history.shape[0]
    assert amax_new.numel() == count and amax_use.numel() == count
    assert amax_new.is_contiguous() and amax_use.is_contiguous()
    _check(lib().fp8_amax_history_update(_ptr(history), count, history.shape[-1], _ptr(amax_new), _ptr(amax_use),
                                         _stream()), "fp8_amax_history_update")
    return amax_use


def tensor_gemm_fprop(A: Fp8TensorScaled, B: Fp8TensorScaled, bias: Optional[torch.Tensor] = None,
                      epi: int = EPI_BIAS_GELU, out: Optional[torch.Tensor] = None,
                      aux: Optional[torch.Tensor] = None, want_aux: bool = True):
    """Y (bf16 [M][N]) = epilogue(sA sB A B^T); returns (Y, Z-or-None)."""
    M, N, K = A.rows, B.rows, A.k
    dev = A.q.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    if aux is None and want_aux and epi == EPI_BIAS_GELU:
        aux = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_tensor_gemm_fprop(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(bias), int(epi),
                                       _ptr(out), _ptr(aux), _stream()), "fp8_tensor_gemm_fprop")
    return out, aux


def tensor_gemm_dgrad(A: Fp8TensorScaled, B: Fp8TensorScaled, aux: torch.Tensor, epi: int = EPI_DGELU_BGRAD,
                      out: Optional[torch.Tensor] = None, bgrad: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None):
    """dZ (bf16 [M][N]) = (sA sB A B^T) * gelu'(aux) (+ bias gradient [N])."""
    M, N, K = A.rows, B.rows, A.k
    dev = A.q.device
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws_bytes = 0
    if epi == EPI_DGELU_BGRAD:
        if bgrad is None:
            bgrad = torch.empty((N,), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty((workspace_size(M, N) // 4,), dtype=torch.float32, device=dev)
        ws_bytes = workspace.numel() * workspace.element_size()
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_tensor_gemm_dgrad(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(aux), int(epi), _ptr(out),
                                       _ptr(bgrad), _ptr(workspace), ws_bytes, _stream()), "fp8_tensor_gemm_dgrad")
    return out, bgrad


def tensor_gemm_wgrad(A: Fp8TensorScaled, B: Fp8TensorScaled, out: torch.Tensor,
                      accumulate: bool = True) -> torch.Tensor:
    """fp32 out [M][N] (+)= sA sB A B^T."""
    M, N, K = A.rows, B.rows, A.k
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (M, N)
    oa, ob = A.operand(), B.operand()
    _check(lib().fp8_tensor_gemm_wgrad(M, N, K, ctypes.byref(oa), ctypes.byref(ob), _ptr(out),
                                       int(bool(accumulate)), _stream()), "fp8_tensor_gemm_wgrad")
    return out
