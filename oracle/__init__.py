"""Plain CPU oracle for the block-scaled FP8 linear-layer GEMMs.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  It shares no code with
the CUDA library and never calls it.  The arithmetic lives in ``oracle.c``
(binary64, plain loops); this module only marshals numpy arrays.

Sources, by page title:
  * "Replaced cublasLt calls with rocblas gemm + 6 manually crafted epilogues":
    the linear layer Y = X W^T + b, its backward (dX, dW, db = column sum of
    the output gradient), bias length per epilogue (BIAS: output features;
    BGRADB: the GEMM's n), reductions in fp32, GELU derivative before the bias
    gradient.
  * "Weight gradient kernels for dense and MoE models": fp8 x fp8 -> fp32 "nt"
    weight-gradient GEMM that ACCUMULATES (out += a b^T), its k-grouped MoE
    variant, the per-token 1x128 cast of both operands.
  * "FP8 GEMM for the fprop should use fast accumulation": e4m3 forward,
    e4m3 x e5m2 backward, fast vs full accumulation as an explicit flag,
    per-tensor scales (with which fast accumulation needs no promotion).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, brute force over exact rationals, the worked example on the
DeepGEMM page, finite differences, torch's float8 casts).  The FAST
accumulation mode has no separate oracle: the oracle value is the same and
only the error bound differs (8e-3 instead of 2e-3 of sum|a b|).
"""
import ctypes
import os

import numpy as np

from . import build as _build

E4M3 = 0
E5M2 = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB points the pin tests at a deliberately broken copy of the
        # oracle (tests/test_oracle_mutants.py); normally unset.
        path = os.environ.get("ORACLE_LIB") or _build.build()
        lib = ctypes.CDLL(path)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_fp8_decode_table.argtypes = [i32, vp]
        lib.oracle_fp8_max.argtypes = [i32]
        lib.oracle_fp8_max.restype = ctypes.c_double
        lib.oracle_fp8_encode.argtypes = [i32, ctypes.c_float]
        lib.oracle_fp8_encode.restype = ctypes.c_uint8
        lib.oracle_fp8_encode_array.argtypes = [i32, vp, i64, vp]
        lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f32.restype = ctypes.c_float
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_f64_to_bf16_array.argtypes = [vp, i64, vp]
        lib.oracle_quantize.argtypes = [i32, vp, i64, i64, i64, i32, vp, vp, i64]
        lib.oracle_gemm.argtypes = [i64, i64, vp, i64, vp, i64, i32, vp, i64, vp, i64, i32,
                                    vp, i64, vp, i64, vp, vp]
        lib.oracle_mx_quantize.argtypes = [i32, vp, i64, i64, i64, i32, vp, vp, i64]
        lib.oracle_mx_gemm.argtypes = [i64, vp, i64, vp, i64, i32, vp, i64, vp, i64, i32, vp, i64, vp, i64, vp, vp]
        f32 = ctypes.c_float
        lib.oracle_tensor_quantize.argtypes = [i32, vp, i64, i64, i64, i32, f32, vp, vp, vp]
        lib.oracle_amax_history.argtypes = [vp, i64, f32, vp]
        lib.oracle_tensor_gemm.argtypes = [i64, i64, i64, vp, i64, f32, i32, vp, i64, f32, i32, vp, vp]
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu.restype = ctypes.c_double
        lib.oracle_dgelu.argtypes = [ctypes.c_double]
        lib.oracle_dgelu.restype = ctypes.c_double
        lib.oracle_gelu_array.argtypes = [vp, vp, i64]
        lib.oracle_dgelu_array.argtypes = [vp, vp, i64]
        lib.oracle_colsum.argtypes = [vp, i64, i64, vp]
        lib.oracle_operand_rowsum.argtypes = [i32, vp, i64, vp, i64, i64, i64, vp, vp]
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------- codec ----

def decode_table(fmt: int) -> np.ndarray:
    """256 float64 values of the fp8 codes, built from the bit fields."""
    out = np.empty(256, dtype=np.float64)
    _load().oracle_fp8_decode_table(int(fmt), _p(out))
    return out


def fp8_max(fmt: int) -> float:
    return float(_load().oracle_fp8_max(int(fmt)))


def encode(fmt: int, x) -> np.ndarray:
    """Round-to-nearest-even, saturating encode of float32 values."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    q = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_fp8_encode_array(int(fmt), _p(x), x.size, _p(q))
    return q


def decode(fmt: int, q) -> np.ndarray:
    return decode_table(fmt)[np.asarray(q, dtype=np.uint8)]


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) to float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f64_to_bf16(v: float) -> int:
    return int(_load().oracle_f64_to_bf16(float(v)))


def f64_to_bf16_array(v) -> np.ndarray:
    """Round float64 values to bf16 (nearest even); returns uint16 bit patterns."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    out = np.empty(v.shape, dtype=np.uint16)
    _load().oracle_f64_to_bf16_array(_p(v), v.size, _p(out))
    return out


# ------------------------------------------------------------- quantize ----

def quantize(x_bits, fmt: int, transpose: bool = False):
    """Per-128-block cast of a bf16 matrix (bit patterns, [rows][cols]).

    transpose=False: blocks along each row; returns q [rows][cols] (uint8) and
      scale [cols/128][rows] (float32).
    transpose=True: blocks down each column; returns q [cols][rows] and
      scale [rows/128][cols].
    """
    x = np.ascontiguousarray(np.asarray(x_bits, dtype=np.uint16))
    rows, cols = x.shape
    if not transpose:
        assert cols % 128 == 0
        q = np.empty((rows, cols), dtype=np.uint8)
        sc = np.empty((cols // 128, rows), dtype=np.float32)
        _load().oracle_quantize(int(fmt), _p(x), rows, cols, cols, 0, _p(q), _p(sc), rows)
    else:
        assert rows % 128 == 0
        q = np.empty((cols, rows), dtype=np.uint8)
        sc = np.empty((rows // 128, cols), dtype=np.float32)
        _load().oracle_quantize(int(fmt), _p(x), rows, cols, cols, 1, _p(q), _p(sc), cols)
    return q, sc


# ------------------------------------------------------------------ GEMM ----

def gemm(qa, sa, fmt_a, qb, sb, fmt_b, K=None, k0=0, rows=None, cols=None, want_abs=True):
    """Block-scaled "nt" GEMM in float64.

    qa [M][lda] uint8 with scales sa [blocks][M]; qb [N][ldb] with sb [blocks][N].
    Uses K columns starting at k0 (both multiples of 128).  rows / cols select
    output rows / columns (default all).  Returns (acc, S) with
    S = sum_k |a_ik b_jk| of the dequantized operands.
    """
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    M, lda = qa.shape
    N, ldb = qb.shape
    if K is None:
        K = lda - k0
    assert K % 128 == 0 and k0 % 128 == 0 and k0 + K <= lda and k0 + K <= ldb
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    acc = np.empty((nr, nc), dtype=np.float64)
    S = np.empty((nr, nc), dtype=np.float64) if want_abs else None
    _load().oracle_gemm(K, k0, _p(qa), lda, _p(sa), sa.shape[1], int(fmt_a),
                        _p(qb), ldb, _p(sb), sb.shape[1], int(fmt_b),
                        None if r is None else _p(r), nr, None if c is None else _p(c), nc,
                        _p(acc), None if S is None else _p(S))
    return acc, S


# ----------------------------------------------------------------- MXFP8 ----

def mx_quantize(x_bits, fmt: int, transpose: bool = False):
    """MXFP8 cast of a bf16 matrix (bit patterns, [rows][cols]): one power-of-two
    scale 2^e per 32 elements, e the smallest integer in [-127, 127] with
    amax <= FMAX 2^e (0 for an all-zero block), codes enc(x 2^-e).

    transpose=False: blocks along each row; returns q [rows][cols] (uint8) and
      e [cols/32][rows] (int8).
    transpose=True: blocks down each column; returns q [cols][rows] and
      e [rows/32][cols].
    """
    x = np.ascontiguousarray(np.asarray(x_bits, dtype=np.uint16))
    rows, cols = x.shape
    if not transpose:
        assert cols % 32 == 0
        q = np.empty((rows, cols), dtype=np.uint8)
        e = np.empty((cols // 32, rows), dtype=np.int8)
        _load().oracle_mx_quantize(int(fmt), _p(x), rows, cols, cols, 0, _p(q), _p(e), rows)
    else:
        assert rows % 32 == 0
        q = np.empty((cols, rows), dtype=np.uint8)
        e = np.empty((rows // 32, cols), dtype=np.int8)
        _load().oracle_mx_quantize(int(fmt), _p(x), rows, cols, cols, 1, _p(q), _p(e), cols)
    return q, e


def mx_gemm(qa, ea, fmt_a, qb, eb, fmt_b, rows=None, cols=None, want_abs=True):
    """MXFP8 "nt" GEMM in float64: acc[i][j] = sum_k dec(qa[i,k]) 2^ea[k/32,i] *
    dec(qb[j,k]) 2^eb[k/32,j]; returns (acc, S) with S the sum of |products|."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    ea = np.ascontiguousarray(ea, dtype=np.int8)
    eb = np.ascontiguousarray(eb, dtype=np.int8)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2 and K % 32 == 0 and ea.shape[0] == K // 32 and eb.shape[0] == K // 32
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else r.size
    nc = N if c is None else c.size
    acc = np.empty((nr, nc), dtype=np.float64)
    S = np.empty((nr, nc), dtype=np.float64) if want_abs else None
    _load().oracle_mx_gemm(K, _p(qa), K, _p(ea), ea.shape[1], int(fmt_a), _p(qb), K, _p(eb), eb.shape[1],
                           int(fmt_b), None if r is None else _p(r), nr, None if c is None else _p(c), nc,
                           _p(acc), None if S is None else _p(S))
    return acc, S


# ------------------------------------------------------ per-tensor scaling ----

def tensor_quantize(x_bits, fmt: int, amax_in: float, transpose: bool = False):
    """Per-tensor cast of a bf16 matrix (bit patterns, [rows][cols]) with one
    scale from the given amax: inv = fl32(FMAX/amax), scale = fl32(amax/FMAX),
    q = enc(fl32(x inv)), saturating above amax.  Returns (q, scale, amax of
    x); q is [rows][cols], or [cols][rows] with transpose=True."""
    x = np.ascontiguousarray(np.asarray(x_bits, dtype=np.uint16))
    rows, cols = x.shape
    q = np.empty((cols, rows) if transpose else (rows, cols), dtype=np.uint8)
    sc = np.empty(1, dtype=np.float32)
    am = np.empty(1, dtype=np.float32)
    _load().oracle_tensor_quantize(int(fmt), _p(x), rows, cols, cols, int(bool(transpose)),
                                   float(np.float32(amax_in)), _p(q), _p(sc), _p(am))
    return q, sc[0], am[0]


def amax_history(hist, amax_new: float):
    """Delayed scaling: push amax_new to the front of the history (the oldest
    entry drops out); returns (updated history, largest entry)."""
    h = np.array(hist, dtype=np.float32, copy=True)
    use = np.empty(1, dtype=np.float32)
    _load().oracle_amax_history(_p(h), h.size, float(np.float32(amax_new)), _p(use))
    return h, use[0]


def tensor_gemm(qa, sa: float, fmt_a, qb, sb: float, fmt_b, want_abs=True):
    """Per-tensor scaled "nt" GEMM in float64: acc[i][j] = sa sb sum_k
    dec(qa[i,k]) dec(qb[j,k]); returns (acc, S), S the same sum of |products|."""
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    M, K = qa.shape
    N, K2 = qb.shape
    assert K == K2
    acc = np.empty((M, N), dtype=np.float64)
    S = np.empty((M, N), dtype=np.float64) if want_abs else None
    _load().oracle_tensor_gemm(M, N, K, _p(qa), K, float(np.float32(sa)), int(fmt_a), _p(qb), K,
                               float(np.float32(sb)), int(fmt_b), _p(acc), None if S is None else _p(S))
    return acc, S


# ------------------------------------------------------------- epilogues ----

def gelu(z) -> np.ndarray:
    z = np.ascontiguousarray(np.asarray(z, dtype=np.float64))
    y = np.empty_like(z)
    _load().oracle_gelu_array(_p(z), _p(y), z.size)
    return y


def dgelu(z) -> np.ndarray:
    z = np.ascontiguousarray(np.asarray(z, dtype=np.float64))
    y = np.empty_like(z)
    _load().oracle_dgelu_array(_p(z), _p(y), z.size)
    return y


def colsum(dz) -> np.ndarray:
    dz = np.ascontiguousarray(np.asarray(dz, dtype=np.float64))
    M, N = dz.shape
    out = np.empty(N, dtype=np.float64)
    _load().oracle_colsum(_p(dz), M, N, _p(out))
    return out


def operand_rowsum(q, scale, fmt: int, want_abs=True):
    """Bias gradient reduced from the weight-gradient GEMM's fp8 operand
    (BGRADB on "Replaced cublasLt calls with rocblas gemm + 6 manually crafted
    epilogues": db computed with dW by reducing its gradient operand):
    out[r] = sum_k scale[k // 128, r] * dec(q[r, k]), binary64.  `q` is
    [rows][K] codes, `scale` [K/128][>= rows] fp32.  Returns (out, S) with S
    the magnitude sums (None unless want_abs)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    rows, K = q.shape
    assert K % 128 == 0 and scale.shape[0] == K // 128 and scale.shape[1] >= rows
    out = np.empty(rows, dtype=np.float64)
    S = np.empty(rows, dtype=np.float64) if want_abs else None
    _load().oracle_operand_rowsum(fmt, _p(q), K, _p(scale), scale.shape[1], rows, K, _p(out),
                                  _p(S) if want_abs else None)
    return out, S


def fprop_epilogue(acc, bias_bits=None, cols=None, gelu_on=True):
    """Z = acc + bias[j] (bias length N, the output features), Y = gelu(Z).

    bias_bits: bf16 bit patterns of length N (or None).  cols: which output
    columns acc holds (default all).  Returns (Z, Y) in float64; Y is Z when
    gelu_on is False."""
    acc = np.asarray(acc, dtype=np.float64)
    Z = acc.copy()
    if bias_bits is not None:
        b = bf16_to_f64(bias_bits).reshape(-1)
        if cols is not None:
            b = b[np.asarray(cols)]
        if b.shape[0] != acc.shape[1]:
            raise ValueError("bias must have one entry per output feature (column)")
        Z = Z + b[None, :]
    Y = gelu(Z) if gelu_on else Z
    return Z, Y


def dgrad_epilogue(acc, zaux_bits):
    """dZ = acc * gelu'(Z) with Z the stored bf16 pre-activation."""
    z = bf16_to_f64(zaux_bits)
    return np.asarray(acc, dtype=np.float64) * dgelu(z)


def wgrad(acc, prefill=None):
    """out = prefill + acc (the page's out += a b^T); prefill None means out = acc."""
    acc = np.asarray(acc, dtype=np.float64)
    if prefill is None:
        return acc
    return np.asarray(prefill, dtype=np.float64) + acc


def grouped_wgrad(qa, sa, fmt_a, qb, sb, fmt_b, k_sizes, prefill=None, rows=None, cols=None):
    """k-grouped weight gradient: for group g, out_g (+)= A[:, off_g:off_g+K_g] B[:, same]^T.

    qa [M][sumK], qb [N][sumK]; scales [sumK/128][M|N]; k_sizes: G ints, each
    a multiple of 128 (zero allowed).  prefill: [G][rows][cols] or None.
    Returns (out [G][nr][nc], S [G][nr][nc]).
    """
    outs, Ss = [], []
    off = 0
    for g, kg in enumerate(k_sizes):
        kg = int(kg)
        acc, S = gemm(qa, sa, fmt_a, qb, sb, fmt_b, K=kg, k0=off, rows=rows, cols=cols)
        pre = None if prefill is None else prefill[g]
        outs.append(wgrad(acc, pre))
        Ss.append(S)
        off += kg
    return np.stack(outs), np.stack(Ss)
