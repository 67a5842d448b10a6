"""Plain CPU oracle for the quantized GEMV/GEMM path (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package never imports the product: the two share no code.

The arithmetic lives in ``wq_oracle.c`` (plain C, single-threaded, fp64 /
int64 accumulation); this module only builds it with gcc and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "wq_oracle.c")
_HDR = os.path.join(_HERE, "wq_oracle.h")
_LIB = os.path.join(_HERE, "libwq_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libwq_oracle.so`` (gcc, -O2, no fast-math,
    no FP contraction so x86 and Arm give identical results)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every call of this module through another build of the oracle
    (used by the mutation test, which builds copies with a planted mistake)."""
    global _lib
    saved = _load()
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def _bind(lib):
    """Declare the C signatures on a loaded oracle library."""
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.wqo_f16_to_double.restype = ctypes.c_double
    lib.wqo_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.wqo_bf16_to_double.restype = ctypes.c_double
    lib.wqo_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.wqo_double_to_f16.restype = ctypes.c_uint16
    lib.wqo_double_to_f16.argtypes = [ctypes.c_double]
    lib.wqo_double_to_bf16.restype = ctypes.c_uint16
    lib.wqo_double_to_bf16.argtypes = [ctypes.c_double]
    lib.wqo_double_to_f32.restype = ctypes.c_float
    lib.wqo_double_to_f32.argtypes = [ctypes.c_double]
    for name in ("wqo_code3", "wqo_code4", "wqo_zero4"):
        getattr(lib, name).restype = I
        getattr(lib, name).argtypes = [P, I, I, I]
    for name in ("wqo_unpack3", "wqo_unpack4", "wqo_unpack_zeros4"):
        getattr(lib, name).restype = None
        getattr(lib, name).argtypes = [P, I, I, P]
    lib.wqo_wq8_gemv.restype = None
    lib.wqo_wq8_gemv.argtypes = [P, P, P, I, I, I, I, P, I, P, P]
    lib.wqo_wq3_gemv.restype = None
    lib.wqo_wq3_gemv.argtypes = [P, P, P, P, I, I, I, P, I, P, P]
    lib.wqo_wq4_gemm.restype = None
    lib.wqo_wq4_gemm.argtypes = [P, I, P, P, P, P, I, I, I, I, P, I, P, P]
    lib.wqo_wq8_dequant.restype = None
    lib.wqo_wq8_dequant.argtypes = [P, P, I, I, I, P]
    lib.wqo_wq3_dequant.restype = None
    lib.wqo_wq3_dequant.argtypes = [P, P, P, I, I, P]
    lib.wqo_wq4_dequant.restype = None
    lib.wqo_wq4_dequant.argtypes = [I, P, P, P, P, I, I, I, P]
    lib.wqo_w8a8_quant_rows.restype = None
    lib.wqo_w8a8_quant_rows.argtypes = [P, I, I, P, P]
    lib.wqo_w8a8_quant_rows_smooth.restype = None
    lib.wqo_w8a8_quant_rows_smooth.argtypes = [P, P, I, I, P, P]
    lib.wqo_w8a8_outlier_columns.restype = None
    lib.wqo_w8a8_outlier_columns.argtypes = [P, I, I, ctypes.c_float, P]
    lib.wqo_w8a8_outlier_rows.restype = I
    lib.wqo_w8a8_outlier_rows.argtypes = [P, P, P, P, P, P, I, I, I, P, I, P, P, P]
    lib.wqo_w8a8_gemm_rows.restype = I
    lib.wqo_w8a8_gemm_rows.argtypes = [P, P, P, P, I, I, I, P, I, P, P, P]
    return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    """Contiguous array of exactly `dtype` (no silent conversion of values)."""
    a = np.asarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _cols(cols, N):
    if cols is None:
        return None, N
    c = np.ascontiguousarray(np.asarray(cols, dtype=np.int32))
    if c.size and (c.min() < 0 or c.max() >= N):
        raise ValueError("column index out of range")
    return c, int(c.size)


# ---- scalar formats ---------------------------------------------------------

def f16_to_double(bits: int) -> float:
    return _load().wqo_f16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return _load().wqo_bf16_to_double(int(bits))


def double_to_f16(v: float) -> int:
    return int(_load().wqo_double_to_f16(float(v)))


def double_to_bf16(v: float) -> int:
    return int(_load().wqo_double_to_bf16(float(v)))


def round_f16(y: np.ndarray) -> np.ndarray:
    """Round an array of doubles to fp16 bit patterns (uint16), RNE."""
    lib = _load()
    flat = np.asarray(y, dtype=np.float64).ravel()
    out = np.fromiter((lib.wqo_double_to_f16(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(y))


def round_f32(y: np.ndarray) -> np.ndarray:
    """Round an array of doubles to fp32 (RNE, the C conversion)."""
    lib = _load()
    flat = np.asarray(y, dtype=np.float64).ravel()
    out = np.fromiter((lib.wqo_double_to_f32(float(v)) for v in flat), dtype=np.float32, count=flat.size)
    return out.reshape(np.shape(y))


def round_bf16(y: np.ndarray) -> np.ndarray:
    """Round an array of doubles to bf16 bit patterns (uint16), RNE."""
    lib = _load()
    flat = np.asarray(y, dtype=np.float64).ravel()
    out = np.fromiter((lib.wqo_double_to_bf16(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(y))


def decode_f16(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.fromiter((lib.wqo_f16_to_double(int(b)) for b in flat), dtype=np.float64,
                       count=flat.size).reshape(np.shape(bits))


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(bits, dtype=np.uint16).ravel()
    return np.fromiter((lib.wqo_bf16_to_double(int(b)) for b in flat), dtype=np.float64,
                       count=flat.size).reshape(np.shape(bits))


# ---- unpackers ----------------------------------------------------------------

def unpack3(mat: np.ndarray, K: int, N: int) -> np.ndarray:
    mat = _c(mat, np.int32)
    assert mat.shape == (3 * K // 32, N)
    out = np.empty((K, N), dtype=np.uint8)
    _load().wqo_unpack3(_ptr(mat), K, N, _ptr(out))
    return out


def unpack4(qweight: np.ndarray, K: int, N: int) -> np.ndarray:
    qweight = _c(qweight, np.int32)
    assert qweight.shape == (K // 8, N)
    out = np.empty((K, N), dtype=np.uint8)
    _load().wqo_unpack4(_ptr(qweight), K, N, _ptr(out))
    return out


def unpack_zeros4(qzeros: np.ndarray, G: int, N: int) -> np.ndarray:
    qzeros = _c(qzeros, np.int32)
    assert qzeros.shape == (G, N // 8)
    out = np.empty((G, N), dtype=np.uint8)
    _load().wqo_unpack_zeros4(_ptr(qzeros), G, N, _ptr(out))
    return out


# ---- products -------------------------------------------------------------------

def wq8_gemv(x, w, scales, group, cols=None):
    """y, abs_sum (float64 [M, ncols]) of y = x . (scales * q), int8 group-wise."""
    x = _c(x, np.float32); w = _c(w, np.int8); scales = _c(scales, np.float32)
    M, K = x.shape
    K2, N = w.shape
    assert K2 == K and scales.shape == (K // group, N) and K % group == 0
    c, nc = _cols(cols, N)
    y = np.empty((M, nc)); a = np.empty((M, nc))
    _load().wqo_wq8_gemv(_ptr(x), _ptr(w), _ptr(scales), M, K, N, group, _ptr(c), nc, _ptr(y), _ptr(a))
    return y, a


def wq3_gemv(x_bits, mat, scales_bits, zeros_bits, cols=None):
    """3-bit per-column GEMV; x, scales, zeros are fp16 bit patterns (uint16)."""
    x = _c(x_bits, np.uint16); mat = _c(mat, np.int32)
    scales = _c(scales_bits, np.uint16); zeros = _c(zeros_bits, np.uint16)
    M, K = x.shape
    R, N = mat.shape
    assert K % 32 == 0 and R == 3 * K // 32 and scales.shape == (N,) and zeros.shape == (N,)
    c, nc = _cols(cols, N)
    y = np.empty((M, nc)); a = np.empty((M, nc))
    _load().wqo_wq3_gemv(_ptr(x), _ptr(mat), _ptr(scales), _ptr(zeros), M, K, N, _ptr(c), nc, _ptr(y), _ptr(a))
    return y, a


def wq4_gemm(x_bits, act_bf16, qweight, scales_bits, qzeros, g_idx, group, cols=None):
    """4-bit group-wise GEMM; x and scales are fp16 (act_bf16=0) or bf16 bit patterns."""
    x = _c(x_bits, np.uint16); qweight = _c(qweight, np.int32); scales = _c(scales_bits, np.uint16)
    M, K = x.shape
    R, N = qweight.shape
    assert K % 8 == 0 and R == K // 8 and K % group == 0 and N % 8 == 0
    G = K // group
    assert scales.shape == (G, N)
    qz = None if qzeros is None else _c(qzeros, np.int32)
    if qz is not None:
        assert qz.shape == (G, N // 8)
    gi = None if g_idx is None else _c(g_idx, np.int32)
    if gi is not None:
        assert gi.shape == (K,) and gi.min() >= 0 and gi.max() < G
    c, nc = _cols(cols, N)
    y = np.empty((M, nc)); a = np.empty((M, nc))
    _load().wqo_wq4_gemm(_ptr(x), int(bool(act_bf16)), _ptr(qweight), _ptr(scales), _ptr(qz), _ptr(gi),
                         M, K, N, group, _ptr(c), nc, _ptr(y), _ptr(a))
    return y, a


# ---- dequantization (dense weights, the unfused baseline) -------------------

def wq8_dequant(w, scales, group):
    """Exact w(k,n) = scales[k/group, n] * q[k,n] as float64 [K, N]."""
    w = _c(w, np.int8); scales = _c(scales, np.float32)
    K, N = w.shape
    assert K % group == 0 and scales.shape == (K // group, N)
    out = np.empty((K, N))
    _load().wqo_wq8_dequant(_ptr(w), _ptr(scales), K, N, group, _ptr(out))
    return out


def wq3_dequant(mat, scales_bits, zeros_bits, K):
    """Exact w(k,n) = s[n] * q(k,n) - zero[n] (fp16 scale and stored zero) as float64 [K, N]."""
    mat = _c(mat, np.int32); scales = _c(scales_bits, np.uint16); zeros = _c(zeros_bits, np.uint16)
    R, N = mat.shape
    assert K % 32 == 0 and R == 3 * K // 32 and scales.shape == (N,) and zeros.shape == (N,)
    out = np.empty((K, N))
    _load().wqo_wq3_dequant(_ptr(mat), _ptr(scales), _ptr(zeros), K, N, _ptr(out))
    return out


def wq4_dequant(act_bf16, qweight, scales_bits, qzeros, g_idx, group):
    """Exact w(k,n) = s[g(k), n] * (q(k,n) - z[g(k), n]) as float64 [K, N]."""
    qweight = _c(qweight, np.int32); scales = _c(scales_bits, np.uint16)
    R, N = qweight.shape
    K = 8 * R
    assert K % group == 0 and scales.shape == (K // group, N)
    qz = None if qzeros is None else _c(qzeros, np.int32)
    gi = None if g_idx is None else _c(g_idx, np.int32)
    if gi is not None:
        assert gi.shape == (K,) and gi.min() >= 0 and gi.max() < K // group
    out = np.empty((K, N))
    _load().wqo_wq4_dequant(int(bool(act_bf16)), _ptr(qweight), _ptr(scales), _ptr(qz), _ptr(gi), K, N, group,
                            _ptr(out))
    return out


def w8a8_quant_rows(X_bits):
    """Per-row dynamic int8 quantization of bf16 X (bit patterns): (Xq int8, Sx fp32)."""
    X = _c(X_bits, np.uint16)
    M, K = X.shape
    Xq = np.empty((M, K), dtype=np.int8); Sx = np.empty((M,), dtype=np.float32)
    _load().wqo_w8a8_quant_rows(_ptr(X), M, K, _ptr(Xq), _ptr(Sx))
    return Xq, Sx


def w8a8_quant_rows_smooth(X_bits, smooth):
    """Smoothquant's activation side: X / smooth per channel (fp32), then per-row quantization."""
    X = _c(X_bits, np.uint16); s = _c(smooth, np.float32)
    M, K = X.shape
    assert s.shape == (K,)
    Xq = np.empty((M, K), dtype=np.int8); Sx = np.empty((M,), dtype=np.float32)
    _load().wqo_w8a8_quant_rows_smooth(_ptr(X), _ptr(s), M, K, _ptr(Xq), _ptr(Sx))
    return Xq, Sx


def w8a8_gemm_rows(Xq, Sx, W, Sw, rows=None):
    """acc (int64), y (float64, before rounding), abs_sum for the listed rows."""
    Xq = _c(Xq, np.int8); Sx = _c(Sx, np.float32); W = _c(W, np.int8); Sw = _c(Sw, np.float32)
    M, K = Xq.shape
    K2, N = W.shape
    assert K2 == K and Sx.shape == (M,) and Sw.shape == (N,)
    if rows is None:
        r, nr = None, M
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32)); nr = int(r.size)
        assert r.size == 0 or (r.min() >= 0 and r.max() < M)
    acc = np.empty((nr, N), dtype=np.int64); y = np.empty((nr, N)); a = np.empty((nr, N))
    ovf = _load().wqo_w8a8_gemm_rows(_ptr(Xq), _ptr(Sx), _ptr(W), _ptr(Sw), M, K, N, _ptr(r), nr,
                                     _ptr(acc), _ptr(y), _ptr(a))
    return acc, y, a, bool(ovf)


def w8a8_outlier(X_bits, W, Sw, threshold, rows=None):
    """LLM.int8(): (is_outlier, Xq, Sx, acc, y, abs_sum, overflow).  Columns with some
    |x| > threshold go through the 16-bit part; Xq / Sx quantize X with those
    columns set to zero."""
    X = _c(X_bits, np.uint16); W = _c(W, np.int8); Sw = _c(Sw, np.float32)
    M, K = X.shape
    K2, N = W.shape
    assert K2 == K and Sw.shape == (N,)
    flags = np.empty((K,), dtype=np.uint8)
    _load().wqo_w8a8_outlier_columns(_ptr(X), M, K, float(threshold), _ptr(flags))
    Xm = X.copy()
    Xm[:, flags.astype(bool)] = 0          # bf16 +0: the regular part only
    Xq, Sx = w8a8_quant_rows(Xm)
    if rows is None:
        r, nr = None, M
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32)); nr = int(r.size)
    acc = np.empty((nr, N), dtype=np.int64); y = np.empty((nr, N)); a = np.empty((nr, N))
    ovf = _load().wqo_w8a8_outlier_rows(_ptr(X), _ptr(flags), _ptr(Xq), _ptr(Sx), _ptr(W), _ptr(Sw), M, K, N,
                                        _ptr(r), nr, _ptr(acc), _ptr(y), _ptr(a))
    return flags.astype(bool), Xq, Sx, acc, y, a, bool(ovf)


def w8a8_gemm(X_bits, W, Sw, rows=None):
    """The whole W8A8 path: quantize rows, integer product, rescale."""
    Xq, Sx = w8a8_quant_rows(X_bits)
    acc, y, a, ovf = w8a8_gemm_rows(Xq, Sx, W, Sw, rows)
    return Xq, Sx, acc, y, a, ovf
