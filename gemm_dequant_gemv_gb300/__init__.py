"""Python binding of libwq.so (ctypes): the same entry points as include/wq.h.

This module only marshals arguments: tensors become device pointers
(``data_ptr()``), streams become ``cudaStream_t`` handles, and a non-zero
status raises :class:`WQError`.  Every step of the computation runs in the
CUDA kernels of libwq.so; there is no fallback of any kind, and importing this
package fails loudly when the library has not been built.

PyTorch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")

WQ_OK, WQ_ERR_NULL, WQ_ERR_SHAPE, WQ_ERR_ALIGN, WQ_ERR_UNSUPPORTED, WQ_ERR_WORKSPACE, WQ_ERR_CUDA, \
    WQ_ERR_TIMEOUT = range(8)
WQ_F16, WQ_BF16 = 1, 2
WQ_FLAG_PDL = 1

# Every entry point of include/wq.h, with its ctypes signature.
_P, _I, _U, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_size_t
SIGNATURES = {
    "wq_status_string": (ctypes.c_char_p, [_I]),
    "wq_abi_version": (_I, []),
    "wq_read_timeout_flag": (_I, [_I]),
    "wq8_gemv": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _U, _P]),
    "wq3_gemv": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _U, _P]),
    "wq4_gemm": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _SZ, _U, _P]),
    "wq4_actorder_prepare": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "wq4_gemm_sorted": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _U, _P]),
    "wq8_dequant": (_I, [_P, _P, _P, _I, _I, _I, _U, _P]),
    "wq3_dequant": (_I, [_P, _P, _P, _P, _I, _I, _U, _P]),
    "wq4_dequant": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _U, _P]),
    "w8a8_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _SZ, _U, _P]),
    "w8a8_gemm_smooth": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _SZ, _U, _P]),
    "w8a8_gemm_outlier": (_I, [_P, _P, _P, _P, _I, _I, _I, ctypes.c_float, _P, _P, _P, _P, _P, _SZ, _U, _P]),
    "w8a8_gemm_outlier_workspace_bytes": (_SZ, [_I, _I, _I]),
    "w8a8_gemm_workspace_bytes": (_SZ, [_I, _I, _I]),
    "w8a8_gemm_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _U, _P]),
    "w8a8_gemm_noalloc_max_scratch_bytes": (_SZ, []),
    "wq4_repack_tiled": (_I, [_P, _P, _I, _I, _I, _P, _P, _P]),
    "wq4_gemm_tiled": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _U, _P]),
}


class WQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: status {status} ({status_string(status)})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(nvcc for sm_103a is required; there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()


def library() -> ctypes.CDLL:
    return _lib


def status_string(status: int) -> str:
    return _lib.wq_status_string(int(status)).decode()


def abi_version() -> int:
    return int(_lib.wq_abi_version())


def read_timeout_flag(clear: bool = False) -> int:
    return int(_lib.wq_read_timeout_flag(int(bool(clear))))


def _ptr(t) -> int | None:
    """Device pointer of a tensor (or an int address, or None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(fn: str, status: int) -> None:
    if status != WQ_OK:
        raise WQError(fn, status)


def wq8_gemv(x, w, scales, y, M, K, N, group_size, flags=0, stream=None):
    _check("wq8_gemv", _lib.wq8_gemv(_ptr(x), _ptr(w), _ptr(scales), _ptr(y), M, K, N, group_size,
                                     flags, _stream(stream)))


def wq3_gemv(x, mat, scales, zeros, y, M, K, N, flags=0, stream=None):
    _check("wq3_gemv", _lib.wq3_gemv(_ptr(x), _ptr(mat), _ptr(scales), _ptr(zeros), _ptr(y), M, K, N,
                                     flags, _stream(stream)))


def wq4_gemm(x, qweight, scales, qzeros, g_idx, y, M, K, N, group_size, act_dtype,
             workspace=None, workspace_bytes=0, flags=0, stream=None):
    _check("wq4_gemm", _lib.wq4_gemm(_ptr(x), _ptr(qweight), _ptr(scales), _ptr(qzeros), _ptr(g_idx),
                                     _ptr(y), M, K, N, group_size, act_dtype, _ptr(workspace),
                                     workspace_bytes, flags, _stream(stream)))


def wq4_actorder_prepare(qweight, g_idx, K, N, group_size, qweight_sorted, perm, stream=None):
    _check("wq4_actorder_prepare", _lib.wq4_actorder_prepare(_ptr(qweight), _ptr(g_idx), K, N, group_size,
                                                             _ptr(qweight_sorted), _ptr(perm), _stream(stream)))


def wq4_gemm_sorted(x, qweight_sorted, scales, qzeros, perm, y, M, K, N, group_size, act_dtype, flags=0,
                    stream=None):
    _check("wq4_gemm_sorted", _lib.wq4_gemm_sorted(_ptr(x), _ptr(qweight_sorted), _ptr(scales), _ptr(qzeros),
                                                   _ptr(perm), _ptr(y), M, K, N, group_size, act_dtype, flags,
                                                   _stream(stream)))


def wq4_repack_tiled(qweight, g_idx, K, N, group_size, qweight_tiled, perm=None, stream=None):
    _check("wq4_repack_tiled", _lib.wq4_repack_tiled(_ptr(qweight), _ptr(g_idx), K, N, group_size,
                                                     _ptr(qweight_tiled), _ptr(perm), _stream(stream)))


def wq4_gemm_tiled(x, qweight_tiled, scales, qzeros, perm, y, M, K, N, group_size, act_dtype, flags=0,
                   stream=None):
    _check("wq4_gemm_tiled", _lib.wq4_gemm_tiled(_ptr(x), _ptr(qweight_tiled), _ptr(scales), _ptr(qzeros),
                                                 _ptr(perm), _ptr(y), M, K, N, group_size, act_dtype, flags,
                                                 _stream(stream)))


def wq8_dequant(w, scales, w_out, K, N, group_size, flags=0, stream=None):
    _check("wq8_dequant", _lib.wq8_dequant(_ptr(w), _ptr(scales), _ptr(w_out), K, N, group_size, flags,
                                           _stream(stream)))


def wq3_dequant(mat, scales, zeros, w_out, K, N, flags=0, stream=None):
    _check("wq3_dequant", _lib.wq3_dequant(_ptr(mat), _ptr(scales), _ptr(zeros), _ptr(w_out), K, N, flags,
                                           _stream(stream)))


def wq4_dequant(qweight, scales, qzeros, g_idx, w_out, K, N, group_size, act_dtype, flags=0, stream=None):
    _check("wq4_dequant", _lib.wq4_dequant(_ptr(qweight), _ptr(scales), _ptr(qzeros), _ptr(g_idx), _ptr(w_out),
                                           K, N, group_size, act_dtype, flags, _stream(stream)))


def w8a8_gemm_workspace_bytes(M, K, N) -> int:
    return int(_lib.w8a8_gemm_workspace_bytes(M, K, N))


def w8a8_gemm(X, W, Sw, Y, M, K, N, Xq_out=None, Sx_out=None, acc_out=None, workspace=None,
              workspace_bytes=0, flags=0, stream=None):
    _check("w8a8_gemm", _lib.w8a8_gemm(_ptr(X), _ptr(W), _ptr(Sw), _ptr(Y), M, K, N, _ptr(Xq_out),
                                       _ptr(Sx_out), _ptr(acc_out), _ptr(workspace), workspace_bytes,
                                       flags, _stream(stream)))


def w8a8_gemm_smooth(X, smooth, W, Sw, Y, M, K, N, Xq_out=None, Sx_out=None, acc_out=None, workspace=None,
                     workspace_bytes=0, flags=0, stream=None):
    _check("w8a8_gemm_smooth", _lib.w8a8_gemm_smooth(_ptr(X), _ptr(smooth), _ptr(W), _ptr(Sw), _ptr(Y), M, K, N,
                                                     _ptr(Xq_out), _ptr(Sx_out), _ptr(acc_out), _ptr(workspace),
                                                     workspace_bytes, flags, _stream(stream)))


def w8a8_gemm_outlier_workspace_bytes(M, K, N) -> int:
    return int(_lib.w8a8_gemm_outlier_workspace_bytes(M, K, N))


def w8a8_gemm_outlier(X, W, Sw, Y, M, K, N, threshold=6.0, Xq_out=None, Sx_out=None, acc_out=None,
                      n_outliers_out=None, workspace=None, workspace_bytes=0, flags=0, stream=None):
    _check("w8a8_gemm_outlier", _lib.w8a8_gemm_outlier(_ptr(X), _ptr(W), _ptr(Sw), _ptr(Y), M, K, N, float(threshold),
                                                       _ptr(Xq_out), _ptr(Sx_out), _ptr(acc_out),
                                                       _ptr(n_outliers_out), _ptr(workspace), workspace_bytes,
                                                       flags, _stream(stream)))


def w8a8_gemm_noalloc_max_scratch_bytes() -> int:
    return int(_lib.w8a8_gemm_noalloc_max_scratch_bytes())


def w8a8_gemm_noalloc(X, W, Sw, Y, M, K, N, Xq_out=None, Sx_out=None, acc_out=None, flags=0, stream=None):
    """w8a8_gemm on the library's built-in scratch: allocates nothing.  All calls
    on one device share that scratch, so calls that can overlap race."""
    _check("w8a8_gemm_noalloc", _lib.w8a8_gemm_noalloc(_ptr(X), _ptr(W), _ptr(Sw), _ptr(Y), M, K, N, _ptr(Xq_out),
                                                       _ptr(Sx_out), _ptr(acc_out), flags, _stream(stream)))
