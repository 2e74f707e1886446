"""CPU oracle for fp32 addmm and groups==1 NCHW conv2d -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  It is a ctypes wrapper around
``oracle.c`` (plain C, fp64 accumulation), which shares no code with the CUDA
path.  Every function here returns fp64 numpy arrays.

Definitions followed (ExecuTorch WebGPU pull-request pages):
  * addmm -- "Add optimized addmm op", Solution / Implementation paragraphs:
    out = beta*self + alpha*(mat1 @ mat2), self broadcast from [N] or given as
    [M, N], mat2 read as mat2[k*N + n].
  * conv2d -- "et_vk conv2d: route standard (groups==1) conv through an im2col
    tiled GEMM", Problem / Solution / Implementation paragraphs: direct
    convolution, ih = oh*sH - pH + kh*dH, out-of-range taps read 0, per-channel
    bias, NCHW output.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_HDR = os.path.join(_HERE, "oracle.h")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_dbl = ctypes.c_double
_ptr = ctypes.c_void_p


def build(force: bool = False, extra_flags=(), out_path: str | None = None) -> str:
    """Compiles oracle.c with gcc (-O2, no fast-math) into a shared library."""
    out_path = out_path or _LIB_PATH
    stale = (not os.path.exists(out_path)
             or os.path.getmtime(out_path) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = out_path + f".tmp{os.getpid()}"
        # -ffp-contract=off: no fused multiply-adds, so the fp32 loop rounds
        # every product and every partial sum to fp32 on any host
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
               *extra_flags,
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out_path)
    return out_path


def _load(path: str | None = None):
    lib = ctypes.CDLL(path or build())
    lib.oracle_addmm.restype = ctypes.c_int
    lib.oracle_addmm.argtypes = [_ptr, ctypes.c_int, _ptr, _ptr, _i64, _i64, _i64, _dbl, _dbl,
                                 _ptr, _i64, ctypes.c_int, _ptr, _ptr]
    lib.oracle_addmm_fp32_naive.restype = ctypes.c_int
    lib.oracle_addmm_fp32_naive.argtypes = [_ptr, ctypes.c_int, _ptr, _ptr, _i64, _i64, _i64,
                                            ctypes.c_float, ctypes.c_float, _ptr]
    lib.oracle_conv_out_size.restype = _i64
    lib.oracle_conv_out_size.argtypes = [_i64] * 5
    lib.oracle_conv2d.restype = ctypes.c_int
    lib.oracle_conv2d.argtypes = [_ptr, _ptr, _ptr] + [_i64] * 13 + [_ptr, _i64, ctypes.c_int,
                                                                      _ptr, _ptr]
    lib.oracle_default_threads.restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    return lib


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load()
        return _lib


def _f32(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.float32)


def _p(a):
    return None if a is None else a.ctypes.data


class OracleError(RuntimeError):
    pass


def default_threads() -> int:
    return int(lib().oracle_default_threads())


def addmm(self, mat1, mat2, beta=1.0, alpha=1.0, rows=None, nthreads=0, self_2d=None,
          _lib=None):
    """fp64 reference of beta*self + alpha*(mat1 @ mat2) on the selected rows.

    Returns (ref, S), both [len(rows), N] fp64 (all rows when rows is None).
    ``self`` may be None when beta == 0.  ``self_2d`` defaults to self.ndim == 2.
    """
    L = _lib or lib()
    mat1 = _f32(mat1)
    mat2 = _f32(mat2)
    self = _f32(self)
    M, K = mat1.shape
    K2, N = mat2.shape
    if K2 != K:
        raise OracleError("mat2 must be [K, N]")
    if self_2d is None:
        self_2d = bool(self is not None and self.ndim == 2)
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = M if rows_arr is None else rows_arr.shape[0]
    ref = np.empty((nrows, N), dtype=np.float64)
    sabs = np.empty((nrows, N), dtype=np.float64)
    rc = L.oracle_addmm(_p(self), int(self_2d), _p(mat1), _p(mat2), M, N, K, float(beta),
                        float(alpha), _p(rows_arr), nrows, int(nthreads), _p(ref), _p(sabs))
    if rc != 0:
        raise OracleError(f"oracle_addmm returned {rc}")
    return ref, sabs


def addmm_fp32_naive(self, mat1, mat2, beta=1.0, alpha=1.0, _lib=None):
    """beta*self + alpha*(mat1 @ mat2) with one fp32 accumulator per output."""
    L = _lib or lib()
    mat1, mat2, self = _f32(mat1), _f32(mat2), _f32(self)
    M, K = mat1.shape
    N = mat2.shape[1]
    out = np.empty((M, N), dtype=np.float32)
    rc = L.oracle_addmm_fp32_naive(_p(self), int(self.ndim == 2), _p(mat1), _p(mat2), M, N, K,
                                   float(beta), float(alpha), _p(out))
    if rc != 0:
        raise OracleError(f"oracle_addmm_fp32_naive returned {rc}")
    return out


def conv_out_size(n, k, stride, pad, dil, _lib=None) -> int:
    return int((_lib or lib()).oracle_conv_out_size(n, k, stride, pad, dil))


def _pair(v):
    if isinstance(v, (tuple, list)):
        return int(v[0]), int(v[1])
    return int(v), int(v)


def conv2d(x, w, bias=None, stride=1, padding=0, dilation=1, channels=None, nthreads=0,
           _lib=None):
    """fp64 direct convolution on the selected output channels.

    x [B,IC,H,W], w [OC,IC,KH,KW], bias [OC] or None.  stride / padding /
    dilation are ints or (h, w) pairs.  Returns (ref, S), both
    [B, len(channels), OH, OW] fp64 (all channels when channels is None).
    """
    L = _lib or lib()
    x, w, bias = _f32(x), _f32(w), _f32(bias)
    B, IC, H, W = x.shape
    OC, IC2, KH, KW = w.shape
    if IC2 != IC:
        raise OracleError("weight must be [OC, IC, KH, KW] with the input's IC")
    sH, sW = _pair(stride)
    pH, pW = _pair(padding)
    dH, dW = _pair(dilation)
    OH = conv_out_size(H, KH, sH, pH, dH, _lib=L)
    OW = conv_out_size(W, KW, sW, pW, dW, _lib=L)
    if OH < 1 or OW < 1:
        raise OracleError("empty output")
    ch = None if channels is None else np.ascontiguousarray(channels, dtype=np.int64)
    nocs = OC if ch is None else ch.shape[0]
    ref = np.empty((B, nocs, OH, OW), dtype=np.float64)
    sabs = np.empty((B, nocs, OH, OW), dtype=np.float64)
    rc = L.oracle_conv2d(_p(x), _p(w), _p(bias), B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW,
                         _p(ch), nocs, int(nthreads), _p(ref), _p(sabs))
    if rc != 0:
        raise OracleError(f"oracle_conv2d returned {rc}")
    return ref, sabs


def load_variant(path: str):
    """Loads another build of oracle.c (used by tests that plant a mistake)."""
    return _load(path)
