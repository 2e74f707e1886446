"""Python binding of libimc's C ABI (include/imc.h).

The functions named like the C entry points take raw integer device pointers
and return the C status code.  ``addmm`` and ``conv2d`` wrap them for torch
CUDA tensors (PyTorch supplies device memory and the current stream only;
every step of the computation runs in libimc's kernels).  There is no CPU
fallback: the library must be built (``python -m addmm_implicit_im2col_gb300.build``)
and loading it raises otherwise.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libimc.so")

IMC_OK = 0
IMC_ERR_NULL = -1
IMC_ERR_SHAPE = -2
IMC_ERR_ARG = -3
IMC_ERR_ALIAS = -4
IMC_ERR_CUDA = -5
IMC_ERR_TIMEOUT = -6
IMC_ERR_DEVICE = -7
IMC_ERR_SCRATCH = -8
NOALLOC_SCRATCH_BYTES = 32 << 20

MODES = {"default": 0, "tf32": 1, "simt": 2, "force_tc3": 3, "force_tc1": 4, "direct": 5}
ACT_RELU = 0x100
KERNELS = {0: "none", 1: "tc3", 2: "tc1", 3: "simt", 4: "fill", 5: "direct"}

# Every symbol the header declares, with (restype, argtypes).
_i64, _dbl, _vp, _int = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
SIGNATURES = {
    "gemm_addmm_f32": (_int, [_vp, _int, _vp, _vp, _vp, _i64, _i64, _i64, _dbl, _dbl, _vp]),
    "gemm_addmm_f32_ex": (_int, [_vp, _int, _vp, _vp, _vp, _i64, _i64, _i64, _dbl, _dbl, _int,
                                 _vp]),
    "conv2d_gemm_f32": (_int, [_vp, _vp, _vp, _vp] + [_i64] * 10 + [_vp]),
    "conv2d_gemm_f32_ex": (_int, [_vp, _vp, _vp, _vp] + [_i64] * 10 + [_int, _vp]),
    "conv2d_gemm_f32_nd": (_int, [_vp, _vp, _vp, _vp] + [_i64] * 13 + [_int, _vp]),
    "gemm_addmm_f32_ws": (_int, [_vp, _int, _vp, _vp, _vp, _i64, _i64, _i64, _dbl, _dbl, _int,
                                 _vp, ctypes.c_size_t, _vp]),
    "gemm_addmm_f32_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, _int]),
    "conv2d_gemm_f32_ws": (_int, [_vp, _vp, _vp, _vp] + [_i64] * 13 + [_int, _vp, ctypes.c_size_t,
                                                                      _vp]),
    "conv2d_gemm_f32_workspace_bytes": (ctypes.c_size_t, [_i64] * 13 + [_int]),
    "gemm_addmm_f32_noalloc": (_int, [_vp, _int, _vp, _vp, _vp, _i64, _i64, _i64, _dbl, _dbl,
                                      _int, _vp]),
    "linear_f32": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp]),
    "linear_f32_ws": (_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, ctypes.c_size_t, _vp]),
    "linear_f32_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, _int]),
    "gemm_addmm_f32_host": (_int, [_vp, _int, _vp, _vp, _vp, _i64, _i64, _i64, _dbl, _dbl, _int,
                                   _vp]),
    "conv2d_gemm_f32_host": (_int, [_vp, _vp, _vp, _vp] + [_i64] * 13 + [_int, _vp]),
    "imc_status_string": (ctypes.c_char_p, [_int]),
    "imc_last_kernel": (_int, []),
    "imc_last_kernel_name": (ctypes.c_char_p, []),
    "imc_launch_count": (ctypes.c_uint64, []),
    "imc_check_device_error": (_int, [_vp]),
    "imc_version": (_int, []),
    "imc_release_memory": (_int, []),
    "imc_selftest_wait_timeout": (_int, [_int, _vp]),
}

_lock = threading.Lock()
_lib = None


class ImcError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})" if what else
                         f"{status_string(status)} ({status})")


def load(path: str | None = None):
    """Loads libimc.so (once) and declares every exported signature."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"{p} is not built; run python -m addmm_implicit_im2col_gb300.build")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


# ------------------------------------------------------ raw C-ABI mirrors
def gemm_addmm_f32(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, stream) -> int:
    return load().gemm_addmm_f32(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, stream)


def gemm_addmm_f32_ex(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, stream) -> int:
    return load().gemm_addmm_f32_ex(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode,
                                    stream)


def gemm_addmm_f32_ws(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, workspace,
                      workspace_bytes, stream) -> int:
    return load().gemm_addmm_f32_ws(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode,
                                    workspace, workspace_bytes, stream)


def gemm_addmm_f32_noalloc(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode,
                           stream) -> int:
    """The addmm entry point that allocates nothing (fixed library buffer)."""
    return load().gemm_addmm_f32_noalloc(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha,
                                         mode, stream)


def gemm_addmm_f32_workspace_bytes(M, N, K, mode) -> int:
    return int(load().gemm_addmm_f32_workspace_bytes(M, N, K, mode))


def conv2d_gemm_f32(x, w, bias, out, B, IC, H, W, OC, KH, KW, stride, pad, dilation,
                    stream) -> int:
    return load().conv2d_gemm_f32(x, w, bias, out, B, IC, H, W, OC, KH, KW, stride, pad,
                                  dilation, stream)


def conv2d_gemm_f32_ex(x, w, bias, out, B, IC, H, W, OC, KH, KW, stride, pad, dilation, mode,
                       stream) -> int:
    return load().conv2d_gemm_f32_ex(x, w, bias, out, B, IC, H, W, OC, KH, KW, stride, pad,
                                     dilation, mode, stream)


def conv2d_gemm_f32_nd(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, mode,
                       stream) -> int:
    return load().conv2d_gemm_f32_nd(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW,
                                     dH, dW, mode, stream)


def conv2d_gemm_f32_ws(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, mode,
                       workspace, workspace_bytes, stream) -> int:
    return load().conv2d_gemm_f32_ws(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW,
                                     dH, dW, mode, workspace, workspace_bytes, stream)


def conv2d_gemm_f32_workspace_bytes(B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW,
                                    mode) -> int:
    return int(load().conv2d_gemm_f32_workspace_bytes(B, IC, H, W, OC, KH, KW, sH, sW, pH, pW,
                                                      dH, dW, mode))


def linear_f32(x, w, bias, out, M, N, K, mode, stream) -> int:
    return load().linear_f32(x, w, bias, out, M, N, K, mode, stream)


def linear_f32_ws(x, w, bias, out, M, N, K, mode, workspace, workspace_bytes, stream) -> int:
    return load().linear_f32_ws(x, w, bias, out, M, N, K, mode, workspace, workspace_bytes, stream)


def linear_f32_workspace_bytes(M, N, K, mode) -> int:
    return int(load().linear_f32_workspace_bytes(M, N, K, mode))


def gemm_addmm_f32_host(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode,
                        stream) -> int:
    return load().gemm_addmm_f32_host(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode,
                                      stream)


def conv2d_gemm_f32_host(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, mode,
                         stream) -> int:
    return load().conv2d_gemm_f32_host(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW,
                                       dH, dW, mode, stream)


def selftest_wait_timeout(limit_us, stream=None) -> int:
    return load().imc_selftest_wait_timeout(int(limit_us), stream)


def release_memory() -> int:
    return load().imc_release_memory()


def status_string(status: int) -> str:
    return load().imc_status_string(status).decode()


def last_kernel() -> str:
    return KERNELS.get(load().imc_last_kernel(), "unknown")


def last_kernel_name() -> str:
    """Name and form of the main kernel of this thread's last successful call."""
    return load().imc_last_kernel_name().decode()


def launch_count() -> int:
    return int(load().imc_launch_count())


def check_device_error(stream=None) -> int:
    return load().imc_check_device_error(stream)


# ------------------------------------------------------- torch-level API
def _stream_ptr(device):
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_tensor(t, name, ndim=None, host=False):
    import torch
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    where = "CPU" if host else "CUDA"
    placed = t.device.type == "cpu" if host else t.is_cuda
    if not placed or t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 {where} tensor")
    if ndim is not None and t.dim() not in ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")


def _mode(mode, relu):
    return MODES[mode] | (ACT_RELU if relu else 0)


def _addmm_dims(self, mat1, mat2, host):
    _check_tensor(mat1, "mat1", (2,), host)
    _check_tensor(mat2, "mat2", (2,), host)
    _check_tensor(self, "self", (1, 2), host)
    M, K = mat1.shape
    K2, N = mat2.shape
    if K2 != K:
        raise ValueError(f"mat2 must be [K, N] = [{K}, N], got {list(mat2.shape)}")
    self_2d = 0
    if self is not None:
        if self.dim() == 2:
            if list(self.shape) != [M, N]:
                raise ValueError("a 2-D self must be [M, N]")
            self_2d = 1
        elif self.shape[0] != N:
            raise ValueError("a 1-D self must be [N]")
    return M, N, K, self_2d


def _aligned16(t):
    return t.data_ptr() % 16 == 0


def addmm(self, mat1, mat2, *, beta=1.0, alpha=1.0, mode="default", relu=False, out=None):
    """out = beta*self + alpha*(mat1 @ mat2) on the GPU (aten.addmm semantics).

    self is [N] or [M, N]; alpha and beta default to 1.0.  ``mode`` is one of
    ``MODES``; ``relu`` fuses max(v, 0) into the epilogue.  Returns ``out``
    (allocated with torch when not given).
    """
    import torch
    M, N, K, self_2d = _addmm_dims(self, mat1, mat2, host=False)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=mat1.device)
    else:
        _check_tensor(out, "out", (2,))
    # scratch for the transposed mat2 comes from torch's allocator; the size
    # query assumes 16-byte aligned operands, and imc.h documents the extra
    # mat1 copy (M * Kp * 4 bytes) an unaligned mat1 needs
    nbytes = gemm_addmm_f32_workspace_bytes(M, N, K, MODES[mode])
    if nbytes and K % 4 == 0 and not _aligned16(mat1):
        nbytes += M * K * 4 + 256
    ws = torch.empty(nbytes, dtype=torch.uint8, device=mat1.device) if nbytes else None
    rc = gemm_addmm_f32_ws(_ptr(self), self_2d, _ptr(mat1), _ptr(mat2), _ptr(out), M, N, K,
                           float(beta), float(alpha), _mode(mode, relu), _ptr(ws), nbytes,
                           _stream_ptr(mat1.device))
    if rc != IMC_OK:
        raise ImcError(rc, "gemm_addmm_f32")
    return out


def linear(x, w, bias=None, *, mode="default", relu=False, out=None):
    """out = x @ w^T (+ bias) on the GPU (aten.linear semantics).

    x is [M, K], w is [N, K] (the transposed weight), bias [N] or None.
    """
    import torch
    _check_tensor(x, "x", (2,))
    _check_tensor(w, "w", (2,))
    _check_tensor(bias, "bias", (1,))
    M, K = x.shape
    N, K2 = w.shape
    if K2 != K:
        raise ValueError(f"w must be [N, K] = [N, {K}], got {list(w.shape)}")
    if bias is not None and bias.shape[0] != N:
        raise ValueError("bias must be [N]")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out", (2,))
    nbytes = linear_f32_workspace_bytes(M, N, K, MODES[mode])
    if MODES[mode] != MODES["simt"] and K % 4 == 0:
        # the size query assumes 16-byte aligned operands; imc.h documents the
        # copies an unaligned x (M * Kp * 4) or weight (hi and lo, 2 * N * Kp * 4)
        # needs
        if not _aligned16(x):
            nbytes += M * K * 4 + 256
        if not _aligned16(w):
            nbytes += 2 * N * K * 4 + 256
    ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device) if nbytes else None
    rc = linear_f32_ws(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), M, N, K, _mode(mode, relu),
                       _ptr(ws), nbytes, _stream_ptr(x.device))
    if rc != IMC_OK:
        raise ImcError(rc, "linear_f32")
    return out


def conv_out_size(n, k, stride, pad, dil) -> int:
    span = n + 2 * pad - dil * (k - 1) - 1
    return -1 if span < 0 else span // stride + 1


def _pair(v):
    return (int(v[0]), int(v[1])) if isinstance(v, (tuple, list)) else (int(v), int(v))


def _conv_dims(x, w, bias, stride, padding, dilation, host):
    _check_tensor(x, "x", (4,), host)
    _check_tensor(w, "w", (4,), host)
    _check_tensor(bias, "bias", (1,), host)
    B, IC, H, W = x.shape
    OC, IC2, KH, KW = w.shape
    if IC2 != IC:
        raise ValueError("weight must be [OC, IC, KH, KW] with the input's IC (groups == 1)")
    if bias is not None and bias.shape[0] != OC:
        raise ValueError("bias must be [OC]")
    sH, sW = _pair(stride)
    pH, pW = _pair(padding)
    dH, dW = _pair(dilation)
    OH = conv_out_size(H, KH, sH, pH, dH)
    OW = conv_out_size(W, KW, sW, pW, dW)
    if OH < 1 or OW < 1:
        raise ValueError("empty convolution output")
    return B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, OH, OW


def conv2d(x, w, bias=None, stride=1, padding=0, dilation=1, *, mode="default", relu=False,
           out=None):
    """groups==1 NCHW conv2d via the implicit-im2col GEMM.

    x [B, IC, H, W], w [OC, IC, KH, KW], bias [OC] or None; stride, padding and
    dilation are ints or (h, w) pairs.  Returns out [B, OC, OH, OW].
    """
    import torch
    B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, OH, OW = _conv_dims(
        x, w, bias, stride, padding, dilation, host=False)
    if out is None:
        out = torch.empty((B, OC, OH, OW), dtype=torch.float32, device=x.device)
    else:
        _check_tensor(out, "out", (4,))
    nbytes = conv2d_gemm_f32_workspace_bytes(B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW,
                                             MODES[mode])
    ws = torch.empty(nbytes, dtype=torch.uint8, device=x.device) if nbytes else None
    rc = conv2d_gemm_f32_ws(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), B, IC, H, W, OC, KH, KW,
                            sH, sW, pH, pW, dH, dW, _mode(mode, relu), _ptr(ws), nbytes,
                            _stream_ptr(x.device))
    if rc != IMC_OK:
        raise ImcError(rc, "conv2d_gemm_f32")
    return out


# ------------------------------------------------- host-buffer entry points
def _host_stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def addmm_host(self, mat1, mat2, *, beta=1.0, alpha=1.0, mode="default", relu=False, out=None,
               stream=None):
    """addmm on CPU tensors through gemm_addmm_f32_host: the library copies the
    inputs to the GPU, computes there and copies ``out`` back, all enqueued on
    ``stream`` (a torch.cuda.Stream; None: the current stream).  Returns ``out``
    at once; it holds the result after ``stream.synchronize()``.  Page-locked
    tensors (``pin_memory()``) let the copies run asynchronously.
    """
    import torch
    M, N, K, self_2d = _addmm_dims(self, mat1, mat2, host=True)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, pin_memory=mat1.is_pinned())
    else:
        _check_tensor(out, "out", (2,), host=True)
    rc = gemm_addmm_f32_host(_ptr(self), self_2d, _ptr(mat1), _ptr(mat2), _ptr(out), M, N, K,
                             float(beta), float(alpha), _mode(mode, relu), _host_stream(stream))
    if rc != IMC_OK:
        raise ImcError(rc, "gemm_addmm_f32_host")
    return out


def conv2d_host(x, w, bias=None, stride=1, padding=0, dilation=1, *, mode="default", relu=False,
                out=None, stream=None):
    """conv2d on CPU tensors through conv2d_gemm_f32_host (as ``addmm_host``)."""
    import torch
    B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, OH, OW = _conv_dims(
        x, w, bias, stride, padding, dilation, host=True)
    if out is None:
        out = torch.empty((B, OC, OH, OW), dtype=torch.float32, pin_memory=x.is_pinned())
    else:
        _check_tensor(out, "out", (4,), host=True)
    rc = conv2d_gemm_f32_host(_ptr(x), _ptr(w), _ptr(bias), _ptr(out), B, IC, H, W, OC, KH, KW,
                              sH, sW, pH, pW, dH, dW, _mode(mode, relu), _host_stream(stream))
    if rc != IMC_OK:
        raise ImcError(rc, "conv2d_gemm_f32_host")
    return out
