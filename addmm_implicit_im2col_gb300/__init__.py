"""fp32 addmm and groups==1 NCHW conv2d as one tiled GEMM on sm_103a.

The compute runs in the CUDA library ``libimc.so`` built from ``csrc/``;
``binding`` wraps its C ABI.  Importing this package does not load the
library: the first call into ``binding`` does, and raises if it is missing.
"""
__all__ = ["binding", "synth"]


def __getattr__(name):
    if name in ("addmm", "conv2d", "linear", "gemm_addmm_f32", "conv2d_gemm_f32", "linear_f32"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
