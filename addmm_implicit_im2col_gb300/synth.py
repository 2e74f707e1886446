"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the benchmark.

This module only draws numbers: it holds none of the addmm / convolution
arithmetic, and neither the oracle nor the CUDA path is imported from here.

Generator: a counter-based SplitMix64 stream.  Element ``i`` of stream
``key`` is ``mix64(key + (i + 1) * GOLDEN)`` where ``mix64`` is the SplitMix64
finaliser (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014).  Uniforms take the top 24 bits (so every U(0,1)
value is an exact fp32 number); normals use the Box-Muller transform on two
53-bit uniforms.  ``N(mu, sigma)`` takes the standard deviation as its second
argument (torch.normal convention).

Every tensor of a workload gets its own stream key derived from
(seed, workload id, tensor id), so tensors never share draws.
"""
from __future__ import annotations

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, workload: int, tensor: int) -> int:
    """64-bit key of one tensor's stream."""
    with np.errstate(over="ignore"):
        a = _mix64(np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF)]) + GOLDEN)[0]
        b = np.uint64(((workload & 0xFFFFFFFF) << 32) | (tensor & 0xFFFFFFFF))
        return int(_mix64(np.array([a ^ b]))[0])


def raw_u64(key: int, start: int, count: int) -> np.ndarray:
    """Draws ``start .. start+count-1`` of stream ``key`` as uint64."""
    with np.errstate(over="ignore"):
        i = np.arange(start + 1, start + count + 1, dtype=np.uint64)
        return _mix64(np.uint64(key) + i * GOLDEN)


def uniform(key: int, n: int, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    """n fp32 values lo + (hi - lo) * u with u on the 2^-24 grid of [0, 1)."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        u = (raw_u64(key, s, c) >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))
        out[s:s + c] = (lo + (hi - lo) * u).astype(np.float32)
    return out


def normal(key: int, n: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """n fp32 values mean + std * z, z standard normal by Box-Muller."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        r = raw_u64(key, 2 * s, 2 * c)
        u1 = ((r[0::2] >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / (1 << 53))
        u2 = (r[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / (1 << 53))
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        out[s:s + c] = (mean + std * z).astype(np.float32)
    return out


def integers(key: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n fp32 values drawn uniformly from the integers lo..hi (inclusive)."""
    r = raw_u64(key, 0, n)
    span = np.uint64(hi - lo + 1)
    return (lo + (r % span).astype(np.int64)).astype(np.float32)


def log_uniform(key: int, n: int, lo_exp: float, hi_exp: float) -> np.ndarray:
    """n fp32 values +-10^e, e uniform in [lo_exp, hi_exp), the sign from the
    stream's lowest bit (a wide dynamic range)."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        r = raw_u64(key, s, c)
        u = (r >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))
        sign = np.where((r & np.uint64(1)) == 0, 1.0, -1.0)
        out[s:s + c] = (sign * 10.0 ** (lo_exp + (hi_exp - lo_exp) * u)).astype(np.float32)
    return out


def sample_rows(key: int, total: int, count: int) -> np.ndarray:
    """``count`` distinct sorted indices in [0, total), chosen by the stream."""
    if count >= total:
        return np.arange(total, dtype=np.int64)
    order = np.argsort(raw_u64(key, 0, total), kind="stable")
    return np.sort(order[:count]).astype(np.int64)


# --------------------------------------------------------------------------
# Workload recipes (shapes and value distributions of the pages' workloads)
# --------------------------------------------------------------------------

def _draw(spec, key, n):
    kind = spec[0]
    if kind == "U":
        return uniform(key, n, spec[1], spec[2])
    if kind == "N":
        return normal(key, n, spec[1], spec[2])
    if kind == "I":
        return integers(key, n, spec[1], spec[2])
    if kind == "L":
        return log_uniform(key, n, spec[1], spec[2])
    raise ValueError(kind)


def addmm_inputs(M, N, K, *, self_2d, seed=0, workload=0, mat1=("U", -1.0, 1.0),
                 mat2=("U", -1.0, 1.0), self_=("U", -1.0, 1.0)):
    """Returns (self, mat1, mat2) as contiguous fp32 numpy arrays.

    self is [M, N] when self_2d else [N]; mat1 is [M, K]; mat2 is [K, N].
    """
    a = _draw(mat1, stream_key(seed, workload, 1), M * K).reshape(M, K)
    b = _draw(mat2, stream_key(seed, workload, 2), K * N).reshape(K, N)
    s = _draw(self_, stream_key(seed, workload, 3), (M * N) if self_2d else N)
    s = s.reshape(M, N) if self_2d else s
    return s, a, b


def conv_inputs(B, IC, H, W, OC, KH, KW, *, seed=0, workload=0, x=("U", 0.0, 1.0),
                w=("N", 0.0, 1.0), bias=("N", 0.0, 0.02)):
    """Returns (x [B,IC,H,W], w [OC,IC,KH,KW], bias [OC] or None) as fp32 numpy arrays."""
    xx = _draw(x, stream_key(seed, workload, 1), B * IC * H * W).reshape(B, IC, H, W)
    ww = _draw(w, stream_key(seed, workload, 2), OC * IC * KH * KW).reshape(OC, IC, KH, KW)
    bb = None if bias is None else _draw(bias, stream_key(seed, workload, 3), OC)
    return xx, ww, bb


# The workloads of the pages' benchmark table, one entry per case.  ``wid`` is
# the stream id of the case; ``rows`` is how many output rows (addmm) the
# oracle checks at full size.
ADDMM_CASES = {
    "tiny_selfN": dict(M=64, N=80, K=96, self_2d=False, alpha=1.0, beta=1.0, wid=11,
                       mat1=("U", -1.0, 1.0), mat2=("U", -1.0, 1.0), self_=("U", -1.0, 1.0)),
    "tiny_selfMN": dict(M=64, N=80, K=96, self_2d=True, alpha=2.0, beta=0.5, wid=12,
                        mat1=("U", -1.0, 1.0), mat2=("U", -1.0, 1.0), self_=("U", -1.0, 1.0)),
}
for _M in (1024, 577):
    for _K, _N in ((768, 3072), (3072, 768), (768, 768)):
        _s = 1.0 / np.sqrt(_K)
        ADDMM_CASES[f"linear_M{_M}_K{_K}_N{_N}"] = dict(
            M=_M, N=_N, K=_K, self_2d=False, alpha=1.0, beta=1.0, wid=20 + len(ADDMM_CASES),
            mat1=("N", 0.0, 1.0), mat2=("U", -_s, _s), self_=("N", 0.0, 0.02))
ADDMM_CASES["large_8192x4096x4096"] = dict(
    M=8192, N=4096, K=4096, self_2d=False, alpha=1.0, beta=1.0, wid=51,
    mat1=("N", 0.0, 1.0 / 64.0), mat2=("N", 0.0, 1.0 / 64.0), self_=("N", 0.0, 1.0), rows=256)
ADDMM_CASES["tall_32768x1024x1024"] = dict(
    M=32768, N=1024, K=1024, self_2d=True, alpha=0.75, beta=1.25, wid=52,
    mat1=("N", 0.0, 1.0 / 32.0), mat2=("N", 0.0, 1.0 / 32.0), self_=("N", 0.0, 1.0), rows=256)

CONV_CASES = {
    "stem_768_7x7_s4": dict(B=1, IC=3, H=768, W=768, OC=128, KH=7, KW=7, stride=4, pad=3,
                            dilation=1, wid=31, x=("U", 0.0, 1.0),
                            w=("N", 0.0, 1.0 / np.sqrt(147.0)), bias=("N", 0.0, 0.02)),
    "body_56_3x3_d1": dict(B=8, IC=256, H=56, W=56, OC=256, KH=3, KW=3, stride=1, pad=1,
                           dilation=1, wid=41, x=("N", 0.0, 1.0),
                           w=("N", 0.0, 1.0 / 48.0), bias=("N", 0.0, 0.02)),
    "body_56_3x3_d2": dict(B=8, IC=256, H=56, W=56, OC=256, KH=3, KW=3, stride=1, pad=2,
                           dilation=2, wid=42, x=("N", 0.0, 1.0),
                           w=("N", 0.0, 1.0 / 48.0), bias=("N", 0.0, 0.02)),
}


def make_addmm_case(name, seed=0):
    c = ADDMM_CASES[name]
    s, a, b = addmm_inputs(c["M"], c["N"], c["K"], self_2d=c["self_2d"], seed=seed,
                           workload=c["wid"], mat1=c["mat1"], mat2=c["mat2"], self_=c["self_"])
    return c, s, a, b


def make_conv_case(name, seed=0):
    c = CONV_CASES[name]
    x, w, bias = conv_inputs(c["B"], c["IC"], c["H"], c["W"], c["OC"], c["KH"], c["KW"],
                             seed=seed, workload=c["wid"], x=c["x"], w=c["w"], bias=c["bias"])
    return c, x, w, bias


def checked_rows(name, total, count=256, seed=0):
    """The seeded output rows a full-size case is checked on."""
    c = ADDMM_CASES.get(name) or CONV_CASES.get(name)
    return sample_rows(stream_key(seed, c["wid"], 99), total, count)
