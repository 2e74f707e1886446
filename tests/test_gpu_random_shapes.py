"""GPU parity on seeded random shapes: addmm, linear and conv2d in every mode against
the oracle, to reach planner paths the hand-picked cases may miss (tile widths
of 16 mod 32, K-slices, ragged edges, the conv's two slab forms with few input
channels, per-axis stride / padding / dilation).

Shapes come from a fixed numpy generator (the same list on every run), sized so
that the oracle finishes each case in about a second at most; a few extreme
addmm shapes (a handful of rows or columns, K up to 20000 with a small output)
stand beside the general ones.  The tolerance is
the one the other parity tests use: 1e-5 * S + 1e-6 per element for 3xTF32 and
SIMT, 2e-3 * S + 1e-6 for 1xTF32 (S = the sum of |products| of the element).
"""
import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

TOL = {"default": 1e-5, "force_tc3": 1e-5, "force_tc1": 2e-3, "simt": 1e-5}
MODES = ["default", "force_tc3", "force_tc1"]


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    binding.load()


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def within(got, ref, S, c, what):
    err = np.abs(np.asarray(got, np.float64) - ref)
    ratio = float((err / (c * S + 1e-6)).max()) if err.size else 0.0
    assert ratio <= 1.0, f"{what}: worst |err|/tol = {ratio:.3g}"


def _addmm_shapes(n=60, seed=2024):
    rng = np.random.RandomState(seed)
    out = []
    while len(out) < n:
        M, N, K = int(rng.randint(1, 1300)), int(rng.randint(1, 3300)), int(rng.randint(1, 1300))
        if M * N * K > 6e8:
            continue
        out.append((M, N, K, bool(rng.randint(2)), float(rng.choice([1.0, 0.5, -1.25, 0.0])),
                    float(rng.choice([1.0, 2.0, 0.75]))))
    return out


def _addmm_extreme_shapes(n=16, seed=4242):
    """Few rows with long rows, long K with a small output (many K-slices), and
    one to eight columns."""
    rng = np.random.RandomState(seed)
    out = []
    while len(out) < n:
        kind = len(out) % 3
        if kind == 0:
            M, N, K = int(rng.randint(1, 17)), int(rng.randint(1, 9000)), int(rng.randint(1, 9000))
        elif kind == 1:
            M, N, K = int(rng.randint(1, 400)), int(rng.randint(1, 400)), int(rng.randint(2000, 20000))
        else:
            M, N, K = int(rng.randint(1, 9000)), int(rng.randint(1, 9)), int(rng.randint(1, 4000))
        if M * N * K > 3e8:
            continue
        out.append((M, N, K, bool(rng.randint(2))))
    return out


def _conv_shapes(n=60, seed=7):
    rng = np.random.RandomState(seed)
    out = []
    while len(out) < n:
        B, IC, OC = int(rng.randint(1, 4)), int(rng.randint(1, 40)), int(rng.randint(1, 300))
        KH, KW = int(rng.randint(1, 8)), int(rng.randint(1, 8))
        s = (int(rng.randint(1, 5)), int(rng.randint(1, 5)))
        p = (int(rng.randint(0, 4)), int(rng.randint(0, 4)))
        d = (int(rng.randint(1, 3)), int(rng.randint(1, 3)))
        H = int(rng.randint(1, 90))
        kind = len(out) % 3
        if kind == 0:
            W = int(rng.randint(1, 130))
        else:
            # few input channels, W and OW multiples of 4 (kind 1), or OW a
            # multiple of 32 and OH of 4 (kind 2): the slab form's territory
            IC = int(rng.randint(1, 8 if kind == 1 else 5))
            OW = 4 * int(rng.randint(2, 48)) if kind == 1 else 32 * int(rng.randint(1, 5))
            w_min = (OW - 1) * s[1] + d[1] * (KW - 1) + 1 - 2 * p[1]
            W = (max(w_min, 4) + 3) // 4 * 4
            if kind == 2:
                OH = 4 * int(rng.randint(1, 12))
                H = max(1, (OH - 1) * s[0] + d[0] * (KH - 1) + 1 - 2 * p[0])
        OH = (H + 2 * p[0] - d[0] * (KH - 1) - 1) // s[0] + 1
        OW = (W + 2 * p[1] - d[1] * (KW - 1) - 1) // s[1] + 1
        if OH < 1 or OW < 1 or B * OC * OH * OW * IC * KH * KW > 2.5e8:
            continue
        out.append((B, IC, H, W, OC, KH, KW, s, p, d))
    return out


def _conv_t_shapes(n=16, seed=31):
    """Stem-like convs the transposed slab form takes: IC < 8, OC <= 128, W and
    OW multiples of 4, 114 to 152 tiles of 8 output rows x 32 columns over the
    batch, at least 3/4 of the tiles' positions real, the input window of a
    tile at most 64 KB and K at most 2048."""
    rng = np.random.RandomState(seed)
    out = []
    while len(out) < n:
        IC, OC = int(rng.randint(1, 8)), int(rng.randint(1, 129))
        KH, KW = int(rng.randint(1, 8)), int(rng.randint(1, 8))
        s = (int(rng.randint(1, 5)), int(rng.randint(1, 5)))
        p = (int(rng.randint(0, 4)), int(rng.randint(0, 4)))
        d = (int(rng.randint(1, 3)), int(rng.randint(1, 3)))
        OW = 4 * int(rng.randint(6, 64))
        OH = int(rng.randint(8, 120))
        w_min = (OW - 1) * s[1] + d[1] * (KW - 1) + 1 - 2 * p[1]
        W = (max(w_min, 4) + 3) // 4 * 4
        H = max(1, (OH - 1) * s[0] + d[0] * (KH - 1) + 1 - 2 * p[0])
        OH = (H + 2 * p[0] - d[0] * (KH - 1) - 1) // s[0] + 1
        OW = (W + 2 * p[1] - d[1] * (KW - 1) - 1) // s[1] + 1
        if OH < 1 or OW < 1 or OW % 4:
            continue
        tw, th = -(-OW // 32), -(-OH // 8)
        B = max(1, round(133 / (tw * th)))
        tiles = B * tw * th
        off = (4 - p[1] % 4) % 4
        bw = (off + 31 * s[1] + (KW - 1) * d[1] + 1 + 3) // 4 * 4
        rows = 7 * s[0] + (KH - 1) * d[0] + 1
        if not (114 <= tiles <= 152) or 4 * OW * OH < 3 * tw * 32 * th * 8:
            continue
        if bw > 256 or rows > 256 or IC * rows * bw * 4 > 65536 or IC * KH * KW > 2048:
            continue
        out.append((B, IC, H, W, OC, KH, KW, s, p, d))
    return out


def _linear_shapes(n=24, seed=99):
    rng = np.random.RandomState(seed)
    out = []
    while len(out) < n:
        M, N, K = int(rng.randint(1, 1500)), int(rng.randint(1, 3300)), int(rng.randint(1, 3300))
        if M * N * K > 6e8:
            continue
        out.append((M, N, K, bool(rng.randint(2)), bool(rng.randint(2))))
    return out


ADDMM = _addmm_shapes()
ADDMM_EXTREME = _addmm_extreme_shapes()
CONV = _conv_shapes()
CONV_T = _conv_t_shapes()
LINEAR = _linear_shapes()


@pytest.mark.parametrize("idx", range(len(ADDMM)))
def test_random_addmm(idx):
    M, N, K, s2, beta, alpha = ADDMM[idx]
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=s2, workload=1000 + idx)
    relu = idx % 3 == 1
    for mode in MODES:
        # 1xTF32: the tensor core truncates both operands, a product is off by
        # up to ~1.95e-3 of |a*b| times |alpha|, so its bound holds for
        # |alpha| <= 1 only (the pages' reading kept as written)
        al = max(-1.0, min(1.0, alpha)) if mode == "force_tc1" else alpha
        ref, S = oracle.addmm(s, a, b, beta=beta, alpha=al)
        if relu:
            ref = np.maximum(ref, 0.0)
        out = binding.addmm(dev(s), dev(a), dev(b), beta=beta, alpha=al, mode=mode, relu=relu)
        torch.cuda.synchronize()
        within(out.cpu().numpy(), ref, S, TOL[mode],
               f"addmm {M}x{N}x{K} self_2d={s2} beta={beta} alpha={al} {mode} "
               f"({binding.last_kernel_name()})")


@pytest.mark.parametrize("idx", range(len(ADDMM_EXTREME)))
def test_random_addmm_extreme_shapes(idx):
    M, N, K, s2 = ADDMM_EXTREME[idx]
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=s2, workload=1800 + idx)
    ref, S = oracle.addmm(s, a, b)
    for mode in MODES:
        out = binding.addmm(dev(s), dev(a), dev(b), mode=mode)
        torch.cuda.synchronize()
        within(out.cpu().numpy(), ref, S, TOL[mode],
               f"addmm {M}x{N}x{K} self_2d={s2} {mode} ({binding.last_kernel_name()})")


@pytest.mark.parametrize("idx", range(len(CONV)))
def test_random_conv(idx):
    B, IC, H, W, OC, KH, KW, st, pd, dl = CONV[idx]
    x, w, bias = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=1100 + idx)
    ref, S = oracle.conv2d(x, w, bias, st, pd, dl)
    relu = idx % 3 == 1
    if relu:
        ref = np.maximum(ref, 0.0)
    for mode in MODES:
        out = binding.conv2d(dev(x), dev(w), dev(bias), st, pd, dl, mode=mode, relu=relu)
        torch.cuda.synchronize()
        within(out.cpu().numpy(), ref, S, TOL[mode],
               f"conv {B}x{IC}x{H}x{W}->{OC} {KH}x{KW} s{st} p{pd} d{dl} {mode} "
               f"({binding.last_kernel_name()})")


@pytest.mark.parametrize("idx", range(len(LINEAR)))
def test_random_linear(idx):
    M, N, K, with_bias, relu = LINEAR[idx]
    x = synth.normal(synth.stream_key(0, 1200 + idx, 1), M * K).reshape(M, K)
    sc = 1.0 / np.sqrt(K)
    w = synth.uniform(synth.stream_key(0, 1200 + idx, 2), N * K, -sc, sc).reshape(N, K)
    b = synth.normal(synth.stream_key(0, 1200 + idx, 3), N, 0.0, 0.02) if with_bias else None
    ref, S = oracle.addmm(b, x, np.ascontiguousarray(w.T), beta=1.0 if b is not None else 0.0,
                          alpha=1.0, self_2d=False)
    if relu:
        ref = np.maximum(ref, 0.0)
    for mode in MODES:
        out = binding.linear(dev(x), dev(w), dev(b), mode=mode, relu=relu)
        torch.cuda.synchronize()
        within(out.cpu().numpy(), ref, S, TOL[mode],
               f"linear {M}x({K}->{N}) bias={with_bias} relu={relu} {mode} "
               f"({binding.last_kernel_name()})")


def _offset(a):
    """a on the device one float past a 16-byte boundary (same values)."""
    a = np.ascontiguousarray(a)
    buf = torch.empty(a.size + 1, dtype=torch.float32, device="cuda")
    v = buf[1:].view(a.shape)
    v.copy_(torch.from_numpy(a))
    return v


@pytest.mark.parametrize("idx", range(0, len(ADDMM), 4))
def test_random_addmm_integer_and_unaligned(idx):
    # integer inputs: every product and partial sum is exact in fp32 and TF32,
    # so each path must match the oracle bit for bit; then the same with every
    # operand and the output one float off a 16-byte boundary
    M, N, K, s2, beta, alpha = ADDMM[idx]
    spec = ("I", -3, 3)
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=s2, workload=1300 + idx, mat1=spec, mat2=spec,
                                 self_=spec)
    beta, alpha = (1.0, 1.0) if beta != 0.0 else (0.0, 1.0)
    ref, _ = oracle.addmm(s, a, b, beta=beta, alpha=alpha)
    for mode in MODES + ["simt"]:
        got = binding.addmm(dev(s), dev(a), dev(b), beta=beta, alpha=alpha, mode=mode)
        assert np.array_equal(got.cpu().numpy().astype(np.float64), ref), \
            f"addmm {M}x{N}x{K} {mode} ({binding.last_kernel_name()})"
        out = _offset(np.zeros((M, N), np.float32))
        got = binding.addmm(_offset(s), _offset(a), _offset(b), beta=beta, alpha=alpha, mode=mode,
                            out=out)
        assert np.array_equal(got.cpu().numpy().astype(np.float64), ref), \
            f"unaligned addmm {M}x{N}x{K} {mode} ({binding.last_kernel_name()})"


@pytest.mark.parametrize("idx", range(0, len(CONV), 4))
def test_random_conv_integer_and_unaligned(idx):
    B, IC, H, W, OC, KH, KW, st, pd, dl = CONV[idx]
    spec = ("I", -3, 3)
    x, w, bias = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=1400 + idx, x=spec, w=spec,
                                   bias=spec)
    ref, _ = oracle.conv2d(x, w, bias, st, pd, dl)
    for mode in MODES + ["simt"]:
        got = binding.conv2d(dev(x), dev(w), dev(bias), st, pd, dl, mode=mode)
        assert np.array_equal(got.cpu().numpy().astype(np.float64), ref), \
            f"conv {CONV[idx]} {mode} ({binding.last_kernel_name()})"
        out = _offset(np.zeros(ref.shape, np.float32))
        got = binding.conv2d(_offset(x), _offset(w), _offset(bias), st, pd, dl, mode=mode, out=out)
        assert np.array_equal(got.cpu().numpy().astype(np.float64), ref), \
            f"unaligned conv {CONV[idx]} {mode} ({binding.last_kernel_name()})"


@pytest.mark.parametrize("idx", range(len(CONV_T)))
def test_random_conv_transposed_form(idx):
    B, IC, H, W, OC, KH, KW, st, pd, dl = CONV_T[idx]
    x, w, bias = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=1600 + idx)
    channels = np.arange(idx % min(5, OC), OC, 9)  # every 9th channel keeps the oracle quick
    ref, S = oracle.conv2d(x, w, bias, st, pd, dl, channels=channels)
    for mode in MODES:
        got = binding.conv2d(dev(x), dev(w), dev(bias), st, pd, dl, mode=mode).cpu().numpy()
        if binding.last_kernel() != "simt":  # the default mode takes SIMT for tiny problems
            assert binding.last_kernel_name().endswith(",slab_t>"), binding.last_kernel_name()
        within(got[:, channels], ref, S, TOL[mode], f"conv {CONV_T[idx]} {mode}")


@pytest.mark.parametrize("idx", range(0, len(LINEAR), 4))
def test_random_linear_unaligned(idx):
    M, N, K, with_bias, _ = LINEAR[idx]
    spec = ("I", -3, 3)
    from addmm_implicit_im2col_gb300.synth import _draw  # the seeded integer draws
    x = _draw(spec, synth.stream_key(0, 1500 + idx, 1), M * K).reshape(M, K)
    w = _draw(spec, synth.stream_key(0, 1500 + idx, 2), N * K).reshape(N, K)
    b = _draw(spec, synth.stream_key(0, 1500 + idx, 3), N) if with_bias else None
    ref, _ = oracle.addmm(b, x, np.ascontiguousarray(w.T), beta=1.0 if b is not None else 0.0,
                          alpha=1.0, self_2d=False)
    for mode in MODES + ["simt"]:
        out = _offset(np.zeros((M, N), np.float32))
        got = binding.linear(_offset(x), _offset(w), None if b is None else _offset(b), mode=mode,
                             out=out)
        assert np.array_equal(got.cpu().numpy().astype(np.float64), ref), \
            f"unaligned linear {M}x({K}->{N}) {mode} ({binding.last_kernel_name()})"


# Wide dynamic range: every operand +-10^e with e uniform in [-15, 15).  The
# bound as the other tests write it, 1e-5 * S with S = sum_k |a*b|, leaves out
# beta*self (the conv's bias): where that term is many orders larger than the
# products, rounding the result to fp32 alone exceeds 1e-5 * S, for SIMT FFMA
# as for any fp32 arithmetic.  These cases therefore measure the error
# against S' = |alpha| * S + |beta * self| (conv: S + |bias|), the magnitudes
# of every term of the expression (reading R18).
WIDE = ("L", -15.0, 15.0)


@pytest.mark.parametrize("idx", range(8))
def test_wide_dynamic_range_addmm(idx):
    rng = np.random.RandomState(300 + idx)
    M, N, K = int(rng.randint(1, 900)), int(rng.randint(1, 1500)), int(rng.randint(1, 900))
    s2 = bool(idx % 2)
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=s2, workload=1600 + idx, mat1=WIDE, mat2=WIDE,
                                 self_=WIDE)
    ref, S = oracle.addmm(s, a, b)
    Sx = S + np.abs(np.broadcast_to(s.astype(np.float64), ref.shape))
    for mode in MODES + ["simt"]:
        out = binding.addmm(dev(s), dev(a), dev(b), mode=mode)
        torch.cuda.synchronize()
        within(out.cpu().numpy(), ref, Sx, TOL[mode],
               f"wide-range addmm {M}x{N}x{K} {mode} ({binding.last_kernel_name()})")


@pytest.mark.parametrize("idx", range(8))
def test_wide_dynamic_range_conv(idx):
    rng = np.random.RandomState(400 + idx)
    IC, H, W = int(rng.randint(1, 40)), int(rng.randint(3, 60)), int(rng.randint(3, 90))
    OC = int(rng.randint(1, 200))
    x, w, bias = synth.conv_inputs(1, IC, H, W, OC, 3, 3, workload=1700 + idx, x=WIDE, w=WIDE,
                                   bias=WIDE)
    ref, S = oracle.conv2d(x, w, bias, 1, 1, 1)
    Sx = S + np.abs(bias.astype(np.float64))[None, :, None, None]
    for mode in MODES + ["simt"]:
        out = binding.conv2d(dev(x), dev(w), dev(bias), 1, 1, 1, mode=mode)
        torch.cuda.synchronize()
        within(out.cpu().numpy(), ref, Sx, TOL[mode],
               f"wide-range conv {IC}x{H}x{W}->{OC} {mode} ({binding.last_kernel_name()})")
