"""GPU parity: the CUDA path against the fp64 CPU oracle, element by element.

Bound (per element): |gpu - ref| <= c * S + 1e-6 with S = sum_k |a_ik * b_kj|
(conv: sum over in-range taps of |w * x|), c = 1e-5 for the default
(fp32-accurate) mode and the SIMT kernel, c = 2e-3 for the explicit 1xTF32
mode.  Integer-valued inputs (|v| <= 4) make every product and partial sum
exact in fp32 and TF32, so those cases must match bit for bit.

Every call goes through the C ABI (binding.py marshals torch tensors into it)
and the tests assert which kernel ran.
"""
import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

TOL = {"default": 1e-5, "simt": 1e-5, "force_tc3": 1e-5, "tf32": 2e-3, "force_tc1": 2e-3}


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    binding.load()
    yield
    assert binding.check_device_error(None) == binding.IMC_OK, "a kernel hit its wait limit"


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def within(got, ref, S, c, what=""):
    got = np.asarray(got, np.float64)
    err = np.abs(got - ref)
    tol = c * S + 1e-6
    ratio = float((err / tol).max()) if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert ratio <= 1.0, f"{what}: worst |err|/tol = {ratio:.3g}"
    return ratio


def run_addmm(s, a, b, beta, alpha, mode, rows=None):
    out = binding.addmm(dev(s), dev(a), dev(b), beta=beta, alpha=alpha, mode=mode)
    torch.cuda.synchronize()
    kern = binding.last_kernel()
    got = out.cpu().numpy()
    ref, S = oracle.addmm(s, a, b, beta=beta, alpha=alpha, rows=rows,
                          self_2d=(s is not None and s.ndim == 2))
    if rows is not None:
        got = got[rows]
    return got, ref, S, kern


EXPECT = {"simt": "simt", "force_tc3": "tc3", "force_tc1": "tc1"}

SMALL_ADDMM = [  # M, N, K: several tiles, ragged M / N / K tails
    (128, 128, 32), (1, 4, 4), (130, 132, 36), (300, 200, 100), (257, 516, 1028),
    (64, 80, 96), (384, 768, 64), (600, 260, 356),
]


@pytest.mark.parametrize("mode", ["simt", "force_tc3", "force_tc1"])
@pytest.mark.parametrize("mnk", SMALL_ADDMM, ids=lambda t: "x".join(map(str, t)))
def test_addmm_small(mode, mnk):
    M, N, K = mnk
    for self_2d, alpha, beta in [(False, 1.0, 1.0), (True, 2.0, 0.5), (True, -0.75, 1.25)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=1000 + M + N + K)
        got, ref, S, kern = run_addmm(s, a, b, beta, alpha, mode)
        assert kern == EXPECT[mode]
        within(got, ref, S, TOL[mode], f"{mode} {mnk} self_2d={self_2d}")


@pytest.mark.parametrize("mode", ["simt", "force_tc3", "force_tc1"])
@pytest.mark.parametrize("mnk", [(128, 128, 32), (200, 260, 132), (513, 1024, 2048)],
                         ids=lambda t: "x".join(map(str, t)))
def test_addmm_integer_inputs_are_bit_exact(mode, mnk):
    M, N, K = mnk
    spec = ("I", -4, 4)
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=True, workload=77, mat1=spec, mat2=spec,
                                 self_=spec)
    got, ref, _, kern = run_addmm(s, a, b, 1.0, 1.0, mode)
    assert kern == EXPECT[mode]
    assert np.array_equal(got.astype(np.float64), ref), f"max diff {np.abs(got - ref).max()}"


def test_addmm_long_k_tile_path():
    # 160 output tiles of 128 x 256 and 96 k-blocks of 16 per tile: the form of
    # the 3xTF32 kernel that keeps A in tensor memory and one accumulator; the
    # single-product modes run the shared-memory form on the same shape
    M, N, K = 2560, 2048, 1536
    rows = synth.sample_rows(synth.stream_key(0, 30, 9), M, 192)
    for self_2d, alpha, beta in [(False, 1.0, 1.0), (True, -0.5, 2.0)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=30 + self_2d,
                                     mat1=("N", 0.0, 1.0), mat2=("N", 0.0, 1.0 / np.sqrt(K)),
                                     self_=("N", 0.0, 1.0))
        for mode in ("default", "force_tc3", "tf32", "force_tc1"):
            got, ref, S, kern = run_addmm(s, a, b, beta, alpha, mode, rows=rows)
            assert kern == ("tc1" if mode in ("tf32", "force_tc1") else "tc3")
            within(got, ref, S, TOL[mode], f"long-K {mode} self_2d={self_2d}")
    spec = ("I", -2, 2)
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=True, workload=32, mat1=spec, mat2=spec,
                                 self_=spec)
    for mode in ("force_tc3", "force_tc1"):
        got, ref, _, _ = run_addmm(s, a, b, 1.0, 1.0, mode, rows=rows)
        assert np.array_equal(got.astype(np.float64), ref), mode


@pytest.mark.parametrize("mode", ["default", "tf32"])
def test_addmm_ragged_partial_last_wave(mode):
    # 160 to 180 output tiles on 152 SMs with ~96 k-blocks each (a short last
    # wave); ragged M, N and K; [M,N] self with negative alpha, and ReLU
    M, N, K = 2523, 1948, 1532
    rows = np.unique(np.concatenate([synth.sample_rows(synth.stream_key(0, 34, 9), M, 160),
                                     np.arange(M - 40, M)]))
    for self_2d, alpha, beta, relu in [(True, -0.5, 2.0, False), (False, 1.0, 1.0, True)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=34 + self_2d,
                                     mat1=("N", 0.0, 1.0), mat2=("N", 0.0, 1.0 / np.sqrt(K)),
                                     self_=("N", 0.0, 1.0))
        out = binding.addmm(dev(s), dev(a), dev(b), beta=beta, alpha=alpha, mode=mode,
                            relu=relu)
        torch.cuda.synchronize()
        assert binding.last_kernel() == ("tc3" if mode == "default" else "tc1")
        got = out.cpu().numpy()[rows]
        ref, S = oracle.addmm(s, a, b, beta=beta, alpha=alpha, rows=rows, self_2d=self_2d)
        if relu:
            ref = np.maximum(ref, 0.0)
        within(got, ref, S, TOL[mode], f"ragged last wave {mode} self_2d={self_2d} relu={relu}")
    spec = ("I", -2, 2)
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=True, workload=36, mat1=spec, mat2=spec,
                                 self_=spec)
    got, ref, _, _ = run_addmm(s, a, b, 1.0, 1.0, mode, rows=rows)
    assert np.array_equal(got.astype(np.float64), ref), mode


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
def test_addmm_k_not_multiple_of_4_on_tensor_cores(mode):
    # rows of K % 4 != 0 floats are not 16-byte aligned: mat1 is copied to
    # rows of K rounded up to 4 and mat2^T written with that row length; the
    # TMA reads zeros past K
    for M, N, K, self_2d in [(70, 40, 33, False), (5, 7, 3, True), (300, 260, 130, False),
                             (129, 65, 1, True), (256, 96, 2, False), (200, 300, 259, True)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=5 + K)
        # alpha = 1 for 1xTF32: with K of 1 to 3 nothing averages the product's
        # truncation error (up to 2^-9 of |a*b|), and the bound 2e-3*S does not
        # scale with alpha
        alpha = 1.5 if mode == "force_tc3" else 1.0
        got, ref, S, kern = run_addmm(s, a, b, 0.5, alpha, mode)
        assert kern == EXPECT[mode]
        within(got, ref, S, TOL[mode], f"{mode} {M}x{N}x{K}")
    spec = ("I", -4, 4)
    s, a, b = synth.addmm_inputs(300, 260, 130, self_2d=True, workload=7, mat1=spec, mat2=spec,
                                 self_=spec)
    got, ref, _, _ = run_addmm(s, a, b, 1.0, 1.0, mode)
    assert np.array_equal(got.astype(np.float64), ref)


def test_addmm_ragged_k_workloads():
    # the default mode takes the tensor cores for K % 4 != 0: a ragged
    # transformer-sized shape in full, and 8192x4096x4095 on 256 seeded rows
    M, N, K = 577, 770, 767
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=81, mat1=("N", 0.0, 1.0),
                                 mat2=("U", -1 / np.sqrt(K), 1 / np.sqrt(K)),
                                 self_=("N", 0.0, 0.02))
    for mode in ("default", "tf32"):
        got, ref, S, kern = run_addmm(s, a, b, 1.0, 1.0, mode)
        assert kern == ("tc3" if mode == "default" else "tc1")
        within(got, ref, S, TOL[mode], f"577x770x767 {mode}")
    M, N, K = 8192, 4096, 4095
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=82, mat1=("N", 0.0, 1 / 64),
                                 mat2=("N", 0.0, 1 / 64), self_=("N", 0.0, 1.0))
    rows = synth.sample_rows(synth.stream_key(0, 82, 99), M, 256)
    ref, S = oracle.addmm(s, a, b, rows=rows, self_2d=False)
    for mode in ("default", "tf32"):
        out = binding.addmm(dev(s), dev(a), dev(b), mode=mode)
        torch.cuda.synchronize()
        assert binding.last_kernel() == ("tc3" if mode == "default" else "tc1")
        within(out.cpu().numpy()[rows], ref, S, TOL[mode], f"8192x4096x4095 {mode}")
        del out


# Tile widths of 16 mod 32 (the planner takes them from 112 up when they fill
# the 152 SMs better): the last 32-column chunk of such a tile is half inside
# it, and neither epilogue may write the next tile's columns.  Plans (3xTF32):
# 1024x3072x768 -> BN 176, one wave of 144 tiles (A from TMEM, TMA-store
# epilogue; with an [M,N] self the shared-memory form and the generic store);
# 577x768x768 -> BN 112 in 4 K-slices; 600x3070x768 -> BN 112 with N % 4 != 0
# (generic store); 1100x2200x640 -> BN 144, ragged M and N.
HALF_CHUNK = [  # M, N, K, self_2d
    (1024, 3072, 768, False), (1024, 3072, 768, True), (577, 768, 768, False),
    (600, 3070, 768, False), (1100, 2200, 640, False),
]


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
@pytest.mark.parametrize("idx", range(len(HALF_CHUNK)))
def test_addmm_half_chunk_tile_widths(mode, idx):
    M, N, K, s2 = HALF_CHUNK[idx]
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=s2, workload=700 + idx)
    out = binding.addmm(dev(s), dev(a), dev(b), beta=0.75, alpha=1.25, mode=mode)
    torch.cuda.synchronize()
    assert binding.last_kernel() == EXPECT[mode]
    ref, S = oracle.addmm(s, a, b, beta=0.75, alpha=1.25)
    within(out.cpu().numpy(), ref, S, TOL[mode], f"{mode} {M}x{N}x{K} self_2d={s2}")
    if idx in (0, 3):  # integer inputs: bit-exact, and a ReLU on the way out
        si, ai, bi = synth.addmm_inputs(M, N, K, self_2d=s2, workload=720 + idx,
                                        mat1=("I", -3, 3), mat2=("I", -3, 3), self_=("I", -9, 9))
        got = binding.addmm(dev(si), dev(ai), dev(bi), mode=mode, relu=True).cpu().numpy()
        ref, _ = oracle.addmm(si, ai, bi)
        assert np.array_equal(got.astype(np.float64), np.maximum(ref, 0.0))


def test_addmm_unaligned_mat1():
    # mat1 starting 4 bytes past a 16-byte boundary: the library pool path
    # copies it to aligned rows (tensor cores); a caller workspace with room
    # for the mat2 copies alone (what an aligned mat1 needs at least) runs the
    # SIMT kernel
    M, N, K = 300, 260, 132
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=83)
    base = torch.zeros(M * K + 1, device="cuda")
    base[1:] = torch.from_numpy(a.ravel()).cuda()
    A = base[1:].view(M, K)
    assert A.data_ptr() % 16 == 4
    S, B = dev(s), dev(b)
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.empty((M, N), device="cuda")
    rc = binding.gemm_addmm_f32_ex(S.data_ptr(), 0, A.data_ptr(), B.data_ptr(), out.data_ptr(),
                                   M, N, K, 1.0, 1.0, 0, stream)
    assert rc == binding.IMC_OK and binding.last_kernel() == "tc3"
    torch.cuda.synchronize()
    ref, Sr = oracle.addmm(s, a, b)
    within(out.cpu().numpy(), ref, Sr, 1e-5, "unaligned mat1, pool")
    least = 2 * N * K * 4
    ws = torch.empty(least, dtype=torch.uint8, device="cuda")
    got = torch.empty((M, N), device="cuda")
    rc = binding.gemm_addmm_f32_ws(S.data_ptr(), 0, A.data_ptr(), B.data_ptr(), got.data_ptr(),
                                   M, N, K, 1.0, 1.0, 0, ws.data_ptr(), least, stream)
    assert rc == binding.IMC_OK and binding.last_kernel() == "simt"
    torch.cuda.synchronize()
    within(got.cpu().numpy(), ref, Sr, 1e-5, "unaligned mat1, small workspace")
    # with the size the query gives (room for split-K partial sums) it fits
    got = binding.addmm(S, A, B)
    torch.cuda.synchronize()
    assert binding.last_kernel() in ("tc3", "simt")
    within(got.cpu().numpy(), ref, Sr, 1e-5, "unaligned mat1, query-sized workspace")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
def test_addmm_odd_n_on_tensor_cores(mode):
    # mat2 is transposed by the pre-pass, so N needs no alignment
    for M, N, K, self_2d in [(70, 33, 40, False), (300, 257, 132, True), (129, 1, 64, True)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=6)
        got, ref, S, kern = run_addmm(s, a, b, 0.5, 1.5, mode)
        assert kern == EXPECT[mode]
        within(got, ref, S, TOL[mode], f"{mode} {M}x{N}x{K}")


def test_addmm_workspace_paths_agree():
    """The pool-backed entry point and the caller-workspace entry point run the
    same kernels: identical bits."""
    M, N, K = 600, 520, 388
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=True, workload=8)
    S, A, B = dev(s), dev(a), dev(b)
    stream = torch.cuda.current_stream().cuda_stream
    for mode in (0, 1, 3):
        o1 = torch.empty((M, N), device="cuda")
        o2 = torch.empty((M, N), device="cuda")
        rc = binding.gemm_addmm_f32_ex(S.data_ptr(), 1, A.data_ptr(), B.data_ptr(), o1.data_ptr(),
                                       M, N, K, 0.25, 1.5, mode, stream)
        assert rc == 0
        nbytes = binding.gemm_addmm_f32_workspace_bytes(M, N, K, mode)
        assert nbytes > 0
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        rc = binding.gemm_addmm_f32_ws(S.data_ptr(), 1, A.data_ptr(), B.data_ptr(), o2.data_ptr(),
                                       M, N, K, 0.25, 1.5, mode, ws.data_ptr(), nbytes, stream)
        assert rc == 0
        torch.cuda.synchronize()
        assert torch.equal(o1, o2)
        ref, Sref = oracle.addmm(s, a, b, beta=0.25, alpha=1.5)
        within(o1.cpu().numpy(), ref, Sref, 1e-5 if mode != 1 else 2e-3, f"mode {mode}")


@pytest.mark.parametrize("mode", ["default", "simt", "force_tc3"])
def test_addmm_special_cases(mode):
    M, N, K = 256, 132, 64
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=True, workload=9)
    # alpha == 0: out = beta*self, operands never read (NaN there is harmless)
    a_nan = a.copy()
    a_nan[3, 5] = np.nan
    out = binding.addmm(dev(s), dev(a_nan), dev(b), beta=1.5, alpha=0.0, mode=mode)
    assert binding.last_kernel() == "fill"
    assert np.array_equal(out.cpu().numpy(), (np.float32(1.5) * s))
    # beta == 0: self never read
    s_nan = np.full_like(s, np.nan)
    got = binding.addmm(dev(s_nan), dev(a), dev(b), beta=0.0, alpha=2.0, mode=mode).cpu().numpy()
    ref, S = oracle.addmm(None, a, b, beta=0.0, alpha=2.0)
    within(got, ref, S, 1e-5, "beta=0")
    # identity mat2 returns alpha*mat1 + beta*self
    eye = np.eye(K, dtype=np.float32)
    s2 = synth.uniform(synth.stream_key(0, 9, 5), M * K, -1, 1).reshape(M, K)
    got = binding.addmm(dev(s2), dev(a), dev(eye), beta=0.5, alpha=1.0, mode=mode).cpu().numpy()
    ref, S = oracle.addmm(s2, a, eye, beta=0.5, alpha=1.0)
    within(got, ref, S, 1e-5, "identity")
    # K == 0: empty sum
    z = binding.addmm(dev(s), torch.empty((M, 0), device="cuda"), torch.empty((0, N), device="cuda"),
                      beta=2.0, alpha=1.0, mode=mode)
    assert np.array_equal(z.cpu().numpy(), np.float32(2.0) * s)
    # in-place: out is self
    st = dev(s)
    binding.addmm(st, dev(a), dev(b), beta=1.0, alpha=1.0, mode=mode, out=st)
    ref, S = oracle.addmm(s, a, b)
    within(st.cpu().numpy(), ref, S, 1e-5, "in-place")


def test_self_broadcast_equals_full_self():
    M, N, K = 300, 260, 128
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=21)
    for mode in ("simt", "force_tc3"):
        r1 = binding.addmm(dev(s), dev(a), dev(b), beta=0.5, alpha=1.5, mode=mode)
        r2 = binding.addmm(dev(np.tile(s, (M, 1))), dev(a), dev(b), beta=0.5, alpha=1.5, mode=mode)
        assert torch.equal(r1, r2)


@pytest.mark.parametrize("name", [n for n in synth.ADDMM_CASES if "rows" not in
                                  synth.ADDMM_CASES[n]])
def test_addmm_workloads(name):
    c, s, a, b = synth.make_addmm_case(name)
    rows = synth.checked_rows(name, c["M"], 256) if c["M"] > 256 else None
    for mode in ("default", "tf32"):
        got, ref, S, kern = run_addmm(s, a, b, c["beta"], c["alpha"], mode, rows=rows)
        within(got, ref, S, TOL[mode], f"{name} {mode} ({kern})")


@pytest.mark.parametrize("name", [n for n in synth.ADDMM_CASES if "rows" in
                                  synth.ADDMM_CASES[n]])
def test_addmm_large_workloads_sampled_rows(name):
    c, s, a, b = synth.make_addmm_case(name)
    rows = synth.checked_rows(name, c["M"], c["rows"])
    ref, S = oracle.addmm(s, a, b, beta=c["beta"], alpha=c["alpha"], rows=rows,
                          self_2d=c["self_2d"])
    for mode in ("default", "tf32"):
        out = binding.addmm(dev(s), dev(a), dev(b), beta=c["beta"], alpha=c["alpha"], mode=mode)
        torch.cuda.synchronize()
        assert binding.last_kernel() == ("tc3" if mode == "default" else "tc1")
        within(out.cpu().numpy()[rows], ref, S, TOL[mode], f"{name} {mode}")
        del out


def test_exact_boundary_signatures():
    """gemm_addmm_f32 and conv2d_gemm_f32 exactly as declared (default mode,
    scratch from the library's stream-ordered pool), against the oracle."""
    stream = torch.cuda.current_stream().cuda_stream
    for M, N, K, self_2d, beta, alpha in [(600, 520, 388, 1, 0.5, 1.5),
                                          (1000, 2304, 768, 0, 1.0, 1.0)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=bool(self_2d), workload=90 + M)
        S, A, B = dev(s), dev(a), dev(b)
        out = torch.full((M, N), float("nan"), device="cuda")
        rc = binding.gemm_addmm_f32(S.data_ptr(), self_2d, A.data_ptr(), B.data_ptr(),
                                    out.data_ptr(), M, N, K, beta, alpha, stream)
        assert rc == binding.IMC_OK, binding.status_string(rc)
        assert binding.last_kernel() == "tc3"
        torch.cuda.synchronize()
        ref, Sr = oracle.addmm(s, a, b, beta=beta, alpha=alpha)
        within(out.cpu().numpy(), ref, Sr, 1e-5, f"gemm_addmm_f32 {M}x{N}x{K}")
    for (Bn, IC, H, W, OC, KH, KW, st, pd, dl) in [(2, 16, 40, 40, 130, 3, 3, 2, 1, 1),
                                                   (1, 3, 96, 96, 128, 7, 7, 4, 3, 1)]:
        x, w, bias = synth.conv_inputs(Bn, IC, H, W, OC, KH, KW, workload=95 + IC)
        X, Wt, Bias = dev(x), dev(w), dev(bias)
        OH = (H + 2 * pd - dl * (KH - 1) - 1) // st + 1
        OW = (W + 2 * pd - dl * (KW - 1) - 1) // st + 1
        y = torch.full((Bn, OC, OH, OW), float("nan"), device="cuda")
        rc = binding.conv2d_gemm_f32(X.data_ptr(), Wt.data_ptr(), Bias.data_ptr(), y.data_ptr(),
                                     Bn, IC, H, W, OC, KH, KW, st, pd, dl, stream)
        assert rc == binding.IMC_OK, binding.status_string(rc)
        assert binding.last_kernel() == "tc3"
        torch.cuda.synchronize()
        ref, Sr = oracle.conv2d(x, w, bias, st, pd, dl)
        within(y.cpu().numpy(), ref, Sr, 1e-5, f"conv2d_gemm_f32 {Bn}x{IC}x{H}x{W}->{OC}")


# ------------------------------------------------------------------- conv
def run_conv(x, w, bias, stride, pad, dil, mode, channels=None):
    out = binding.conv2d(dev(x), dev(w), dev(bias), stride, pad, dil, mode=mode)
    torch.cuda.synchronize()
    kern = binding.last_kernel()
    got = out.cpu().numpy()
    ref, S = oracle.conv2d(x, w, bias, stride, pad, dil, channels=channels)
    if channels is not None:
        got = got[:, channels]
    return got, ref, S, kern


SMALL_CONV = [  # B, IC, H, W, OC, KH, KW, stride, pad, dil
    (2, 3, 9, 9, 4, 3, 3, 1, 1, 1),
    (1, 3, 64, 64, 128, 7, 7, 4, 3, 1),
    (2, 16, 20, 20, 130, 3, 3, 1, 1, 1),
    (2, 32, 14, 14, 64, 3, 3, 1, 2, 2),
    (3, 8, 17, 13, 200, 5, 3, 2, 1, 1),
    (1, 5, 12, 40, 36, 3, 2, (2, 3), (1, 0), (1, 2)),
    (2, 64, 9, 9, 32, 1, 1, 1, 0, 1),
    # channel-fastest K order with IC not a multiple of 16 (per-element tap steps)
    (2, 9, 11, 13, 40, 3, 3, 1, 1, 1),
    (2, 12, 15, 9, 70, 3, 5, (1, 2), (1, 2), (2, 1)),
]


def _conv_case(t, workload, spec=None):
    B, IC, H, W, OC, KH, KW = t[:7]
    kw = {} if spec is None else dict(x=spec, w=spec, bias=spec)
    x, w, b = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=workload, **kw)
    return x, w, b, t[7], t[8], t[9]


@pytest.mark.parametrize("mode", ["simt", "force_tc3", "force_tc1"])
@pytest.mark.parametrize("idx", range(len(SMALL_CONV)))
def test_conv_small(mode, idx):
    x, w, b, s, p, d = _conv_case(SMALL_CONV[idx], 300 + idx)
    got, ref, S, kern = run_conv(x, w, b, s, p, d, mode)
    assert kern == EXPECT[mode]
    within(got, ref, S, TOL[mode], f"{mode} conv #{idx}")
    # and without bias
    got, ref, S, _ = run_conv(x, w, None, s, p, d, mode)
    within(got, ref, S, TOL[mode], f"{mode} conv #{idx} no bias")


@pytest.mark.parametrize("mode", ["simt", "force_tc3", "force_tc1"])
@pytest.mark.parametrize("idx", [0, 1, 3, 5, 7, 8])
def test_conv_integer_inputs_are_bit_exact(mode, idx):
    x, w, b, s, p, d = _conv_case(SMALL_CONV[idx], 400 + idx, spec=("I", -4, 4))
    got, ref, _, kern = run_conv(x, w, b, s, p, d, mode)
    assert kern == EXPECT[mode]
    assert np.array_equal(got.astype(np.float64), ref)


# Shapes that steer the tensor-core conv's work split (128-position x BN-channel
# tiles on 152 SMs; the last wave's tiles cut into K-slices whose partial sums
# a second kernel adds):
SCHED_CONV = [  # B, IC, H, W, OC, KH, KW, stride, pad, dil, channels checked (None: all)
    # 160 tiles: one whole wave, then 8 tiles in 9 K-slices (BN 256, one accumulator)
    (5, 64, 64, 64, 256, 3, 3, 1, 1, 1, np.arange(0, 256, 9)),
    # OC 320: two channel tiles of 160; 14 tiles, all K-sliced
    (2, 32, 20, 20, 320, 3, 3, 1, 1, 1, None),
    # 11x11 taps, stride 4
    (1, 3, 67, 67, 64, 11, 11, 4, 2, 1, None),
    # K = 9 < one k-block of 16; BN 16
    (2, 1, 30, 30, 16, 3, 3, 1, 1, 1, None),
    # dilation 4 with padding 4, 48 channels
    (1, 4, 30, 30, 48, 3, 3, 1, 4, 4, None),
    # 1x1, K = 520 (not a multiple of 16), 290 tiles: two waves, two accumulators
    (2, 520, 136, 136, 96, 1, 1, 1, 0, 1, np.arange(0, 96, 5)),
    # 5x5 stride 2, tiles running into the next image
    (3, 24, 40, 40, 96, 5, 5, 2, 2, 1, None),
    # dilation 2 with padding 2
    (2, 16, 32, 32, 64, 3, 3, 1, 2, 2, None),
    # 1000 positions per image in 8 tiles each, the last one short; 24 tiles, K-sliced
    (3, 32, 40, 25, 64, 3, 3, 1, 1, 1, None),
]


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1", "default"])
@pytest.mark.parametrize("idx", range(len(SCHED_CONV)))
def test_conv_work_split(mode, idx):
    t = SCHED_CONV[idx]
    x, w, b, s, p, d = _conv_case(t[:10], 320 + idx)
    got, ref, S, kern = run_conv(x, w, b, s, p, d, mode, channels=t[10])
    if mode in EXPECT:
        assert kern == EXPECT[mode]
    within(got, ref, S, TOL[mode], f"{mode} sched conv #{idx}")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
@pytest.mark.parametrize("idx", [0, 1, 5])
def test_conv_work_split_integer_bit_exact(mode, idx):
    t = SCHED_CONV[idx]
    x, w, b, s, p, d = _conv_case(t[:10], 420 + idx, spec=("I", -2, 2))
    got, ref, _, kern = run_conv(x, w, b, s, p, d, mode, channels=t[10])
    assert kern == EXPECT[mode]
    assert np.array_equal(got.astype(np.float64), ref)


def test_conv_1x1_matches_addmm_path():
    B, IC, H, W, OC = 2, 64, 16, 16, 128
    x, w, b = synth.conv_inputs(B, IC, H, W, OC, 1, 1, workload=55)
    conv = binding.conv2d(dev(x), dev(w), dev(b), mode="force_tc3").cpu().numpy()
    for bi in range(B):
        bias2d = np.repeat(b[:, None], H * W, axis=1).astype(np.float32)
        mm = binding.addmm(dev(bias2d), dev(w.reshape(OC, IC)), dev(x[bi].reshape(IC, H * W)),
                           mode="force_tc3").cpu().numpy()
        ref, S = oracle.addmm(bias2d, w.reshape(OC, IC), x[bi].reshape(IC, H * W))
        within(mm, ref, S, 1e-5, "1x1 via addmm")
        within(conv[bi].reshape(OC, H * W), ref, S, 1e-5, "1x1 via conv")


def test_conv_empty_channels_and_bias_only():
    x = dev(np.ones((0, 3, 8, 8), np.float32))
    w = dev(np.ones((4, 3, 3, 3), np.float32))
    out = binding.conv2d(x, w, None, 1, 1, 1)
    assert out.shape == (0, 4, 8, 8)
    xz = dev(np.ones((2, 0, 8, 8), np.float32))
    wz = dev(np.ones((4, 0, 3, 3), np.float32))
    bias = dev(np.array([1, 2, 3, 4], np.float32))
    out = binding.conv2d(xz, wz, bias, 1, 1, 1).cpu().numpy()
    assert binding.last_kernel() == "fill"
    assert np.array_equal(out, np.broadcast_to(np.array([1, 2, 3, 4], np.float32)[None, :, None,
                                                                                  None], out.shape))


@pytest.mark.parametrize("name", list(synth.CONV_CASES))
def test_conv_workloads(name):
    c, x, w, b = synth.make_conv_case(name)
    for mode in ("default", "tf32"):
        got, ref, S, kern = run_conv(x, w, b, c["stride"], c["pad"], c["dilation"], mode)
        assert kern == ("tc3" if mode == "default" else "tc1")
        assert binding.last_kernel_name().startswith("k_tc_conv<"), binding.last_kernel_name()
        within(got, ref, S, TOL[mode], f"{name} {mode}")


# Few input channels (IC < 8) with W % 4 == 0 and OW % 4 == 0: the slab form
# (position tiles of 4 output rows x 32 output columns; each tile's input
# window comes into shared memory by one TMA box, the im2col values are read
# from there; whole tiles leave by 4-D TMA stores clipped at the image edges).
SLAB_CONV = [  # B, IC, H, W, OC, KH, KW, stride, pad, dil, channels checked (None: all)
    # ragged right and bottom edges (OW 120 = 3.75 column tiles, OH 102), pad 1
    (2, 3, 102, 120, 64, 3, 3, 1, 1, 1, None),
    # pad 0 (box starts on the window), 5x5
    (1, 4, 40, 68, 32, 5, 5, 1, 0, 1, None),
    # stride 2, dilation 2, pad 2, OH 33
    (2, 2, 66, 128, 48, 3, 3, 2, 2, 2, None),
    # per-axis stride / pad / dilation, OH 29
    (2, 5, 31, 64, 40, 3, 5, (1, 2), (1, 2), (2, 1), None),
    # 160 tiles: one wave, then 8 tiles in K-slices (K = 343)
    (1, 7, 80, 256, 32, 7, 7, 1, 3, 1, None),
    # K = 9: one k-block per tile, so one warp group gathers nothing
    (2, 1, 64, 64, 16, 3, 3, 1, 1, 1, None),
    # OC 300: two channel tiles of 160, stride 2
    (1, 3, 64, 128, 300, 5, 5, 2, 2, 1, np.arange(0, 300, 7)),
    # the stem shape at 96x96: OW = OH = 24, three quarters of each tile used
    (1, 3, 96, 96, 128, 7, 7, 4, 3, 1, None),
]


def _slab_form(name):
    """Either slab form: 128-position tiles (",slab>") or the transposed form
    with 256-position tiles and the channels as M (",slab_t>")."""
    return name.endswith(",slab>") or name.endswith(",slab_t>")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1", "default"])
@pytest.mark.parametrize("idx", range(len(SLAB_CONV)))
def test_conv_slab_form(mode, idx):
    t = SLAB_CONV[idx]
    x, w, b, s, p, d = _conv_case(t[:10], 520 + idx)
    got, ref, S, kern = run_conv(x, w, b, s, p, d, mode, channels=t[10])
    if mode in EXPECT:
        assert kern == EXPECT[mode]
    if kern != "simt":  # the default mode may take SIMT for the smallest shapes
        assert _slab_form(binding.last_kernel_name()), binding.last_kernel_name()
    within(got, ref, S, TOL[mode], f"{mode} slab conv #{idx}")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
@pytest.mark.parametrize("idx", [0, 3, 4, 6])
def test_conv_slab_integer_bit_exact(mode, idx):
    t = SLAB_CONV[idx]
    x, w, b, s, p, d = _conv_case(t[:10], 540 + idx, spec=("I", -3, 3))
    got, ref, _, _ = run_conv(x, w, b, s, p, d, mode, channels=t[10])
    assert _slab_form(binding.last_kernel_name()), binding.last_kernel_name()
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
def test_conv_slab_relu_no_bias(mode):
    t = SLAB_CONV[0]
    x, w, _, s, p, d = _conv_case(t[:10], 560)
    out = binding.conv2d(dev(x), dev(w), None, s, p, d, mode=mode, relu=True)
    torch.cuda.synchronize()
    assert _slab_form(binding.last_kernel_name()), binding.last_kernel_name()
    ref, S = oracle.conv2d(x, w, None, s, p, d)
    within(out.cpu().numpy(), np.maximum(ref, 0.0), S, TOL[mode], f"slab relu {mode}")


def test_conv_slab_reads_only_the_taps():
    # 2x2 taps at stride 4: input columns 4j+2 and 4j+3 belong to no output's
    # window.  The slab holds them; a NaN there must not reach any output.
    B, IC, H, W, OC = 1, 3, 32, 128, 24
    x, w, b = synth.conv_inputs(B, IC, H, W, OC, 2, 2, workload=561)
    x = x.copy()
    x[:, :, :, 2::4] = np.nan
    x[:, :, :, 3::4] = np.inf
    got, ref, S, _ = run_conv(x, w, b, 4, 0, 1, "force_tc3")
    assert _slab_form(binding.last_kernel_name()), binding.last_kernel_name()
    assert np.isfinite(ref).all()
    within(got, ref, S, 1e-5, "slab conv, NaN outside the taps")


# The transposed slab form (OC <= 128, one 256-position tile of 8 output rows x
# 32 columns per SM at most): channels are the MMA's M, positions its N.
SLAB_T_CONV = [  # B, IC, H, W, OC, KH, KW, stride, pad, dil, channels checked (None: all)
    # the stem: 3 -> 128 channels, 768x768, 7x7 stride 4 (144 tiles)
    (1, 3, 768, 768, 128, 7, 7, 4, 3, 1, np.arange(0, 128, 9)),
    # ragged: OH 50 (7 row tiles, the last 2 rows used), OW 108 (4 column tiles), OC 40; 140 tiles
    (5, 3, 100, 216, 40, 5, 5, 2, 2, 1, None),
    # 3x3 stride 1, OC 128, 128 tiles
    (8, 3, 64, 64, 128, 3, 3, 1, 1, 1, np.arange(0, 128, 3)),
    # K = 9: a single k-block; 144 tiles
    (6, 1, 64, 96, 64, 3, 3, 1, 1, 1, None),
    # per-axis stride / pad / dilation, OH 38, OW 32; 120 tiles
    (24, 5, 40, 64, 24, 3, 5, (1, 2), (1, 2), (2, 1), None),
    # K = 343: 22 k-blocks through 3 or 7 stages; 120 tiles
    (5, 7, 48, 128, 64, 7, 7, 1, 3, 1, np.arange(0, 64, 5)),
]

# Slab-form shapes past the transposed form's reach: more tiles than SMs, fewer
# than 3/4 of them, or OC > 128.
SLAB_WIDE_CONV = [
    (4, 3, 256, 256, 64, 7, 7, 2, 3, 1, np.arange(0, 64, 5)),  # 256 tiles of 256 positions
    (1, 3, 256, 256, 64, 7, 7, 2, 3, 1, None),                  # 64 tiles
    (1, 3, 64, 128, 160, 5, 5, 2, 2, 1, None),                  # OC 160
]


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1", "default"])
@pytest.mark.parametrize("idx", range(len(SLAB_T_CONV)))
def test_conv_slab_transposed_form(mode, idx):
    t = SLAB_T_CONV[idx]
    x, w, b, s, p, d = _conv_case(t[:10], 570 + idx)
    got, ref, S, kern = run_conv(x, w, b, s, p, d, mode, channels=t[10])
    if mode in EXPECT:
        assert kern == EXPECT[mode]
    if kern != "simt":
        assert binding.last_kernel_name().endswith(",slab_t>"), binding.last_kernel_name()
    within(got, ref, S, TOL[mode], f"{mode} transposed slab conv #{idx}")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
@pytest.mark.parametrize("idx", range(len(SLAB_WIDE_CONV)))
def test_conv_slab_form_past_the_transposed_reach(mode, idx):
    t = SLAB_WIDE_CONV[idx]
    x, w, b, s, p, d = _conv_case(t[:10], 580 + idx)
    got, ref, S, _ = run_conv(x, w, b, s, p, d, mode, channels=t[10])
    assert binding.last_kernel_name().endswith(",slab>"), binding.last_kernel_name()
    within(got, ref, S, TOL[mode], f"{mode} slab conv (wide) #{idx}")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
@pytest.mark.parametrize("idx", [1, 3, 4, 5])
def test_conv_slab_transposed_integer_bit_exact(mode, idx):
    t = SLAB_T_CONV[idx]
    x, w, b, s, p, d = _conv_case(t[:10], 590 + idx, spec=("I", -3, 3))
    got, ref, _, _ = run_conv(x, w, b, s, p, d, mode, channels=t[10])
    assert binding.last_kernel_name().endswith(",slab_t>")
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
def test_conv_slab_transposed_relu_no_bias(mode):
    t = SLAB_T_CONV[1]
    x, w, _, s, p, d = _conv_case(t[:10], 596)
    out = binding.conv2d(dev(x), dev(w), None, s, p, d, mode=mode, relu=True)
    torch.cuda.synchronize()
    assert binding.last_kernel_name().endswith(",slab_t>")
    ref, S = oracle.conv2d(x, w, None, s, p, d)
    within(out.cpu().numpy(), np.maximum(ref, 0.0), S, TOL[mode], f"transposed slab relu {mode}")


def test_conv_slab_shape_with_unaligned_input_takes_the_global_gather():
    # same shape as a slab case, x one float off a 16-byte boundary: no TMA
    # box can start there, so the gather reads global memory instead
    t = SLAB_CONV[0]
    x, w, b, s, p, d = _conv_case(t[:10], 562)
    buf = torch.empty(x.size + 1, dtype=torch.float32, device="cuda")
    xv = buf[1:].view(x.shape)
    xv.copy_(torch.from_numpy(x))
    assert xv.data_ptr() % 16 != 0
    out = binding.conv2d(xv, dev(w), dev(b), s, p, d, mode="force_tc3")
    torch.cuda.synchronize()
    assert binding.last_kernel_name() == "k_tc_conv<3xtf32>"
    ref, S = oracle.conv2d(x, w, b, s, p, d)
    within(out.cpu().numpy(), ref, S, 1e-5, "unaligned x")


# OC > 256 in two channel tiles whose even split is 16 mod 32 wide (275 ->
# 138): the tiles are widened to 160 so that no 32-channel output block of one
# tile reaches into the next; global gather and slab form, both epilogues
# (whole tiles by TMA store, K-slice partial sums).
@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1"])
@pytest.mark.parametrize("shape", [
    (1, 21, 6, 71, 275, 1, 6, (3, 2), (2, 2), (2, 2)),   # channel-fastest gather
    (1, 3, 64, 128, 275, 3, 3, 1, 1, 1),                # slab form
    (2, 40, 30, 30, 300, 3, 3, 1, 1, 1),                # K-sliced tail tiles
])
def test_conv_several_channel_tiles(mode, shape):
    x, w, b, s, p, d = _conv_case(shape, 580 + shape[4] + shape[1])
    got, ref, S, kern = run_conv(x, w, b, s, p, d, mode)
    assert kern == EXPECT[mode]
    within(got, ref, S, TOL[mode], f"{mode} conv {shape}")


def test_launch_counter_and_watchdog():
    n0 = binding.launch_count()
    s, a, b = synth.addmm_inputs(256, 256, 64, self_2d=False, workload=3)
    binding.addmm(dev(s), dev(a), dev(b), mode="force_tc3")  # mat2 pre-pass + main kernel
    binding.addmm(dev(s), dev(a), dev(b), mode="simt")
    torch.cuda.synchronize()
    assert binding.launch_count() == n0 + 3
    assert binding.check_device_error(None) == binding.IMC_OK


def test_calls_captured_in_a_cuda_graph():
    # the device entry points enqueue only stream-ordered work (scratch from the
    # caller, launches with programmatic-dependent-launch edges), so a graph
    # captured once replays them on new inputs written into the same buffers
    M, N, K = 640, 768, 512
    s0, a0, b0 = synth.addmm_inputs(M, N, K, self_2d=False, workload=60)
    x0, w0, bias0 = synth.conv_inputs(2, 32, 20, 20, 96, 3, 3, workload=61)
    S, A, B = dev(s0), dev(a0), dev(b0)
    X, W, Bias = dev(x0), dev(w0), dev(bias0)
    binding.addmm(S, A, B)  # first calls set per-device attributes outside the capture
    binding.conv2d(X, W, Bias, 1, 1, 1)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = binding.addmm(S, A, B, beta=0.5, alpha=2.0)
        y = binding.conv2d(X, W, Bias, 1, 1, 1)
    for rep in range(3):
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=62 + rep)
        x, w, bias = synth.conv_inputs(2, 32, 20, 20, 96, 3, 3, workload=65 + rep)
        for t, v in ((S, s), (A, a), (B, b), (X, x), (W, w), (Bias, bias)):
            t.copy_(torch.from_numpy(v))
        graph.replay()
        torch.cuda.synchronize()
        ref, Sa = oracle.addmm(s, a, b, beta=0.5, alpha=2.0, self_2d=False)
        within(out.cpu().numpy(), ref, Sa, 1e-5, f"graph replay {rep} addmm")
        ref, Sc = oracle.conv2d(x, w, bias, 1, 1, 1)
        within(y.cpu().numpy(), ref, Sc, 1e-5, f"graph replay {rep} conv")


def test_stem_like_conv_captured_in_a_cuda_graph():
    # the transposed slab form (input window by TMA, output by TMA boxes) replayed
    # from a graph on new inputs, beside a slab-form conv past its reach
    shapes = [(3, 3, 320, 512, 32, 7, 7, 4, 3, 1), (2, 3, 64, 128, 160, 5, 5, 2, 2, 1)]
    bufs, outs = [], []
    for i, (B_, IC, H, W, OC, KH, KW, st, pd, dl) in enumerate(shapes):
        x0, w0, b0 = synth.conv_inputs(B_, IC, H, W, OC, KH, KW, workload=600 + i)
        bufs.append((dev(x0), dev(w0), dev(b0)))
        binding.conv2d(*bufs[-1], st, pd, dl)  # attributes set outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for (X, W, Bias), t in zip(bufs, shapes):
            outs.append(binding.conv2d(X, W, Bias, t[7], t[8], t[9]))
    for rep in range(2):
        new = []
        for i, ((X, W, Bias), t) in enumerate(zip(bufs, shapes)):
            x, w, b = synth.conv_inputs(*t[:7], workload=610 + 2 * i + rep)
            for dst, v in ((X, x), (W, w), (Bias, b)):
                dst.copy_(torch.from_numpy(v))
            new.append((x, w, b))
        graph.replay()
        torch.cuda.synchronize()
        for (x, w, b), t, y in zip(new, shapes, outs):
            ref, S = oracle.conv2d(x, w, b, t[7], t[8], t[9])
            within(y.cpu().numpy(), ref, S, 1e-5, f"graph replay {rep} conv {t}")
    # the two shapes take the two slab forms
    binding.conv2d(*bufs[0], 4, 3, 1)
    assert binding.last_kernel_name().endswith(",slab_t>"), binding.last_kernel_name()
    binding.conv2d(*bufs[1], 2, 2, 1)
    assert binding.last_kernel_name().endswith(",slab>"), binding.last_kernel_name()


def test_a_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    # failure path of the bounded barrier waits, without a fault: a kernel
    # waits on a barrier nothing completes, gives up after 20 ms, and the host
    # reads IMC_ERR_TIMEOUT; afterwards the library works as before
    assert binding.check_device_error(None) == binding.IMC_OK
    assert binding.selftest_wait_timeout(20000) == binding.IMC_OK
    assert binding.check_device_error(None) == binding.IMC_ERR_TIMEOUT
    assert binding.check_device_error(None) == binding.IMC_OK  # read and cleared
    s, a, b = synth.addmm_inputs(300, 260, 132, self_2d=True, workload=70)
    got, ref, S, kern = run_addmm(s, a, b, 0.5, 1.5, "default")
    assert kern == "tc3"
    within(got, ref, S, 1e-5, "after a timeout")


def test_pool_backed_calls_on_four_streams():
    """The exact boundary signatures take their scratch from the library's
    stream-ordered pool: calls interleaved on four streams (each call's scratch
    freed on its own stream while other streams keep allocating) must each give
    their own oracle result."""
    streams = [torch.cuda.Stream() for _ in range(4)]
    jobs = []
    for i in range(12):
        M, N, K = 300 + 37 * i, 520 + 24 * (i % 5), 388 + 16 * (i % 3)
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=bool(i % 2), workload=760 + i)
        jobs.append(("addmm", (s, a, b), [dev(s), dev(a), dev(b)], (M, N, K, i % 2)))
    for i in range(8):
        shape = (2, 16 + 8 * (i % 3), 24, 24, 96 + 32 * (i % 4), 3, 3)
        x, w, bias = synth.conv_inputs(*shape, workload=780 + i)
        jobs.append(("conv", (x, w, bias), [dev(x), dev(w), dev(bias)], shape))
    outs = []
    for j, (kind, host, devs, dims) in enumerate(jobs):
        st = streams[j % 4]
        st.wait_stream(torch.cuda.current_stream())  # the inputs were written on it
        with torch.cuda.stream(st):
            if kind == "addmm":
                M, N, K, s2 = dims
                out = torch.full((M, N), float("nan"), device="cuda")
                rc = binding.gemm_addmm_f32(devs[0].data_ptr(), s2, devs[1].data_ptr(),
                                            devs[2].data_ptr(), out.data_ptr(), M, N, K, 1.0, 1.0,
                                            st.cuda_stream)
            else:
                B, IC, H, W, OC, KH, KW = dims
                out = torch.full((B, OC, H, W), float("nan"), device="cuda")
                rc = binding.conv2d_gemm_f32(devs[0].data_ptr(), devs[1].data_ptr(),
                                             devs[2].data_ptr(), out.data_ptr(), B, IC, H, W, OC,
                                             KH, KW, 1, 1, 1, st.cuda_stream)
            assert rc == binding.IMC_OK, binding.status_string(rc)
            for t in devs:
                t.record_stream(st)
        outs.append(out)
    torch.cuda.synchronize()
    for (kind, host, _, dims), out in zip(jobs, outs):
        if kind == "addmm":
            ref, S = oracle.addmm(*host)
        else:
            ref, S = oracle.conv2d(host[0], host[1], host[2], 1, 1, 1)
        within(out.cpu().numpy(), ref, S, 1e-5, f"{kind} {dims} on a side stream")
    assert binding.check_device_error(None) == binding.IMC_OK


def _plant_non_finite(a, spots):
    """a with the given (index, kind) entries replaced: kind 'inf', '-inf',
    'nan' (canonical quiet NaN) or 'nan_low' (a NaN whose payload lies only in
    the 13 low mantissa bits, which a TF32 truncation would clear)."""
    a = a.copy()
    bits = a.view(np.uint32)
    for idx, kind in spots:
        if kind == "nan_low":
            bits[idx] = np.uint32(0x7F800001)
        else:
            a[idx] = {"inf": np.inf, "-inf": -np.inf, "nan": np.nan}[kind]
    return a


def _same_non_finite(got, ref, S, tol, mode, what):
    """The contract for non-finite inputs (imc.h): SIMT follows IEEE
    arithmetic, so its NaN / +inf / -inf pattern equals the reference's.  On
    the tensor cores an output the reference has as NaN is non-finite (a NaN
    whose payload lies only in the 13 low mantissa bits reads as an infinity
    there), one it has as +inf or -inf is that infinity (or NaN in 3xTF32,
    whose cross products can multiply an infinity by a zero low part), and
    every output the reference has finite is finite and within tolerance."""
    got = np.asarray(got, np.float64)
    if mode == "simt":
        assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{what}: NaN positions differ"
    else:
        assert np.all(~np.isfinite(got[np.isnan(ref)])), f"{what}: a NaN output came out finite"
    for sign, pos in ((np.isposinf, "+inf"), (np.isneginf, "-inf")):
        r = sign(ref)
        ok = sign(got[r]) | (np.isnan(got[r]) if mode == "force_tc3" else False)
        assert np.all(ok), f"{what}: a {pos} output came out as something else"
    fin = np.isfinite(ref)
    assert np.all(np.isfinite(got[fin])), f"{what}: a finite output came out non-finite"
    within(got[fin], ref[fin], S[fin], tol, what + " (finite outputs)")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1", "simt"])
def test_addmm_non_finite_inputs_propagate(mode):
    M, N, K = 200, 300, 132
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=790)
    a = _plant_non_finite(a, [((3, 5), "inf"), ((7, 9), "-inf"), ((11, 2), "nan"),
                              ((13, 4), "nan_low")])
    b = _plant_non_finite(b, [((6, 40), "inf"), ((8, 41), "nan_low"), ((9, 42), "-inf")])
    b[5, 7] = 0.0  # row 3 of mat1 holds inf at k = 5: inf * 0 is NaN in column 7
    ref, S = oracle.addmm(s, a, b)
    out = binding.addmm(dev(s), dev(a), dev(b), mode=mode)
    torch.cuda.synchronize()
    assert binding.last_kernel() == {"force_tc3": "tc3", "force_tc1": "tc1", "simt": "simt"}[mode]
    _same_non_finite(out.cpu().numpy(), ref, S, TOL[mode], mode, f"addmm {mode} non-finite")


@pytest.mark.parametrize("mode", ["force_tc3", "force_tc1", "simt"])
@pytest.mark.parametrize("ic", [3, 32])  # slab form / channel-fastest gather
def test_conv_non_finite_inputs_propagate(mode, ic):
    B, H, W, OC = 1, 32, 64, 40
    x, w, bias = synth.conv_inputs(B, ic, H, W, OC, 3, 3, workload=791 + ic)
    x = _plant_non_finite(x, [((0, 1, 5, 7), "inf"), ((0, 2, 20, 30), "nan_low"),
                              ((0, 0, 10, 50), "-inf"), ((0, 1, 25, 12), "nan")])
    w = _plant_non_finite(w, [((17, 0, 1, 1), "nan_low"), ((30, 2, 0, 2), "inf")])
    # padding taps read 0 and are multiplied like any other (an infinite
    # weight times a padding zero is NaN): the reference is the oracle on the
    # explicitly zero-padded input, which equals the padded form for finite data
    xp = np.pad(x, ((0, 0), (0, 0), (1, 1), (1, 1)))
    ref, S = oracle.conv2d(xp, w, bias, 1, 0, 1)
    out = binding.conv2d(dev(x), dev(w), dev(bias), 1, 1, 1, mode=mode)
    torch.cuda.synchronize()
    _same_non_finite(out.cpu().numpy(), ref, S, TOL[mode], mode, f"conv IC={ic} {mode} non-finite")
