"""GPU parity for the widened rows: aten.linear (weight given as [N,K]), the
fused ReLU epilogue flag, and the direct conv2d kernel kept as a baseline.

Every result is compared with the fp64 oracle element by element under the
same bound as the other parity tests (ReLU is 1-Lipschitz, so the bound of
the pre-activation value carries over).
"""
import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

TOL = {"default": 1e-5, "simt": 1e-5, "force_tc3": 1e-5, "tf32": 2e-3, "force_tc1": 2e-3,
       "direct": 1e-5}
EXPECT = {"simt": "simt", "force_tc3": "tc3", "force_tc1": "tc1", "direct": "direct"}


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    binding.load()
    yield
    assert binding.check_device_error(None) == binding.IMC_OK


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def within(got, ref, S, c, what=""):
    got = np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), what
    ratio = float((np.abs(got - ref) / (c * S + 1e-6)).max())
    assert ratio <= 1.0, f"{what}: worst |err|/tol = {ratio:.3g}"


LINEAR = [(1024, 3072, 768), (577, 768, 3072), (130, 132, 36), (300, 257, 128), (64, 80, 96)]


@pytest.mark.parametrize("mode", ["simt", "force_tc3", "force_tc1", "default"])
@pytest.mark.parametrize("mnk", LINEAR, ids=lambda t: "x".join(map(str, t)))
def test_linear_matches_oracle(mode, mnk):
    M, N, K = mnk
    x = synth.normal(synth.stream_key(0, 600 + M, 1), M * K).reshape(M, K)
    s = 1.0 / np.sqrt(K)
    w = synth.uniform(synth.stream_key(0, 600 + M, 2), N * K, -s, s).reshape(N, K)
    b = synth.normal(synth.stream_key(0, 600 + M, 3), N, 0.0, 0.02)
    for bias in (b, None):
        out = binding.linear(dev(x), dev(w), dev(bias), mode=mode)
        torch.cuda.synchronize()
        if mode in EXPECT:
            assert binding.last_kernel() == EXPECT[mode]
        ref, S = oracle.addmm(bias, x, np.ascontiguousarray(w.T), beta=1.0 if bias is not None
                              else 0.0, alpha=1.0, self_2d=False)
        within(out.cpu().numpy(), ref, S, TOL[mode], f"linear {mnk} {mode} bias={bias is not None}")


@pytest.mark.parametrize("mode", ["default", "force_tc3", "force_tc1"])
def test_linear_k_not_multiple_of_4_on_tensor_cores(mode):
    # weight rows of K % 4 != 0 floats: the weight (hi and lo) and x are
    # copied to rows of K rounded up to 4 in the scratch
    for M, N, K in [(70, 40, 33), (1024, 768, 770), (300, 257, 3)]:
        x = synth.uniform(synth.stream_key(0, 650 + K, 1), M * K, -1, 1).reshape(M, K)
        w = synth.uniform(synth.stream_key(0, 650 + K, 2), N * K, -1, 1).reshape(N, K)
        b = synth.normal(synth.stream_key(0, 650 + K, 3), N, 0.0, 0.02)
        out = binding.linear(dev(x), dev(w), dev(b), mode=mode)
        torch.cuda.synchronize()
        tiny = M * N * K < (1 << 22)
        assert binding.last_kernel() == EXPECT.get(mode, "simt" if tiny else "tc3")
        ref, S = oracle.addmm(b, x, np.ascontiguousarray(w.T))
        within(out.cpu().numpy(), ref, S, TOL[mode], f"linear {M}x{N}x{K} {mode}")


def test_linear_integer_inputs_are_bit_exact():
    M, N, K = 257, 260, 512
    x = synth.integers(synth.stream_key(0, 660, 1), M * K, -4, 4).reshape(M, K)
    w = synth.integers(synth.stream_key(0, 660, 2), N * K, -4, 4).reshape(N, K)
    b = synth.integers(synth.stream_key(0, 660, 3), N, -4, 4)
    ref, _ = oracle.addmm(b, x, np.ascontiguousarray(w.T))
    for mode in ("simt", "force_tc3", "force_tc1"):
        got = binding.linear(dev(x), dev(w), dev(b), mode=mode).cpu().numpy()
        assert np.array_equal(got.astype(np.float64), ref), mode


@pytest.mark.parametrize("mode", ["simt", "force_tc3", "force_tc1"])
def test_addmm_relu(mode):
    for M, N, K, self_2d in [(300, 260, 128, True), (1024, 768, 3072, False)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=670 + K)
        out = binding.addmm(dev(s), dev(a), dev(b), beta=0.5, alpha=1.5, mode=mode, relu=True)
        torch.cuda.synchronize()
        assert binding.last_kernel() == EXPECT[mode]
        ref, S = oracle.addmm(s, a, b, beta=0.5, alpha=1.5)
        got = out.cpu().numpy()
        assert (got >= 0).all()
        within(got, np.maximum(ref, 0.0), S, TOL[mode], f"addmm relu {mode} {M}x{N}x{K}")
    # epilogue-only path (alpha == 0) applies it too
    out = binding.addmm(dev(s), dev(a), dev(b), beta=-1.0, alpha=0.0, mode=mode, relu=True)
    assert binding.last_kernel() == "fill"
    want = np.broadcast_to(np.maximum(-s, 0).astype(np.float32), (M, N))
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("mode", ["simt", "force_tc3", "force_tc1", "direct"])
def test_conv_relu(mode):
    x, w, b = synth.conv_inputs(2, 16, 20, 20, 130, 3, 3, workload=680)
    out = binding.conv2d(dev(x), dev(w), dev(b), 1, 1, 1, mode=mode, relu=True)
    torch.cuda.synchronize()
    assert binding.last_kernel() == EXPECT[mode]
    ref, S = oracle.conv2d(x, w, b, 1, 1, 1)
    within(out.cpu().numpy(), np.maximum(ref, 0.0), S, TOL[mode], f"conv relu {mode}")


DIRECT = [  # B, IC, H, W, OC, KH, KW, stride, pad, dil (IC % 4 == 0: the 4-channel form)
    (2, 3, 9, 9, 4, 3, 3, 1, 1, 1),
    (1, 3, 64, 64, 128, 7, 7, 4, 3, 1),
    (2, 32, 14, 14, 64, 3, 3, 1, 2, 2),
    (1, 5, 12, 40, 36, 3, 2, (2, 3), (1, 0), (1, 2)),
    (1, 8, 12, 40, 20, 3, 2, (2, 3), (1, 0), (1, 2)),
]


@pytest.mark.parametrize("idx", range(len(DIRECT)))
def test_direct_conv_matches_oracle(idx):
    B, IC, H, W, OC, KH, KW, st, pd, dl = DIRECT[idx]
    x, w, b = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=690 + idx)
    out = binding.conv2d(dev(x), dev(w), dev(b), st, pd, dl, mode="direct")
    torch.cuda.synchronize()
    assert binding.last_kernel() == "direct"
    ref, S = oracle.conv2d(x, w, b, st, pd, dl)
    within(out.cpu().numpy(), ref, S, 1e-5, f"direct conv #{idx}")
    xi, wi, bi = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=695 + idx,
                                   x=("I", -4, 4), w=("I", -4, 4), bias=("I", -4, 4))
    got = binding.conv2d(dev(xi), dev(wi), dev(bi), st, pd, dl, mode="direct").cpu().numpy()
    ref, _ = oracle.conv2d(xi, wi, bi, st, pd, dl)
    assert np.array_equal(got.astype(np.float64), ref)


def test_direct_conv_workload_channels():
    # the benchmark's body conv on the direct kernel, checked on 16 channels
    c, x, w, b = synth.make_conv_case("body_56_3x3_d1")
    out = binding.conv2d(dev(x), dev(w), dev(b), c["stride"], c["pad"], c["dilation"],
                         mode="direct").cpu().numpy()
    ch = np.arange(0, 256, 16)
    ref, S = oracle.conv2d(x, w, b, c["stride"], c["pad"], c["dilation"], channels=ch)
    within(out[:, ch], ref, S, 1e-5, "direct body conv")
