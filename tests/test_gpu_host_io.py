"""GPU parity of the host-buffer entry points (gemm_addmm_f32_host,
conv2d_gemm_f32_host): inputs and output in host memory, the library copies
them and runs the same kernels as the device entry points.

Checked against the fp64 oracle with the bounds of test_gpu_parity, and bit
for bit against the device entry point on the same inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

TOL = {"default": 1e-5, "tf32": 2e-3, "simt": 1e-5}


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    binding.load()
    yield
    assert binding.check_device_error(None) == binding.IMC_OK, "a kernel hit its wait limit"


def host(a, pinned):
    if a is None:
        return None
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.pin_memory() if pinned else t


def within(got, ref, S, c, what):
    err = np.abs(np.asarray(got, np.float64) - ref)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= c * S + 1e-6), f"{what}: worst {float((err / (c * S + 1e-6)).max()):.3g}"


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
@pytest.mark.parametrize("mode", ["default", "tf32", "simt"])
def test_addmm_host_matches_oracle_and_device_path(mode, pinned):
    for M, N, K, self_2d, beta, alpha in [(300, 200, 100, False, 1.0, 1.0),
                                          (257, 516, 1028, True, 0.5, 2.0)]:
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=700 + M)
        stream = torch.cuda.Stream()
        out = binding.addmm_host(host(s, pinned), host(a, pinned), host(b, pinned), beta=beta,
                                 alpha=alpha, mode=mode, stream=stream)
        stream.synchronize()
        ref, S = oracle.addmm(s, a, b, beta=beta, alpha=alpha, self_2d=self_2d)
        within(out.numpy(), ref, S, TOL[mode], f"addmm_host {mode} {M}x{N}x{K}")
        d = binding.addmm(torch.from_numpy(s).cuda(), torch.from_numpy(a).cuda(),
                          torch.from_numpy(b).cuda(), beta=beta, alpha=alpha, mode=mode)
        assert torch.equal(d.cpu(), out), "host and device entry points differ"


def test_addmm_host_in_place_on_self():
    M, N, K = 200, 260, 132
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=True, workload=710)
    self_h = host(s, True)
    out = binding.addmm_host(self_h, host(a, True), host(b, True), beta=1.25, alpha=0.75,
                             out=self_h)
    torch.cuda.current_stream().synchronize()
    assert out.data_ptr() == self_h.data_ptr()
    ref, S = oracle.addmm(s, a, b, beta=1.25, alpha=0.75, self_2d=True)
    within(self_h.numpy(), ref, S, 1e-5, "addmm_host in place")


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_conv2d_host_matches_oracle_and_device_path(pinned):
    for (B, IC, H, W, OC, KH, KW, st, pad, dil) in [(2, 16, 20, 20, 130, 3, 3, 1, 1, 1),
                                                    (1, 3, 64, 64, 128, 7, 7, 4, 3, 1),
                                                    (1, 5, 12, 40, 36, 3, 2, (2, 3), (1, 0),
                                                     (1, 2))]:
        x, w, bias = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=720 + OC)
        stream = torch.cuda.Stream()
        out = binding.conv2d_host(host(x, pinned), host(w, pinned), host(bias, pinned), st, pad,
                                  dil, stream=stream)
        stream.synchronize()
        ref, S = oracle.conv2d(x, w, bias, st, pad, dil)
        within(out.numpy(), ref, S, 1e-5, f"conv2d_host {(B, IC, H, W, OC, KH, KW)}")
        d = binding.conv2d(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(),
                           torch.from_numpy(bias).cuda(), st, pad, dil)
        assert torch.equal(d.cpu(), out), "host and device entry points differ"


def test_host_calls_on_two_streams_overlap_safely():
    # consecutive calls on different streams share nothing: each result is
    # that of its own inputs
    M, N, K = 512, 384, 256
    cases = [synth.addmm_inputs(M, N, K, self_2d=False, workload=730 + i) for i in range(4)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for i, (s, a, b) in enumerate(cases):
        outs.append(binding.addmm_host(host(s, True), host(a, True), host(b, True),
                                       stream=streams[i % 2]))
    for st in streams:
        st.synchronize()
    for (s, a, b), out in zip(cases, outs):
        ref, S = oracle.addmm(s, a, b, beta=1.0, alpha=1.0, self_2d=False)
        within(out.numpy(), ref, S, 1e-5, "two streams")


def test_release_memory_after_work():
    s, a, b = synth.addmm_inputs(256, 256, 256, self_2d=False, workload=740)
    out = binding.addmm_host(host(s, True), host(a, True), host(b, True))
    torch.cuda.synchronize()
    assert binding.release_memory() == binding.IMC_OK
    # the pool is re-used (and grows again) after a release
    out2 = binding.addmm_host(host(s, True), host(a, True), host(b, True))
    torch.cuda.synchronize()
    assert torch.equal(out, out2)


def test_calls_from_several_host_threads():
    # four host threads call the device and host entry points at once, each on
    # its own stream; every result is that of its own inputs
    import threading
    cases = [synth.addmm_inputs(384 + 64 * i, 512, 320, self_2d=bool(i % 2), workload=750 + i)
             for i in range(4)]
    results, errors = [None] * 4, []

    def work(i):
        try:
            s, a, b = cases[i]
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                d = binding.addmm(torch.from_numpy(s).cuda(), torch.from_numpy(a).cuda(),
                                  torch.from_numpy(b).cuda(), beta=0.5)
                h = binding.addmm_host(host(s, True), host(a, True), host(b, True), beta=0.5,
                                       stream=st)
            st.synchronize()
            results[i] = (d.cpu(), h)
        except Exception as e:  # reported below
            errors.append(e)

    threads = [threading.Thread(target=work, args=(i,)) for i in range(4)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for (s, a, b), (d, h) in zip(cases, results):
        ref, S = oracle.addmm(s, a, b, beta=0.5, alpha=1.0, self_2d=s.ndim == 2)
        within(d.numpy(), ref, S, 1e-5, "device call from a thread")
        assert torch.equal(d, h)
