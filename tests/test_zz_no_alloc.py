"""gemm_addmm_f32_noalloc: the addmm entry point for callers that cannot
allocate device memory while they run (a runtime whose memory is fixed at
start-up, an operator whose host framework forbids allocation in its compute
callback).  It keeps the tensor-core path's scratch in a fixed buffer inside
the library instead of taking it from a memory pool or from the caller.

The GPU test calls it through the C ABI twice in a row (different shapes, so
the second call runs on whatever the first left in the shared buffer) and
checks each result three ways: bit for bit against gemm_addmm_f32_ws given a
caller workspace of the same size (the same plan runs, so any stale or
overwritten scratch would show), against the oracle within the parity bound
the other tests use, and -- for the call after the first, which did the
set-up -- that free device memory did not change across it.  This file is
named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import binding, build, synth

MiB = 1 << 20


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_checks_come_before_the_size_check_and_any_cuda_call(lib):
    # Fake, never dereferenced addresses: every call below returns before
    # touching the device.  3xTF32 scratch is 2*N*K*4 bytes; N*K = 2048*4096
    # needs 64 MiB, more than the 32 MiB buffer.
    P = 0x10000000
    s, a, b, o = P, P + (1 << 26), P + (1 << 28), P + (1 << 29)
    big = (4096, 2048, 4096)
    rc = binding.gemm_addmm_f32_noalloc(s, 0, a, b, o, *big, 1.0, 1.0, 0, None)
    assert rc == binding.IMC_ERR_SCRATCH
    assert "scratch" in binding.status_string(rc)
    # the argument errors of gemm_addmm_f32_ex win over the size check, in its order
    assert binding.gemm_addmm_f32_noalloc(s, 2, a, b, o, *big, 1.0, 1.0, 0, None) == \
        binding.IMC_ERR_ARG
    assert binding.gemm_addmm_f32_noalloc(s, 0, a, b, o, *big, 1.0, float("nan"), 0, None) == \
        binding.IMC_ERR_ARG
    assert binding.gemm_addmm_f32_noalloc(s, 0, a, b, o, *big, 1.0, 1.0, 0x7, None) == \
        binding.IMC_ERR_ARG
    assert binding.gemm_addmm_f32_noalloc(s, 0, a, b, o, -1, 2048, 4096, 1.0, 1.0, 0, None) == \
        binding.IMC_ERR_SHAPE
    assert binding.gemm_addmm_f32_noalloc(s, 0, a, b, None, *big, 1.0, 1.0, 0, None) == \
        binding.IMC_ERR_NULL
    assert binding.gemm_addmm_f32_noalloc(None, 0, a, b, o, *big, 1.0, 1.0, 0, None) == \
        binding.IMC_ERR_NULL
    assert binding.gemm_addmm_f32_noalloc(s, 0, a, b, a, *big, 1.0, 1.0, 0, None) == \
        binding.IMC_ERR_ALIAS
    # the same shape fits in 1xTF32 mode (N*K*4 = 32 MiB): it passes the size
    # check and stops at the ordinary validation (NULL out), launching nothing
    assert binding.gemm_addmm_f32_noalloc(s, 0, a, b, None, *big, 1.0, 1.0, 1, None) == \
        binding.IMC_ERR_NULL


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_twice(lib):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    stream = torch.cuda.current_stream().cuda_stream
    cases = [  # (M, N, K, self_2d, beta, alpha, mode): both use the scratch buffer
        (1000, 1536, 1024, False, 1.0, 1.0, 0),
        (577, 768, 3072, True, 0.5, 2.0, 0),
    ]
    for i, (M, N, K, self_2d, beta, alpha, mode) in enumerate(cases):
        assert binding.gemm_addmm_f32_workspace_bytes(M, N, K, mode) <= binding.NOALLOC_SCRATCH_BYTES
        s, a, b = synth.addmm_inputs(M, N, K, self_2d=self_2d, workload=500 + i,
                                     mat1=("N", 0.0, 1.0), mat2=("U", -0.05, 0.05),
                                     self_=("N", 0.0, 1.0))
        S, A, B = (torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in (s, a, b))
        got = torch.full((M, N), float("nan"), device="cuda")
        want = torch.full((M, N), float("nan"), device="cuda")
        ws = torch.empty(binding.NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
        # the twin first: a caller workspace of the same size gives the same plan
        rc = binding.gemm_addmm_f32_ws(S.data_ptr(), int(self_2d), A.data_ptr(), B.data_ptr(),
                                       want.data_ptr(), M, N, K, beta, alpha, mode, ws.data_ptr(),
                                       binding.NOALLOC_SCRATCH_BYTES, stream)
        assert rc == binding.IMC_OK, binding.status_string(rc)
        torch.cuda.synchronize()
        assert binding.release_memory() == binding.IMC_OK  # the library pool holds nothing
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        rc = binding.gemm_addmm_f32_noalloc(S.data_ptr(), int(self_2d), A.data_ptr(), B.data_ptr(),
                                            got.data_ptr(), M, N, K, beta, alpha, mode, stream)
        assert rc == binding.IMC_OK, binding.status_string(rc)
        assert binding.last_kernel() == "tc3"
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        if i > 0:  # the first call on the device was the set-up that loads the buffer
            assert abs(free0 - free1) < 2 * MiB, f"call {i}: free memory {free0} -> {free1}"
        assert torch.equal(got, want), f"call {i}: differs from gemm_addmm_f32_ws"
        ref, Sabs = oracle.addmm(s, a, b, beta=beta, alpha=alpha)
        err = np.abs(got.cpu().numpy().astype(np.float64) - ref)
        ratio = err / (1e-5 * Sabs + 1e-6)
        assert np.all(ratio <= 1.0), f"call {i}: worst {ratio.max()}"
    assert binding.check_device_error(None) == binding.IMC_OK
