"""gemm_addmm_f32_noalloc: the addmm entry point for callers that cannot
allocate device memory while they run (a runtime whose memory is fixed at
start-up, an operator whose host framework forbids allocation in its compute
callback).  It keeps the tensor-core path's scratch in a fixed buffer inside
the library instead of taking it from a memory pool or from the caller.

The GPU test calls it through the C ABI twice in a row (different shapes, so
the second call runs on whatever the first left in the shared buffer) and
checks each result against the existing entry point's, within the parity
bound the other tests use.  This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import binding, build, synth


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_oversized_problem_is_rejected_before_any_cuda_call(lib):
    # 3xTF32 scratch is 2*N*K*4 bytes; N*K = 2048*4096 needs 64 MiB > 32 MiB
    P = 0x10000000
    rc = binding.gemm_addmm_f32_noalloc(P, 0, P + (1 << 26), P + (1 << 28), P + (1 << 29),
                                        4096, 2048, 4096, 1.0, 1.0, 0, None)
    assert rc == binding.IMC_ERR_SCRATCH
    assert "scratch" in binding.status_string(rc)
    # the same shape fits in 1xTF32 mode (N*K*4 = 32 MiB): it passes the size
    # check and stops at the ordinary validation (NULL out), launching nothing
    rc = binding.gemm_addmm_f32_noalloc(P, 0, P + (1 << 26), P + (1 << 28), None,
                                        4096, 2048, 4096, 1.0, 1.0, 1, None)
    assert rc == binding.IMC_ERR_NULL


@pytest.mark.gpu
def test_noalloc_matches_existing_entry_point_twice(lib):
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
        got = torch.empty((M, N), device="cuda")
        want = torch.empty((M, N), device="cuda")
        rc = binding.gemm_addmm_f32_noalloc(S.data_ptr(), int(self_2d), A.data_ptr(), B.data_ptr(),
                                            got.data_ptr(), M, N, K, beta, alpha, mode, stream)
        assert rc == binding.IMC_OK, binding.status_string(rc)
        assert binding.last_kernel() == "tc3"
        rc = binding.gemm_addmm_f32_ex(S.data_ptr(), int(self_2d), A.data_ptr(), B.data_ptr(),
                                       want.data_ptr(), M, N, K, beta, alpha, mode, stream)
        assert rc == binding.IMC_OK
        torch.cuda.synchronize()
        _, Sabs = oracle.addmm(s, a, b, beta=beta, alpha=alpha)
        err = np.abs(got.cpu().numpy().astype(np.float64) - want.cpu().numpy())
        assert np.all(err <= 1e-5 * Sabs + 1e-6), f"call {i}: worst {np.max(err / (1e-5 * Sabs + 1e-6))}"
    assert binding.check_device_error(None) == binding.IMC_OK
