"""GPU parity at the largest sizes the entry points take.

* addmm whose output has more than 2^31 elements (70000 x 32800): every
  offset into out and into a [M,N] self needs 64-bit arithmetic; N is ragged
  against the 256-column tile.
* conv2d whose output is just under the 2^31-element limit the conv kernels'
  32-bit offsets allow (1 x 1024 x 1448 x 1448).

Inputs are small integers, so every product and partial sum is exact in fp32
and TF32: the sampled outputs must equal the fp64 oracle bit for bit, in every
mode.  The oracle computes only the sampled rows / channels.
"""
import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

INT = ("I", -2, 2)


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    binding.load()
    yield
    torch.cuda.empty_cache()
    assert binding.check_device_error(None) == binding.IMC_OK, "a kernel hit its wait limit"


def _rows(M, N, count, workload):
    rows = set(synth.sample_rows(synth.stream_key(0, workload, 9), M, count).tolist())
    cross = (1 << 31) // N  # the first row whose offsets pass 2^31
    rows |= {0, cross - 1, cross, cross + 1, M - 1}
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("mode", ["default", "tf32", "simt"])
def test_addmm_output_past_2_pow_31_elements(mode):
    M, N, K = 70000, 32800, 16
    assert M * N > (1 << 31)
    _, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=900, mat1=INT, mat2=INT,
                                 self_=INT)
    # self [M,N] = c[m] + r[n]: small integers, built on the device from two
    # host vectors; out is self (in place)
    c = (np.arange(M) % 9 - 4).astype(np.float32)
    r = (np.arange(N) % 5 - 2).astype(np.float32)
    rows = _rows(M, N, 48, 901)
    A, B = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    out = torch.from_numpy(c).cuda()[:, None] + torch.from_numpy(r).cuda()[None, :]
    binding.addmm(out, A, B, beta=0.5, alpha=1.0, mode=mode, out=out)
    torch.cuda.synchronize()
    kern = binding.last_kernel()
    got = out[torch.from_numpy(rows).cuda()].cpu().numpy()
    del out
    torch.cuda.empty_cache()
    self_rows = (c[rows][:, None] + r[None, :]).astype(np.float32)
    ref, _ = oracle.addmm(self_rows, a[rows], b, beta=0.5, alpha=1.0, self_2d=True)
    assert kern == {"default": "tc3", "tf32": "tc1", "simt": "simt"}[mode]
    assert np.array_equal(got.astype(np.float64), ref), \
        f"{mode}: {int((got != ref).sum())} sampled outputs differ"


def test_addmm_output_past_2_pow_31_elements_vector_self():
    # the tensor-core path's TMA-store epilogue (vector self, N % 4 == 0)
    M, N, K = 70000, 32800, 16
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=902, mat1=INT, mat2=INT,
                                 self_=INT)
    rows = _rows(M, N, 48, 903)
    out = binding.addmm(torch.from_numpy(s).cuda(), torch.from_numpy(a).cuda(),
                        torch.from_numpy(b).cuda())
    torch.cuda.synchronize()
    got = out[torch.from_numpy(rows).cuda()].cpu().numpy()
    del out
    torch.cuda.empty_cache()
    ref, _ = oracle.addmm(s, a, b, rows=rows)
    assert binding.last_kernel() == "tc3"
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("mode", ["default", "tf32", "simt"])
def test_conv_output_at_the_32_bit_limit(mode):
    B, IC, H, W, OC, KH, KW = 1, 16, 1448, 1448, 1024, 3, 3
    assert B * OC * H * W < (1 << 31) and B * OC * H * W > (1 << 31) - (1 << 20)
    x, w, bias = synth.conv_inputs(B, IC, H, W, OC, KH, KW, workload=910, x=INT, w=INT,
                                   bias=INT)
    channels = [0, 255, 256, 777, OC - 1]
    out = binding.conv2d(torch.from_numpy(x).cuda(), torch.from_numpy(w).cuda(),
                         torch.from_numpy(bias).cuda(), 1, 1, 1, mode=mode)
    torch.cuda.synchronize()
    kern = binding.last_kernel()
    got = out[:, channels].cpu().numpy()
    del out
    torch.cuda.empty_cache()
    ref, _ = oracle.conv2d(x, w, bias, 1, 1, 1, channels=channels)
    assert kern == {"default": "tc3", "tf32": "tc1", "simt": "simt"}[mode]
    assert np.array_equal(got.astype(np.float64), ref), \
        f"{mode}: {int((got != ref).sum())} sampled outputs differ"
