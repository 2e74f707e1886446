"""C-ABI boundary checks that need no GPU.

The library must load, export every function include/imc.h declares, and
reject bad arguments with the documented status before touching CUDA.  On a
machine without a GPU a well-formed call must fail loudly (IMC_ERR_DEVICE),
never fall back to host code.
"""
import json
import os
import re
import subprocess
import sys

import pytest
import torch

from addmm_implicit_im2col_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "imc.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


# Calls whose arguments are valid up to the device check use fake addresses;
# they run in a child process that sees no GPU (CUDA_VISIBLE_DEVICES=""), so
# they can never launch anything, whatever machine runs the suite.
_CHILD = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
from addmm_implicit_im2col_gb300 import binding
calls = json.loads(sys.argv[2])
print(json.dumps([getattr(binding, fn)(*args) for fn, args in calls]))
"""


def without_gpu(calls):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT, json.dumps(calls)], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("gemm_addmm_f32", "conv2d_gemm_f32", "gemm_addmm_f32_ex", "conv2d_gemm_f32_ex",
                 "conv2d_gemm_f32_nd", "imc_status_string"):
        assert want in names, names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"libimc.so does not export {n}"
        assert n in binding.SIGNATURES, f"binding has no signature for {n}"


def test_library_has_no_torch_dependency(lib):
    # The boundary is plain C: the shared object must not need libtorch.
    import subprocess
    out = subprocess.run(["ldd", binding.LIB_PATH], capture_output=True, text=True).stdout
    assert "torch" not in out and "c10" not in out


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        s = binding.status_string(code)
        assert s.startswith("IMC_")
    assert binding.status_string(-99) == "IMC_ERR_UNKNOWN"
    assert lib.imc_version() >= 100


# fake, never dereferenced device addresses (validation runs before any CUDA call)
P1, P2, P3, P4 = 0x10000000, 0x20000000, 0x30000000, 0x40000000


def g(self=P1, self_2d=0, mat1=P2, mat2=P3, out=P4, M=8, N=8, K=8, beta=1.0, alpha=1.0, mode=0):
    return binding.gemm_addmm_f32_ex(self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode,
                                     None)


def test_addmm_argument_errors(lib):
    assert g(self_2d=2) == binding.IMC_ERR_ARG
    assert g(mode=7) == binding.IMC_ERR_ARG
    assert g(mode=-1) == binding.IMC_ERR_ARG
    assert g(mode=5) == binding.IMC_ERR_ARG             # the direct kernel is conv-only
    assert g(mode=0x200) == binding.IMC_ERR_ARG         # unknown flag bit
    assert g(mode=0x100 | 7) == binding.IMC_ERR_ARG     # ReLU flag on a bad mode
    assert g(alpha=float("nan")) == binding.IMC_ERR_ARG
    assert g(beta=float("inf")) == binding.IMC_ERR_ARG
    assert g(M=-1) == binding.IMC_ERR_SHAPE
    assert g(K=-5) == binding.IMC_ERR_SHAPE
    assert g(N=2 ** 31) == binding.IMC_ERR_SHAPE
    assert g(out=None) == binding.IMC_ERR_NULL
    assert g(mat1=None) == binding.IMC_ERR_NULL
    assert g(mat2=None) == binding.IMC_ERR_NULL
    assert g(self=None) == binding.IMC_ERR_NULL
    # out overlapping an operand
    assert g(out=P2 + 16) == binding.IMC_ERR_ALIAS
    assert g(out=P3) == binding.IMC_ERR_ALIAS
    # out overlapping a [N] self, or a [M,N] self at an offset
    assert g(out=P1) == binding.IMC_ERR_ALIAS
    assert g(self_2d=1, out=P1 + 4) == binding.IMC_ERR_ALIAS


def gargs(self=P1, self_2d=0, mat1=P2, mat2=P3, out=P4, M=8, N=8, K=8, beta=1.0, alpha=1.0,
          mode=0):
    return ["gemm_addmm_f32_ex", [self, self_2d, mat1, mat2, out, M, N, K, beta, alpha, mode, None]]


def test_addmm_unread_operands_may_be_null(lib):
    # beta == 0: self is not read; alpha == 0 or K == 0: operands are not read;
    # out may equal self for an in-place [M,N] addmm.  These pass validation
    # and then need a device.
    got = without_gpu([gargs(self=None, beta=0.0), gargs(mat1=None, mat2=None, alpha=0.0),
                       gargs(mat1=None, mat2=None, K=0), gargs(self_2d=1, self=P4)])
    assert got == [binding.IMC_ERR_DEVICE] * 4


def test_empty_problems_are_noops(lib):
    assert g(M=0, out=None, mat1=None, mat2=None, self=None) == binding.IMC_OK
    assert g(N=0) == binding.IMC_OK
    assert binding.last_kernel() == "none"


def test_workspace_size_query(lib):
    q = binding.gemm_addmm_f32_workspace_bytes
    assert q(1024, 3072, 768, 0) == 2 * 3072 * 768 * 4  # 3xTF32: hi and lo of mat2^T
    assert q(1024, 3072, 768, 1) == 3072 * 768 * 4      # 1xTF32: mat2^T only
    # few output tiles and a long K: the preferred plan adds split-K partial sums
    assert q(1024, 768, 3072, 0) > 2 * 768 * 3072 * 4
    assert q(1024, 3072, 768, 2) == 0                   # SIMT needs none
    assert q(64, 80, 96, 0) == 0                        # tiny: SIMT
    assert q(64, 80, 96, 3) == 2 * 80 * 96 * 4          # forced tensor-core kernel
    # K % 4 != 0: the tensor-core path with rows of 772 floats -- mat2^T hi and
    # lo, then a copy of mat1 -- so that every row the TMA reads is aligned
    assert q(1024, 3072, 770, 0) == 2 * 3072 * 772 * 4 + 1024 * 772 * 4
    assert q(1024, 3072, 770, 1) == 3072 * 772 * 4 + 1024 * 772 * 4
    # linear with K % 4 != 0: the weight copied too (hi and lo), then mat1
    assert binding.linear_f32_workspace_bytes(1024, 3072, 770, 0) == \
        2 * 3072 * 772 * 4 + 1024 * 772 * 4
    assert q(0, 8, 8, 0) == 0 and q(8, 8, -1, 0) == 0 and q(8, 8, 8, 9) == 0


def gws(ws, nbytes, M=256, N=256, K=256, mode=0, out=P4):
    return binding.gemm_addmm_f32_ws(P1, 0, P2, P3, out, M, N, K, 1.0, 1.0, mode, ws, nbytes,
                                     None)


def test_workspace_argument_errors(lib):
    need = binding.gemm_addmm_f32_workspace_bytes(256, 256, 256, 0)
    minimum = 2 * 256 * 256 * 4  # the mat2 copy alone; more lets the plan split K
    assert need >= minimum
    W = 0x50000000
    assert gws(W, minimum - 4) == binding.IMC_ERR_ARG    # too small
    assert gws(None, need) == binding.IMC_ERR_ARG        # missing
    assert gws(W + 4, need) == binding.IMC_ERR_ARG       # not 16-byte aligned
    assert gws(P4 - 16, need) == binding.IMC_ERR_ALIAS   # overlaps out
    assert gws(P2, need) == binding.IMC_ERR_ALIAS        # overlaps mat1
    valid = ["gemm_addmm_f32_ws", [P1, 0, P2, P3, P4, 256, 256, 256, 1.0, 1.0, 0, W, need, None]]
    simt = ["gemm_addmm_f32_ws", [P1, 0, P2, P3, P4, 256, 256, 256, 1.0, 1.0, 2, None, 0, None]]
    at_min = ["gemm_addmm_f32_ws", [P1, 0, P2, P3, P4, 256, 256, 256, 1.0, 1.0, 0, W, minimum,
                                    None]]
    assert without_gpu([valid, simt, at_min]) == [binding.IMC_ERR_DEVICE] * 3  # needs a GPU


def c(x=P1, w=P2, bias=P3, out=P4, B=2, IC=3, H=8, W=8, OC=4, KH=3, KW=3, sH=1, sW=1, pH=1, pW=1,
      dH=1, dW=1, mode=0):
    return binding.conv2d_gemm_f32_nd(x, w, bias, out, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH,
                                      dW, mode, None)


def test_conv_argument_errors(lib):
    assert c(mode=9) == binding.IMC_ERR_ARG
    assert c(B=-1) == binding.IMC_ERR_SHAPE
    assert c(H=0) == binding.IMC_ERR_SHAPE
    assert c(KH=0) == binding.IMC_ERR_SHAPE
    assert c(sW=0) == binding.IMC_ERR_SHAPE
    assert c(pH=-1) == binding.IMC_ERR_SHAPE
    assert c(dW=0) == binding.IMC_ERR_SHAPE
    assert c(H=2, KH=5, pH=0) == binding.IMC_ERR_SHAPE  # empty output
    assert c(B=1 << 16, IC=1 << 10, H=64, W=64) == binding.IMC_ERR_SHAPE  # 2^38 elements
    assert c(out=None) == binding.IMC_ERR_NULL
    assert c(x=None) == binding.IMC_ERR_NULL
    assert c(w=None) == binding.IMC_ERR_NULL
    assert c(out=P1) == binding.IMC_ERR_ALIAS
    assert c(out=P3 - 8) == binding.IMC_ERR_ALIAS
    no_bias = ["conv2d_gemm_f32_nd", [P1, P2, None, P4, 2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1, 0,
                                      None]]
    assert without_gpu([no_bias]) == [binding.IMC_ERR_DEVICE]  # bias is optional
    assert c(B=0) == binding.IMC_OK
    assert c(OC=0) == binding.IMC_OK
    # the symmetric entry point maps onto the per-axis one
    assert binding.conv2d_gemm_f32(P1, P2, P3, P4, 2, 3, 8, 8, 4, 3, 3, 0, 1, 1,
                                   None) == binding.IMC_ERR_SHAPE
    assert binding.conv2d_gemm_f32_ex(P1, P2, P3, P4, 2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 6,
                                      None) == binding.IMC_ERR_ARG


def test_conv_workspace_size_query(lib):
    q = binding.conv2d_gemm_f32_workspace_bytes
    body = (8, 256, 56, 56, 256, 3, 3, 1, 1, 1, 1, 1, 1)
    # hi and lo weight planes, then the partial sums of the last wave's 48
    # tiles (each 56x56 image in 25 tiles of up to 128 positions: 200 tiles on
    # 152 SMs), each cut into 3 K-slices of a 128 x 256 fp32 tile
    parts = 48 * 3 * 128 * 256 * 4
    assert q(*body, 0) == 2 * 256 * 2304 * 4 + parts
    assert q(*body, 1) == 256 * 2304 * 4 + parts
    assert q(*body, 2) == 0
    stem = (1, 3, 768, 768, 128, 7, 7, 4, 4, 3, 3, 1, 1)
    assert q(*stem, 0) == 2 * 128 * 148 * 4    # K = 147 padded to 148
    assert q(2, 3, 9, 9, 4, 3, 3, 1, 1, 1, 1, 1, 1, 0) == 0  # tiny: SIMT
    assert q(2, 3, 2, 2, 4, 5, 5, 1, 1, 0, 0, 1, 1, 0) == 0  # empty output: invalid


def test_conv_workspace_argument_errors(lib):
    args = (P1, P2, P3, P4, 8, 256, 56, 56, 256, 3, 3, 1, 1, 1, 1, 1, 1, 0)
    need = binding.conv2d_gemm_f32_workspace_bytes(*args[4:])
    least = 2 * 256 * 2304 * 4  # the weight planes alone (no K-slices)
    assert need > least
    W = 0x50000000
    f = binding.conv2d_gemm_f32_ws
    assert f(*args, W, least - 1, None) == binding.IMC_ERR_ARG
    assert f(*args, None, need, None) == binding.IMC_ERR_ARG
    assert f(*args, W + 8, need, None) == binding.IMC_ERR_ARG
    assert f(*args, P2 + 64, need, None) == binding.IMC_ERR_ALIAS  # overlaps w
    assert without_gpu([["conv2d_gemm_f32_ws", list(args) + [W, need, None]],
                        ["conv2d_gemm_f32_ws", list(args) + [W, least, None]]]) == [
        binding.IMC_ERR_DEVICE] * 2


def test_mode_flags_and_linear_validation(lib):
    # ReLU flag and the conv-only direct mode pass validation (then need a device)
    relu = gargs(mode=binding.ACT_RELU | 3)
    direct = ["conv2d_gemm_f32_nd", [P1, P2, P3, P4, 2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1,
                                     5 | binding.ACT_RELU, None]]
    lin = ["linear_f32", [P1, P2, P3, P4, 8, 8, 8, 0, None]]
    lin_nobias = ["linear_f32", [P1, P2, None, P4, 8, 8, 8, 1, None]]
    assert without_gpu([relu, direct, lin, lin_nobias]) == [binding.IMC_ERR_DEVICE] * 4
    L = binding.linear_f32
    assert L(P1, P2, P3, None, 8, 8, 8, 0, None) == binding.IMC_ERR_NULL
    assert L(None, P2, P3, P4, 8, 8, 8, 0, None) == binding.IMC_ERR_NULL
    assert L(P1, P2, P3, P1, 8, 8, 8, 0, None) == binding.IMC_ERR_ALIAS
    assert L(P1, P2, P3, P4, -1, 8, 8, 0, None) == binding.IMC_ERR_SHAPE
    assert L(P1, P2, P3, P4, 8, 8, 8, 5, None) == binding.IMC_ERR_ARG
    assert L(P1, P2, P3, P4, 0, 8, 8, 0, None) == binding.IMC_OK
    q = binding.linear_f32_workspace_bytes
    assert q(1024, 3072, 768, 0) == 3072 * 768 * 4  # only the weight's lo part
    assert q(1024, 3072, 768, 1) == 0               # 1xTF32 reads the weight as it is
    assert q(64, 80, 96, 0) == 0


def test_no_gpu_fails_loudly(lib):
    # a well-formed call on a machine without a usable GPU: an error, no host fallback
    conv = ["conv2d_gemm_f32_nd", [P1, P2, P3, P4, 2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1, 0, None]]
    got = without_gpu([gargs(), conv, ["check_device_error", [None]]])
    assert got == [binding.IMC_ERR_DEVICE] * 3


def test_torch_wrappers_validate_before_calling(lib):
    x = torch.zeros(2, 3)
    with pytest.raises(ValueError):
        binding.addmm(torch.zeros(3), x, torch.zeros(3, 4))  # CPU tensors are refused
    with pytest.raises(TypeError):
        binding.addmm(None, [[1.0]], x)


def test_host_buffer_entry_points_check_before_any_cuda_call(lib):
    # Host pointers are checked like device ones (aliasing on the host
    # ranges); a well-formed call then needs a GPU and fails loudly without one.
    H = binding.gemm_addmm_f32_host
    assert H(P1, 0, P2, P3, None, 8, 8, 8, 1.0, 1.0, 0, None) == binding.IMC_ERR_NULL
    assert H(P1, 0, None, P3, P4, 8, 8, 8, 1.0, 1.0, 0, None) == binding.IMC_ERR_NULL
    assert H(P1, 0, P2, P3, P4, -1, 8, 8, 1.0, 1.0, 0, None) == binding.IMC_ERR_SHAPE
    assert H(P1, 2, P2, P3, P4, 8, 8, 8, 1.0, 1.0, 0, None) == binding.IMC_ERR_ARG
    assert H(P1, 0, P2, P3, P4, 8, 8, 8, 1.0, 1.0, 9, None) == binding.IMC_ERR_ARG
    assert H(P1, 0, P2, P3, P2 + 16, 8, 8, 8, 1.0, 1.0, 0, None) == binding.IMC_ERR_ALIAS
    assert H(P1, 0, P2, P3, P4, 0, 8, 8, 1.0, 1.0, 0, None) == binding.IMC_OK  # empty: no work
    C = binding.conv2d_gemm_f32_host
    conv = [P1, P2, P3, P4, 2, 3, 8, 8, 4, 3, 3, 1, 1, 1, 1, 1, 1, 0, None]
    assert C(*conv[:3], None, *conv[4:]) == binding.IMC_ERR_NULL
    assert C(*conv[:3], P1 + 64, *conv[4:]) == binding.IMC_ERR_ALIAS
    bad = list(conv)
    bad[11] = 0  # stride 0
    assert C(*bad) == binding.IMC_ERR_SHAPE
    # a forced tensor-core mode takes K % 4 != 0 (operand rows are padded in
    # the scratch); the call then needs a GPU
    assert without_gpu([["gemm_addmm_f32_host", [P1, 0, P2, P3, P4, 8, 8, 10, 1.0, 1.0, 3,
                                                 None]]]) == [binding.IMC_ERR_DEVICE]
    got = without_gpu([["gemm_addmm_f32_host", [P1, 0, P2, P3, P4, 8, 8, 8, 1.0, 1.0, 0, None]],
                       ["conv2d_gemm_f32_host", conv]])
    assert got == [binding.IMC_ERR_DEVICE] * 2


def test_host_wrappers_take_cpu_tensors_only(lib):
    with pytest.raises(ValueError):
        binding.addmm_host(None, torch.zeros(2, 3, device="meta"), torch.zeros(3, 4))
    with pytest.raises(ValueError):
        binding.addmm_host(None, torch.zeros(2, 3, dtype=torch.float64), torch.zeros(3, 4))
    with pytest.raises(ValueError):
        binding.conv2d_host(torch.zeros(1, 3, 8, 8), torch.zeros(4, 2, 3, 3))


def test_release_memory_without_work_is_ok(lib):
    # no pool exists before the first call that needs scratch: nothing to trim
    assert without_gpu([["release_memory", []]]) == [binding.IMC_OK]


def test_wait_timeout_selftest_checks_its_limit(lib):
    assert binding.selftest_wait_timeout(999) == binding.IMC_ERR_ARG
    assert binding.selftest_wait_timeout(1000001) == binding.IMC_ERR_ARG
    assert without_gpu([["selftest_wait_timeout", [20000, None]]]) == [binding.IMC_ERR_DEVICE]
