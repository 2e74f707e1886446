"""Calls issued back to back on one stream, with no host synchronisation between
them, against the same calls run one at a time.

Every kernel is a dependent launch: it may be placed while the kernel before
it still runs, and waits for that kernel before it touches memory.  These
cases make a missing or misplaced wait visible: the second call's pre-pass
rewrites the scratch the first call's main kernel reads (one workspace for
both), a call reads what the call before it wrote, or writes what the call
before it reads.  The kernels are deterministic, so the chained results must
equal the one-at-a-time results bit for bit.
"""
import numpy as np
import pytest
import torch

from addmm_implicit_im2col_gb300 import binding, build, synth

pytestmark = pytest.mark.gpu

REPS = 3


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    binding.load()
    yield
    assert binding.check_device_error(None) == binding.IMC_OK, "a kernel hit its wait limit"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _stream():
    return torch.cuda.current_stream().cuda_stream


def conv_ws(x, w, b, out, shape, ws, mode="default"):
    B_, IC, H, W, OC, KH, KW, st, pd, dl = shape
    rc = binding.conv2d_gemm_f32_ws(x.data_ptr(), w.data_ptr(), b.data_ptr(), out.data_ptr(), B_,
                                    IC, H, W, OC, KH, KW, st, st, pd, pd, dl, dl,
                                    binding.MODES[mode], ws.data_ptr(), ws.numel(), _stream())
    assert rc == binding.IMC_OK, binding.status_string(rc)
    return binding.last_kernel_name()


def addmm_ws(s, a, b, out, ws, mode="default"):
    (M, K), N = a.shape, b.shape[1]
    rc = binding.gemm_addmm_f32_ws(s.data_ptr(), 0, a.data_ptr(), b.data_ptr(), out.data_ptr(), M,
                                   N, K, 1.0, 1.0, binding.MODES[mode], ws.data_ptr(), ws.numel(),
                                   _stream())
    assert rc == binding.IMC_OK, binding.status_string(rc)
    return binding.last_kernel_name()


def linear_ws(x, w, b, out, ws, mode="default"):
    (M, K), N = x.shape, w.shape[0]
    rc = binding.linear_f32_ws(x.data_ptr(), w.data_ptr(), b.data_ptr(), out.data_ptr(), M, N, K,
                               binding.MODES[mode], ws.data_ptr(), ws.numel(), _stream())
    assert rc == binding.IMC_OK, binding.status_string(rc)
    return binding.last_kernel_name()


def conv_bytes(shape, mode="default"):
    B_, IC, H, W, OC, KH, KW, st, pd, dl = shape
    return binding.conv2d_gemm_f32_workspace_bytes(B_, IC, H, W, OC, KH, KW, st, st, pd, pd, dl,
                                                   dl, binding.MODES[mode])


def out_hw(n, k, st, pd, dl):
    return (n + 2 * pd - dl * (k - 1) - 1) // st + 1


def one_at_a_time(calls):
    """Runs each call with a device synchronisation after it; returns copies."""
    refs = []
    for fn, out in calls:
        fn()
        torch.cuda.synchronize()
        refs.append(out.clone())
    return refs


def chained(calls, refs, what):
    for rep in range(REPS):
        for _, out in calls:
            out.fill_(float("nan"))
        torch.cuda.synchronize()
        for fn, _ in calls:
            fn()
        torch.cuda.synchronize()
        for i, ((_, out), ref) in enumerate(zip(calls, refs)):
            assert torch.equal(out, ref), f"{what}: call {i} differs on repetition {rep}"


# ------------------------------------------ one workspace for two calls
CONV_PAIRS = [
    (1, 3, 768, 768, 128, 7, 7, 4, 3, 1),  # the stem: transposed slab form
    (2, 64, 28, 28, 128, 3, 3, 1, 1, 1),   # the 128-position form, gathered from global memory
]


@pytest.mark.parametrize("mode", ["default", "tf32"])
@pytest.mark.parametrize("shape", CONV_PAIRS)
def test_conv_pair_sharing_one_workspace(shape, mode):
    # the second call's weight pre-pass rewrites the split weight the first
    # call's main kernel reads
    x, w1, b1 = synth.conv_inputs(*shape[:7], workload=700)
    _, w2, b2 = synth.conv_inputs(*shape[:7], workload=701)
    X, W1, B1, W2, B2 = dev(x), dev(w1), dev(b1), dev(w2), dev(b2)
    OH, OW = out_hw(shape[2], shape[5], shape[7], shape[8], shape[9]), \
        out_hw(shape[3], shape[6], shape[7], shape[8], shape[9])
    o1 = torch.empty((shape[0], shape[4], OH, OW), device="cuda")
    o2 = torch.empty_like(o1)
    ws = torch.empty(max(conv_bytes(shape, mode), 16), dtype=torch.uint8, device="cuda")
    kern = conv_ws(X, W1, B1, o1, shape, ws, mode)
    assert kern.startswith("k_tc_conv"), kern
    calls = [(lambda: conv_ws(X, W1, B1, o1, shape, ws, mode), o1),
             (lambda: conv_ws(X, W2, B2, o2, shape, ws, mode), o2)]
    refs = one_at_a_time(calls)
    assert not torch.equal(refs[0], refs[1])
    chained(calls, refs, f"conv pair {shape}")


# (M, N, K): one wave of whole tiles (no split-K sum kernel), and split-K
ADDMM_PAIRS = [(1024, 3072, 768), (577, 768, 3072)]


@pytest.mark.parametrize("mode", ["default", "tf32"])
@pytest.mark.parametrize("mnk", ADDMM_PAIRS)
def test_addmm_pair_sharing_one_workspace(mnk, mode):
    # the second call's mat2 pre-pass rewrites the transposed, split mat2 the
    # first call's main kernel reads
    M, N, K = mnk
    s, a, b1 = synth.addmm_inputs(M, N, K, self_2d=False, workload=710)
    _, _, b2 = synth.addmm_inputs(M, N, K, self_2d=False, workload=711)
    S, A, B1, B2 = dev(s), dev(a), dev(b1), dev(b2)
    o1 = torch.empty((M, N), device="cuda")
    o2 = torch.empty_like(o1)
    nb = binding.gemm_addmm_f32_workspace_bytes(M, N, K, binding.MODES[mode])
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    kern = addmm_ws(S, A, B1, o1, ws, mode)
    assert kern.startswith("k_tc_gemm<3xtf32" if mode == "default" else "k_tc_gemm<1xtf32"), kern
    calls = [(lambda: addmm_ws(S, A, B1, o1, ws, mode), o1),
             (lambda: addmm_ws(S, A, B2, o2, ws, mode), o2)]
    refs = one_at_a_time(calls)
    chained(calls, refs, f"addmm pair {mnk}")


@pytest.mark.parametrize("mode", ["default", "tf32"])
def test_linear_pair_sharing_one_workspace(mode):
    # default: the second call's w_lo pre-pass rewrites the first call's w_lo;
    # 1xTF32: no pre-pass, each call's main kernel is the dependent launch
    M, N, K = 1024, 3072, 768
    gen = torch.Generator().manual_seed(720)
    x = torch.randn(M, K, generator=gen).cuda()
    w1 = (torch.randn(N, K, generator=gen) / K ** 0.5).cuda()
    w2 = (torch.randn(N, K, generator=gen) / K ** 0.5).cuda()
    bias = (torch.randn(N, generator=gen) * 0.02).cuda()
    o1 = torch.empty((M, N), device="cuda")
    o2 = torch.empty_like(o1)
    nb = binding.linear_f32_workspace_bytes(M, N, K, binding.MODES[mode])
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device="cuda")
    calls = [(lambda: linear_ws(x, w1, bias, o1, ws, mode), o1),
             (lambda: linear_ws(x, w2, bias, o2, ws, mode), o2)]
    refs = one_at_a_time(calls)
    chained(calls, refs, "linear pair")


# ------------------------------------------------- calls that feed calls
def test_addmm_reads_what_the_call_before_wrote():
    # y = self + A @ B, then z = self2 + y @ C: the second call's main kernel
    # reads y from its first instruction
    M, N, K, N2 = 1024, 3072, 768, 768
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=730)
    s2, _, c = synth.addmm_inputs(M, N2, N, self_2d=False, workload=731)
    S, A, B, S2, C = dev(s), dev(a), dev(b), dev(s2), dev(c)
    y = torch.empty((M, N), device="cuda")
    z = torch.empty((M, N2), device="cuda")
    nb = max(binding.gemm_addmm_f32_workspace_bytes(M, N, K, binding.MODES["default"]),
             binding.gemm_addmm_f32_workspace_bytes(M, N2, N, binding.MODES["default"]))
    ws1 = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(nb, dtype=torch.uint8, device="cuda")
    calls = [(lambda: addmm_ws(S, A, B, y, ws1), y), (lambda: addmm_ws(S2, y, C, z, ws2), z)]
    refs = one_at_a_time(calls)
    chained(calls, refs, "addmm -> addmm")


def test_addmm_writes_what_the_call_before_reads():
    # y = self + A @ B, then A = self3 + D @ E: the second call must not write
    # A before the first call's main kernel has read it
    M, N, K, K3 = 1024, 3072, 768, 512
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=740)
    s3, d, e = synth.addmm_inputs(M, K, K3, self_2d=False, workload=741)
    S, B, S3, D, E = dev(s), dev(b), dev(s3), dev(d), dev(e)
    A = dev(a)
    y = torch.empty((M, N), device="cuda")
    nb = max(binding.gemm_addmm_f32_workspace_bytes(M, N, K, binding.MODES["default"]),
             binding.gemm_addmm_f32_workspace_bytes(M, K, K3, binding.MODES["default"]))
    ws1 = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(nb, dtype=torch.uint8, device="cuda")
    a0 = A.clone()
    addmm_ws(S, A, B, y, ws1)
    torch.cuda.synchronize()
    y_ref = y.clone()
    addmm_ws(S3, D, E, A, ws2)
    torch.cuda.synchronize()
    a_new = A.clone()
    for rep in range(REPS):
        A.copy_(a0)
        y.fill_(float("nan"))
        torch.cuda.synchronize()
        addmm_ws(S, A, B, y, ws1)
        addmm_ws(S3, D, E, A, ws2)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), f"addmm read an overwritten mat1 on repetition {rep}"
        assert torch.equal(A, a_new)


def test_stem_output_feeds_an_addmm():
    # the stem conv's output [1, 128, 192, 192] read as mat1 [128 * 192, 192]
    shape = (1, 3, 768, 768, 128, 7, 7, 4, 3, 1)
    x, w, bias = synth.conv_inputs(*shape[:7], workload=750)
    X, W, Bias = dev(x), dev(w), dev(bias)
    y = torch.empty((1, 128, 192, 192), device="cuda")
    M, K, N = 128 * 192, 192, 256
    s, _, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=751)
    S, B = dev(s), dev(b)
    z = torch.empty((M, N), device="cuda")
    ws1 = torch.empty(max(conv_bytes(shape), 16), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty(max(binding.gemm_addmm_f32_workspace_bytes(M, N, K, binding.MODES["default"]),
                          16), dtype=torch.uint8, device="cuda")
    ym = y.view(M, K)
    calls = [(lambda: conv_ws(X, W, Bias, y, shape, ws1), y), (lambda: addmm_ws(S, ym, B, z, ws2), z)]
    refs = one_at_a_time(calls)
    chained(calls, refs, "stem -> addmm")


def test_simt_calls_feed_each_other():
    # tiny addmm calls on the SIMT kernel (no scratch): y = s + A @ B, then
    # z = s2 + y @ C, then A = s3 + D @ E (written while nothing may still read it)
    M, N, K = 64, 80, 96
    s, a, b = synth.addmm_inputs(M, N, K, self_2d=False, workload=760)
    s2, _, c = synth.addmm_inputs(M, K, N, self_2d=False, workload=761)
    s3, d, e = synth.addmm_inputs(M, K, 32, self_2d=False, workload=762)
    S, B, S2, C, S3, D, E = (dev(v) for v in (s, b, s2, c, s3, d, e))
    A = dev(a)
    y = torch.empty((M, N), device="cuda")
    z = torch.empty((M, K), device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    a0 = A.clone()

    def run():
        addmm_ws(S, A, B, y, ws, "simt")
        addmm_ws(S2, y, C, z, ws, "simt")
        addmm_ws(S3, D, E, A, ws, "simt")

    for fn in (lambda: addmm_ws(S, A, B, y, ws, "simt"), lambda: addmm_ws(S2, y, C, z, ws, "simt"),
               lambda: addmm_ws(S3, D, E, A, ws, "simt")):
        fn()
        torch.cuda.synchronize()
    assert binding.last_kernel_name() == "k_simt_small", binding.last_kernel_name()
    y_ref, z_ref, a_ref = y.clone(), z.clone(), A.clone()
    for rep in range(REPS):
        A.copy_(a0)
        y.fill_(float("nan"))
        z.fill_(float("nan"))
        torch.cuda.synchronize()
        for _ in range(4):  # the chain four times over: A is rewritten, then read again
            A.copy_(a0)
            run()
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref) and torch.equal(z, z_ref) and torch.equal(A, a_ref), rep


# ------------------------------------------------ a random mix, one workspace
def _mixed_calls():
    """About thirty calls drawn from the random-shape sweep's lists (addmm of
    every size class, linear, convs of the gather, slab and transposed slab
    forms), 3xTF32 and 1xTF32 alternating, in a seeded random order."""
    from test_gpu_random_shapes import ADDMM, ADDMM_EXTREME, CONV, CONV_T, LINEAR
    rng = np.random.RandomState(77)
    picks = ([("addmm", int(i)) for i in rng.choice(len(ADDMM), 10, replace=False)]
             + [("extreme", int(i)) for i in rng.choice(len(ADDMM_EXTREME), 4, replace=False)]
             + [("conv", int(i)) for i in rng.choice(len(CONV), 9, replace=False)]
             + [("conv_t", int(i)) for i in rng.choice(len(CONV_T), 2, replace=False)]
             + [("linear", int(i)) for i in rng.choice(len(LINEAR), 6, replace=False)])
    rng.shuffle(picks)
    calls, need = [], 16
    for n, (kind, i) in enumerate(picks):
        mode = ("default", "tf32")[n % 2]
        m = binding.MODES[mode]
        if kind in ("addmm", "extreme"):
            t = (ADDMM if kind == "addmm" else ADDMM_EXTREME)[i]
            M, N, K, s2 = t[:4]
            beta, alpha = (t[4], t[5]) if kind == "addmm" else (1.0, 1.0)
            s, a, b = (dev(v) for v in synth.addmm_inputs(M, N, K, self_2d=s2, workload=800 + n))
            out = torch.empty((M, N), device="cuda")
            need = max(need, binding.gemm_addmm_f32_workspace_bytes(M, N, K, m))

            def fn(ws, s=s, a=a, b=b, out=out, M=M, N=N, K=K, s2=s2, beta=beta, alpha=alpha, m=m):
                return binding.gemm_addmm_f32_ws(s.data_ptr(), int(s2), a.data_ptr(), b.data_ptr(),
                                                 out.data_ptr(), M, N, K, beta, alpha, m,
                                                 ws.data_ptr(), ws.numel(), _stream())
        elif kind == "linear":
            M, N, K = LINEAR[i][:3]
            gen = torch.Generator().manual_seed(800 + n)
            x = torch.randn(M, K, generator=gen).cuda()
            w = (torch.randn(N, K, generator=gen) / K ** 0.5).cuda()
            bias = (torch.randn(N, generator=gen) * 0.02).cuda()
            out = torch.empty((M, N), device="cuda")
            need = max(need, binding.linear_f32_workspace_bytes(M, N, K, m))

            def fn(ws, x=x, w=w, bias=bias, out=out, M=M, N=N, K=K, m=m):
                return binding.linear_f32_ws(x.data_ptr(), w.data_ptr(), bias.data_ptr(),
                                             out.data_ptr(), M, N, K, m, ws.data_ptr(), ws.numel(),
                                             _stream())
        else:
            B_, IC, H, W, OC, KH, KW, s, p, d = (CONV if kind == "conv" else CONV_T)[i]
            x, w, bias = (dev(v) for v in synth.conv_inputs(B_, IC, H, W, OC, KH, KW,
                                                             workload=800 + n))
            OH = (H + 2 * p[0] - d[0] * (KH - 1) - 1) // s[0] + 1
            OW = (W + 2 * p[1] - d[1] * (KW - 1) - 1) // s[1] + 1
            out = torch.empty((B_, OC, OH, OW), device="cuda")
            geo = (B_, IC, H, W, OC, KH, KW, s[0], s[1], p[0], p[1], d[0], d[1])
            need = max(need, binding.conv2d_gemm_f32_workspace_bytes(*geo, m))

            def fn(ws, x=x, w=w, bias=bias, out=out, geo=geo, m=m):
                return binding.conv2d_gemm_f32_ws(x.data_ptr(), w.data_ptr(), bias.data_ptr(),
                                                  out.data_ptr(), *geo, m, ws.data_ptr(),
                                                  ws.numel(), _stream())
        calls.append((fn, out))
    return calls, need


def test_random_mix_chained_through_one_workspace():
    # every call's scratch is the same buffer, so each pre-pass (or split-K
    # partial sum) rewrites what the call before it read
    calls, need = _mixed_calls()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    names = set()

    def run(fn):
        rc = fn(ws)
        assert rc == binding.IMC_OK, binding.status_string(rc)
        names.add(binding.last_kernel_name())

    wrapped = [(lambda fn=fn: run(fn), out) for fn, out in calls]
    refs = one_at_a_time(wrapped)
    assert any(n.startswith("k_tc_gemm<3x") for n in names), names
    assert any(n.startswith("k_tc_gemm<1x") for n in names), names
    assert any(n.startswith("k_tc_conv") for n in names), names
    chained(wrapped, refs, "random mix")
