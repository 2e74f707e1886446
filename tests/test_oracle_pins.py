"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: hand-derived golden
fixtures, independent library routines (numpy matmul, torch CPU conv2d in
fp64), closed forms and exact identities that follow from the definitions of
addmm and of the implicit-im2col convolution.  ``test_planted_mistakes``
rebuilds the oracle with one deliberate mistake at a time and checks that at
least one pin fails for each.
"""
import json
import os
import tempfile

import numpy as np
import pytest
import torch

import oracle
from addmm_implicit_im2col_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _rand(*shape):
    return rng.uniform(-1, 1, size=shape).astype(np.float32)


def _ints(*shape, lo=-4, hi=4):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


# ------------------------------------------------------------------- pins
# Each pin takes the loaded oracle library L and raises AssertionError on a
# mismatch, so the same pins can run against a build with a planted mistake.

def pin_golden_addmm(L):
    g = json.load(open(os.path.join(GOLDEN, "addmm_hand_2x3x2.json")))
    for case in g["cases"]:
        ref, S = oracle.addmm(np.array(case["self"], np.float32), np.array(g["mat1"], np.float32),
                              np.array(g["mat2"], np.float32), beta=case["beta"],
                              alpha=case["alpha"], _lib=L)
        assert np.array_equal(ref, np.array(case["out"], np.float64)), ref
        assert np.array_equal(S, np.array(case["S"], np.float64)), S


def _golden_conv(L, name):
    g = json.load(open(os.path.join(GOLDEN, name)))
    x = np.array(g["x"], np.float32).reshape(g["x_shape"])
    w = np.array(g["w"], np.float32).reshape(g["w_shape"])
    b = None if g["bias"] is None else np.array(g["bias"], np.float32)
    ref, S = oracle.conv2d(x, w, b, stride=g["stride"], padding=g["padding"],
                           dilation=g["dilation"], _lib=L)
    assert list(ref.shape) == g["out_shape"], ref.shape
    assert np.array_equal(ref.ravel(), np.array(g["out"], np.float64)), ref.ravel()
    assert np.array_equal(S.ravel(), np.array(g["S"], np.float64)), S.ravel()


def pin_golden_conv_s2p1(L):
    _golden_conv(L, "conv_hand_4x4_s2p1.json")


def pin_golden_conv_dil2(L):
    _golden_conv(L, "conv_hand_3x3_dil2.json")


def pin_addmm_vs_numpy(L):
    for (M, K, N) in [(7, 13, 5), (1, 9, 11), (12, 1, 3), (16, 40, 24)]:
        a, b = _rand(M, K), _rand(K, N)
        for self_2d, alpha, beta in [(False, 1.0, 1.0), (True, 2.0, 0.5), (False, -0.75, 1.25)]:
            s = _rand(M, N) if self_2d else _rand(N)
            ref, S = oracle.addmm(s, a, b, beta=beta, alpha=alpha, _lib=L)
            a64, b64, s64 = a.astype(np.float64), b.astype(np.float64), s.astype(np.float64)
            want = beta * (s64 if self_2d else s64[None, :]) + alpha * (a64 @ b64)
            np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(S, np.abs(a64) @ np.abs(b64), rtol=1e-12, atol=1e-12)


def pin_addmm_alpha0(L):
    M, K, N = 6, 5, 7
    a, b, s = _rand(M, K), _rand(K, N), _rand(M, N)
    a[2, 3] = np.nan
    b[1, 1] = np.inf
    ref, S = oracle.addmm(s, a, b, beta=1.5, alpha=0.0, _lib=L)
    assert np.array_equal(ref, 1.5 * s.astype(np.float64))
    assert np.all(S == 0)


def pin_addmm_beta0(L):
    M, K, N = 6, 5, 7
    a, b = _ints(M, K), _ints(K, N)
    s = np.full((N,), np.nan, np.float32)
    ref, _ = oracle.addmm(s, a, b, beta=0.0, alpha=3.0, _lib=L)
    assert np.array_equal(ref, 3.0 * (a.astype(np.float64) @ b.astype(np.float64)))


def pin_addmm_identity(L):
    M, K = 9, 6
    a = _rand(M, K)
    eye = np.eye(K, dtype=np.float32)
    for s in (_rand(K), _rand(M, K)):
        ref, _ = oracle.addmm(s, a, eye, beta=0.25, alpha=2.0, _lib=L)
        s64 = s.astype(np.float64)
        want = 0.25 * (s64 if s.ndim == 2 else s64[None, :]) + 2.0 * a.astype(np.float64)
        assert np.array_equal(ref, want)


def pin_addmm_outer(L):
    a, b = _rand(5, 1), _rand(1, 4)
    ref, S = oracle.addmm(np.zeros(4, np.float32), a, b, beta=1.0, alpha=1.0, _lib=L)
    outer = a.astype(np.float64) * b.astype(np.float64)
    assert np.array_equal(ref, outer)
    assert np.array_equal(S, np.abs(outer))


def pin_addmm_broadcast(L):
    M, K, N = 8, 7, 6
    a, b, row = _rand(M, K), _rand(K, N), _rand(N)
    r1, _ = oracle.addmm(row, a, b, beta=0.5, alpha=1.5, _lib=L)
    r2, _ = oracle.addmm(np.tile(row, (M, 1)), a, b, beta=0.5, alpha=1.5, _lib=L)
    assert np.array_equal(r1, r2)
    # a [M,N] self that is not a broadcast row gives per-row values
    s2 = _rand(M, N)
    r3, _ = oracle.addmm(s2, a, b, beta=1.0, alpha=0.0, _lib=L)
    assert np.array_equal(r3, s2.astype(np.float64))


def pin_addmm_rows(L):
    M, K, N = 20, 11, 9
    a, b, s = _rand(M, K), _rand(K, N), _rand(M, N)
    full, fS = oracle.addmm(s, a, b, beta=0.5, alpha=2.0, _lib=L)
    rows = np.array([0, 3, 19, 7], np.int64)
    part, pS = oracle.addmm(s, a, b, beta=0.5, alpha=2.0, rows=rows, _lib=L)
    assert np.array_equal(part, full[rows]) and np.array_equal(pS, fS[rows])


def pin_addmm_fp32_naive_rounds_in_fp32(L):
    # 2^24 + 1 is not an fp32 number: one fp32 accumulator loses the 1 that a
    # wider sum keeps, so the terms 2^24, 1, -2^24 (in k order) sum to 0 in
    # fp32 and to 1 in fp64
    a = np.array([[2.0 ** 24, 1.0, -(2.0 ** 24)]], np.float32)
    b = np.ones((3, 1), np.float32)
    got = oracle.addmm_fp32_naive(np.zeros(1, np.float32), a, b, _lib=L)
    assert got.dtype == np.float32 and got[0, 0] == 0.0, got
    # bit for bit against a sequential loop of np.float32 operations: every
    # product, partial sum and epilogue term rounded to fp32, terms in k order
    M, K, N = 5, 37, 6
    a, b = _rand(M, K), _rand(K, N)
    for self_2d, alpha, beta in [(False, 1.0, 1.0), (True, 2.0, 0.5), (True, -0.75, 1.25)]:
        s = _rand(M, N) if self_2d else _rand(N)
        got = oracle.addmm_fp32_naive(s, a, b, beta=beta, alpha=alpha, _lib=L)
        want = np.empty((M, N), np.float32)
        for i in range(M):
            for j in range(N):
                acc = np.float32(0.0)
                for k in range(K):
                    acc = np.float32(acc + np.float32(a[i, k] * b[k, j]))
                sv = s[i, j] if self_2d else s[j]
                want[i, j] = np.float32(np.float32(beta) * sv) + np.float32(np.float32(alpha) * acc)
        assert np.array_equal(got, want), np.abs(got - want).max()


CONV_SHAPES = [
    # B, IC, H, W, OC, KH, KW, stride, pad, dil
    (2, 3, 7, 7, 4, 3, 3, (1, 1), (1, 1), (1, 1)),
    (2, 3, 5, 5, 4, 3, 3, (2, 2), (2, 2), (2, 2)),
    (1, 2, 9, 6, 3, 2, 3, (2, 1), (0, 2), (1, 2)),
    (2, 3, 7, 7, 4, 1, 1, (1, 1), (0, 0), (1, 1)),
    (1, 3, 16, 16, 5, 7, 7, (4, 4), (3, 3), (1, 1)),
    (1, 1, 4, 5, 2, 5, 4, (3, 2), (1, 0), (1, 1)),
]


def _torch_conv(x, w, b, s, p, d):
    xt = torch.from_numpy(x.astype(np.float64))
    wt = torch.from_numpy(w.astype(np.float64))
    bt = None if b is None else torch.from_numpy(b.astype(np.float64))
    return torch.nn.functional.conv2d(xt, wt, bt, stride=s, padding=p, dilation=d).numpy()


def pin_conv_vs_torch(L):
    for (B, IC, H, W, OC, KH, KW, s, p, d) in CONV_SHAPES:
        x, w, b = _rand(B, IC, H, W), _rand(OC, IC, KH, KW), _rand(OC)
        ref, S = oracle.conv2d(x, w, b, stride=s, padding=p, dilation=d, _lib=L)
        want = _torch_conv(x, w, b, s, p, d)
        assert ref.shape == want.shape, (ref.shape, want.shape)
        np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-12)
        wantS = _torch_conv(np.abs(x), np.abs(w), None, s, p, d)
        np.testing.assert_allclose(S, wantS, rtol=1e-12, atol=1e-12)


def _im2col(x, KH, KW, s, p, d, OH, OW):
    """Materialised im2col [IC*KH*KW, B*OH*OW] built from numpy slicing of a
    zero-padded copy of x (row kk = (ic*KH + kh)*KW + kw, column
    n = (b*OH + oh)*OW + ow)."""
    B, IC, H, W = x.shape
    xp = np.pad(x.astype(np.float64), ((0, 0), (0, 0), (p[0], p[0]), (p[1], p[1])))
    cols = np.empty((IC, KH, KW, B, OH, OW), np.float64)
    for kh in range(KH):
        for kw in range(KW):
            h0, w0 = kh * d[0], kw * d[1]
            cols[:, kh, kw] = xp[:, :, h0:h0 + s[0] * (OH - 1) + 1:s[0],
                                 w0:w0 + s[1] * (OW - 1) + 1:s[1]].transpose(1, 0, 2, 3)
    return cols.reshape(IC * KH * KW, B * OH * OW)


def pin_conv_vs_im2col(L):
    for (B, IC, H, W, OC, KH, KW, s, p, d) in CONV_SHAPES:
        x, w, b = _rand(B, IC, H, W), _rand(OC, IC, KH, KW), _rand(OC)
        ref, _ = oracle.conv2d(x, w, b, stride=s, padding=p, dilation=d, _lib=L)
        _, _, OH, OW = ref.shape
        col = _im2col(x, KH, KW, s, p, d, OH, OW)
        gemm = w.reshape(OC, -1).astype(np.float64) @ col + b.astype(np.float64)[:, None]
        want = gemm.reshape(OC, B, OH, OW).transpose(1, 0, 2, 3)
        np.testing.assert_allclose(ref, want, rtol=1e-12, atol=1e-12)


def pin_conv_1x1_is_addmm(L):
    B, IC, H, W, OC = 2, 5, 4, 6, 3
    x, w, b = _rand(B, IC, H, W), _rand(OC, IC, 1, 1), _rand(OC)
    ref, _ = oracle.conv2d(x, w, b, _lib=L)
    for bi in range(B):
        bias2d = np.repeat(b[:, None], H * W, axis=1)
        mm, _ = oracle.addmm(bias2d, w.reshape(OC, IC), x[bi].reshape(IC, H * W), _lib=L)
        # equal up to fp64 rounding: the conv adds the bias first, addmm last
        np.testing.assert_allclose(ref[bi].reshape(OC, H * W), mm, rtol=1e-13, atol=1e-13)


def pin_conv_padding_zero(L):
    B, IC, H, W, OC = 1, 2, 5, 6, 2
    x, w, b = _rand(B, IC, H, W), _rand(OC, IC, 3, 3), _rand(OC)
    for p, d, s in [((1, 1), (1, 1), (1, 1)), ((2, 3), (2, 1), (1, 2))]:
        r_pad, _ = oracle.conv2d(x, w, b, stride=s, padding=p, dilation=d, _lib=L)
        xp = np.pad(x, ((0, 0), (0, 0), (p[0], p[0]), (p[1], p[1])))
        r_exp, _ = oracle.conv2d(xp, w, b, stride=s, padding=0, dilation=d, _lib=L)
        assert np.array_equal(r_pad, r_exp)


def pin_conv_ones_count(L):
    B, IC, H, W, OC, KH, KW = 1, 3, 6, 5, 1, 3, 3
    x = np.ones((B, IC, H, W), np.float32)
    w = np.ones((OC, IC, KH, KW), np.float32)
    s, p, d = (2, 1), (2, 1), (1, 2)
    ref, _ = oracle.conv2d(x, w, None, stride=s, padding=p, dilation=d, _lib=L)
    # valid taps of (oh, ow): kh with 0 <= oh*sH - pH + kh*dH < H, likewise kw;
    # counted here by listing the covered input rows / columns.
    OH, OW = ref.shape[2:]
    for oh in range(OH):
        rows = [oh * s[0] - p[0] + kh * d[0] for kh in range(KH)]
        nh = sum(0 <= r < H for r in rows)
        for ow in range(OW):
            cols = [ow * s[1] - p[1] + kw * d[1] for kw in range(KW)]
            nw = sum(0 <= c < W for c in cols)
            assert ref[0, 0, oh, ow] == IC * nh * nw


def pin_conv_out_size(L):
    for n in (1, 2, 5, 8, 56, 768):
        for k in (1, 2, 3, 7):
            for st in (1, 2, 4):
                for pd in (0, 1, 3):
                    for dl in (1, 2):
                        got = oracle.conv_out_size(n, k, st, pd, dl, _lib=L)
                        eff = dl * (k - 1) + 1
                        if n + 2 * pd < eff:
                            assert got == -1
                            continue
                        x = torch.zeros(1, 1, n, 1, dtype=torch.float64)
                        w = torch.zeros(1, 1, k, 1, dtype=torch.float64)
                        want = torch.nn.functional.conv2d(x, w, stride=(st, 1), padding=(pd, 0),
                                                          dilation=(dl, 1)).shape[2]
                        assert got == want, (n, k, st, pd, dl, got, want)


def pin_conv_channels(L):
    B, IC, H, W, OC = 2, 3, 5, 5, 6
    x, w, b = _rand(B, IC, H, W), _rand(OC, IC, 3, 3), _rand(OC)
    full, fS = oracle.conv2d(x, w, b, padding=1, _lib=L)
    ch = np.array([5, 0, 2], np.int64)
    part, pS = oracle.conv2d(x, w, b, padding=1, channels=ch, _lib=L)
    assert np.array_equal(part, full[:, ch]) and np.array_equal(pS, fS[:, ch])


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.lib())


def test_bound_reachable_by_plain_fp32():
    """A naive fp32 loop meets |out - ref| <= 1e-5*S + 1e-6 on the tiny
    workloads and on rows of the transformer-linear workloads, so the bound is
    not tighter than plain fp32 arithmetic."""
    for name in ("tiny_selfN", "tiny_selfMN", "linear_M1024_K3072_N768",
                 "linear_M577_K768_N3072"):
        c, s, a, b = synth.make_addmm_case(name)
        a = a[:48]
        s = s[:48] if c["self_2d"] else s
        ref, S = oracle.addmm(s, a, b, beta=c["beta"], alpha=c["alpha"])
        got = oracle.addmm_fp32_naive(s, a, b, beta=c["beta"], alpha=c["alpha"])
        ratio = np.abs(got - ref) / (1e-5 * S + 1e-6)
        assert ratio.max() <= 1.0, (name, ratio.max())


def test_oracle_rejects_bad_arguments():
    L = oracle.lib()
    with pytest.raises(oracle.OracleError):
        oracle.addmm(_rand(3), _rand(2, 3), _rand(4, 3))
    with pytest.raises(oracle.OracleError):
        oracle.addmm(_rand(3), _rand(2, 3), _rand(3, 3), rows=[5])
    with pytest.raises(oracle.OracleError):
        oracle.conv2d(_rand(1, 1, 2, 2), _rand(1, 1, 5, 5))
    assert oracle.conv_out_size(4, 3, 0, 0, 1, _lib=L) == -1


def test_synth_streams_are_distinct_and_stable():
    k1, k2 = synth.stream_key(0, 1, 1), synth.stream_key(0, 1, 2)
    assert k1 != k2
    u = synth.uniform(k1, 1000, -1, 1)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 0.1
    assert np.array_equal(u, synth.uniform(k1, 1000, -1, 1))
    z = synth.normal(k2, 200000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    rows = synth.sample_rows(k1, 8192, 256)
    assert len(np.unique(rows)) == 256 and rows.min() >= 0 and rows.max() < 8192


PLANTS = {1: "addmm subtracts products", 2: "addmm drops beta*self",
          3: "addmm ignores self_2d", 4: "conv uses dH on the width axis",
          5: "conv drops the bias", 6: "conv shifts ih by one",
          7: "conv output size misses -1", 8: "S sums signed products",
          9: "fp32 loop accumulates in fp64"}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=lambda n: PLANTS[n].replace(" ", "_"))
def test_planted_mistakes_are_caught(plant):
    with tempfile.TemporaryDirectory() as d:
        path = oracle.build(force=True, extra_flags=[f"-DORACLE_PLANT={plant}"],
                            out_path=os.path.join(d, f"liboracle_plant{plant}.so"))
        L = oracle.load_variant(path)
        failed = []
        for pin in PINS:
            try:
                pin(L)
            except (AssertionError, oracle.OracleError, ValueError):
                failed.append(pin.__name__)
        assert failed, f"no pin caught planted mistake {plant}: {PLANTS[plant]}"
