"""Pins of the CPU oracle's contractions (Dense GEMMs, Conv2D forward / weight
gradient / preceding-layer gradient of the ApproxTrain page, Sec. VI-B/C,
Algorithms 3 and 4) against library routines that share nothing with it.

With the exact kind at M = 11 and operands that carry at most 11 fraction bits
and safe exponents, every AMSim product equals the real product, so the
contraction must equal a float64 library contraction of the same operands
(numpy matmul; torch CPU conv2d and its two gradients) up to double rounding.
This fixes the indexing (transposes, leading dimensions, alpha/beta, padding,
stride, dilation, the rot180/transpose of the preceding-layer gradient, the
im2col of the weight gradient).  A Mitchell case is brute-forced on tiny shapes
from elementwise products, and the attention softmax is checked against scipy.
"""
import math

import numpy as np
import pytest


def short_mantissa(shape, rng, bits=11, scale_exp=(-3, 3), zero_frac=0.05):
    """fp32 values with at most `bits` fraction bits and moderate exponents."""
    sig = rng.integers(-(1 << (bits + 1)) + 1, 1 << (bits + 1), size=shape)
    e = rng.integers(scale_exp[0], scale_exp[1] + 1, size=shape)
    v = np.ldexp(sig.astype(np.float64), (e - bits).astype(np.int32))
    v[rng.random(shape) < zero_frac] = 0.0
    return v.astype(np.float32)


def close(got, ref, sumabs, rel=1e-12):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = rel * np.asarray(sumabs) + 1e-300
    return np.all(np.abs(got - ref) <= tol + np.abs(ref) * 2.0 ** -24)


@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
def test_gemm_exact_kind_equals_float64_matmul(orc, ta, tb):
    rng = np.random.default_rng(11)
    m, n, k = 17, 33, 31
    A = short_mantissa((k, m) if ta else (m, k), rng)
    B = short_mantissa((n, k) if tb else (k, n), rng)
    C0 = short_mantissa((m, n), rng)
    alpha, beta = 0.5, -2.0
    out, sa = orc.gemm("exact", 11, A, B, transA=ta, transB=tb, alpha=alpha, beta=beta, C0=C0)
    Ad = A.astype(np.float64).T if ta else A.astype(np.float64)
    Bd = B.astype(np.float64).T if tb else B.astype(np.float64)
    ref = alpha * (Ad @ Bd) + beta * C0.astype(np.float64)
    # the oracle rounds once to fp32 at the end
    assert np.array_equal(out, ref.astype(np.float32)) or close(out, ref, abs(alpha) * sa + abs(beta * C0))
    assert np.allclose(sa, np.abs(Ad) @ np.abs(Bd), rtol=1e-14, atol=0)


def test_gemm_row_subset(orc):
    rng = np.random.default_rng(12)
    A = rng.standard_normal((20, 9)).astype(np.float32)
    B = rng.standard_normal((9, 7)).astype(np.float32)
    full, _ = orc.gemm("mitchell", 7, A, B)
    rows = np.array([19, 0, 7, 7])
    part, _ = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert np.array_equal(part, full[rows])


def test_gemm_mitchell_brute_force_tiny(orc):
    rng = np.random.default_rng(13)
    A = rng.standard_normal((3, 5)).astype(np.float32)
    B = rng.standard_normal((5, 4)).astype(np.float32)
    out, sa = orc.gemm("mitchell", 7, A, B)
    for i in range(3):
        for j in range(4):
            prods = orc.mul("mitchell", 7, A[i, :], B[:, j]).astype(np.float64)
            assert out[i, j] == np.float32(math.fsum(prods))
            assert sa[i, j] == pytest.approx(np.abs(prods).sum(), rel=1e-15)


def test_gemm_empty_k_gives_beta_term(orc):
    A = np.zeros((4, 0), np.float32)
    B = np.zeros((0, 3), np.float32)
    C0 = np.arange(12, dtype=np.float32).reshape(4, 3)
    out, sa = orc.gemm("exact", 7, A, B, beta=1.0, C0=C0)
    assert np.array_equal(out, C0) and np.all(sa == 0)


# ------------------------------------------------------------------ conv
GEOMS = [
    # N, H, W, C, K, R, S, stride, pad, dil
    (2, 7, 6, 3, 4, 3, 3, (1, 1), (1, 1), (1, 1)),
    (1, 9, 8, 2, 5, 3, 2, (2, 1), (1, 0), (1, 1)),
    (2, 8, 9, 3, 2, 3, 3, (1, 2), (2, 2), (2, 1)),
    (1, 5, 5, 4, 3, 1, 1, (1, 1), (0, 0), (1, 1)),
    (1, 10, 7, 2, 3, 2, 3, (3, 2), (1, 2), (1, 2)),
]


def _torch():
    return pytest.importorskip("torch")


@pytest.mark.parametrize("g", GEOMS)
def test_conv_exact_kind_equals_torch_float64(orc, g):
    torch = _torch()
    import torch.nn.functional as F
    N, H, W, C, K, R, S, st, pd, dl = g
    rng = np.random.default_rng(sum(g[:7]))
    desc = orc.conv_desc(N, H, W, C, K, R, S, st, pd, dl)
    P, Q = orc.conv_out_hw(desc)
    x = short_mantissa((N, H, W, C), rng)
    w = short_mantissa((R, S, C, K), rng)
    dy = short_mantissa((N, P, Q, K), rng)
    xt = torch.from_numpy(x.astype(np.float64)).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w.astype(np.float64)).permute(3, 2, 0, 1)       # K C R S
    dyt = torch.from_numpy(dy.astype(np.float64)).permute(0, 3, 1, 2)

    yref = F.conv2d(xt, wt, stride=st, padding=pd, dilation=dl).permute(0, 2, 3, 1).numpy()
    assert yref.shape == (N, P, Q, K)
    pts = np.arange(yref.size)
    y, sa = orc.conv2d_fwd("exact", 11, desc, x, w, pts)
    assert close(y, yref.reshape(-1), sa)

    dxref = torch.nn.grad.conv2d_input((N, C, H, W), wt, dyt, stride=st, padding=pd,
                                       dilation=dl).permute(0, 2, 3, 1).numpy()
    dx, sa = orc.conv2d_bwd_data("exact", 11, desc, dy, w, np.arange(dxref.size))
    assert close(dx, dxref.reshape(-1), sa)

    dwref = torch.nn.grad.conv2d_weight(xt, (K, C, R, S), dyt, stride=st, padding=pd,
                                        dilation=dl).permute(2, 3, 1, 0).numpy()
    dw, sa = orc.conv2d_bwd_filter("exact", 11, desc, x, dy, np.arange(dwref.size))
    assert close(dw, dwref.reshape(-1), sa)


def test_conv1x1_equals_gemm(orc):
    rng = np.random.default_rng(21)
    N, H, W, C, K = 2, 4, 3, 5, 6
    x = rng.standard_normal((N, H, W, C)).astype(np.float32)
    w = rng.standard_normal((1, 1, C, K)).astype(np.float32)
    desc = orc.conv_desc(N, H, W, C, K, 1, 1)
    y, _ = orc.conv2d_fwd("mitchell", 7, desc, x, w, np.arange(N * H * W * K))
    g, _ = orc.gemm("mitchell", 7, x.reshape(-1, C), w.reshape(C, K))
    assert np.array_equal(y, g.reshape(-1))
    dy = rng.standard_normal((N, H, W, K)).astype(np.float32)
    dx, _ = orc.conv2d_bwd_data("mitchell", 7, desc, dy, w, np.arange(N * H * W * C))
    g2, _ = orc.gemm("mitchell", 7, dy.reshape(-1, K), w.reshape(C, K), transB=True)
    assert np.array_equal(dx, g2.reshape(-1))
    dw, _ = orc.conv2d_bwd_filter("mitchell", 7, desc, x, dy, np.arange(C * K))
    g3, _ = orc.gemm("mitchell", 7, x.reshape(-1, C), dy.reshape(-1, K), transA=True)
    assert np.array_equal(dw, g3.reshape(-1))


def test_conv_rejects_bad_descriptor(orc):
    desc = orc.conv_desc(1, 2, 2, 1, 1, 5, 5)     # filter larger than padded input
    with pytest.raises(ValueError):
        orc.conv_out_hw(desc)


# ------------------------------------------------------------------ attention
def test_softmax_matches_scipy(orc):
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(31)
    S = (rng.standard_normal((6, 40)) * 5).astype(np.float32)
    P = orc.softmax_rows(S)
    assert np.allclose(P, sp.softmax(S.astype(np.float64), axis=-1), rtol=1e-14, atol=1e-16)
    assert np.allclose(P.sum(axis=-1), 1.0, rtol=1e-15)


def test_attention_scores_scale_exact(orc):
    rng = np.random.default_rng(32)
    Qm = short_mantissa((8, 16), rng)
    Km = short_mantissa((10, 16), rng)
    S, sa = orc.attention_scores("exact", 11, Qm, Km, 0.125)
    ref = 0.125 * (Qm.astype(np.float64) @ Km.astype(np.float64).T)
    assert close(S, ref, 0.125 * sa)


def test_softmax_backward_matches_finite_differences():
    """The softmax gradient reference equals the derivative of the softmax,
    taken by central differences of the double softmax."""
    import oracle as orc
    rng = np.random.default_rng(71)
    S = rng.standard_normal((5, 9))
    dP = rng.standard_normal((5, 9))
    dS = orc.softmax_rows_backward(orc.softmax_rows(S), dP)
    h = 1e-6
    num = np.empty_like(S)
    for r in range(S.shape[0]):
        for c in range(S.shape[1]):
            Sp, Sm = S.copy(), S.copy()
            Sp[r, c] += h
            Sm[r, c] -= h
            num[r, c] = ((orc.softmax_rows(Sp) - orc.softmax_rows(Sm))[r] * dP[r]).sum() / (2 * h)
    assert np.allclose(dS, num, rtol=1e-6, atol=1e-9)
    # rows of dS sum to zero (the softmax's outputs sum to one)
    assert np.allclose(dS.sum(axis=1), 0.0, atol=1e-12)


# ------------------------------------------------------------------ depthwise conv
DW_GEOMS = [
    # N, H, W, C, D, R, S, stride, pad, dil
    (2, 7, 6, 3, 1, 3, 3, (1, 1), (1, 1), (1, 1)),
    (1, 9, 8, 2, 3, 3, 2, (2, 1), (1, 0), (1, 1)),
    (2, 8, 9, 4, 2, 3, 3, (1, 2), (2, 2), (2, 1)),
    (1, 10, 7, 3, 1, 5, 3, (3, 2), (2, 2), (1, 2)),
    (1, 5, 5, 5, 1, 1, 1, (1, 1), (0, 0), (1, 1)),
]


@pytest.mark.parametrize("g", DW_GEOMS)
def test_dwconv_exact_kind_equals_torch_grouped_float64(orc, g):
    """Depthwise = torch's grouped convolution with one group per input channel
    (weight [C*D, 1, R, S], output channel c*D + d reads channel c)."""
    torch = _torch()
    import torch.nn.functional as F
    N, H, W, C, D, R, S, st, pd, dl = g
    K = C * D
    rng = np.random.default_rng(100 + sum(g[:7]))
    desc = orc.conv_desc(N, H, W, C, K, R, S, st, pd, dl)
    P, Q = orc.conv_out_hw(desc)
    x = short_mantissa((N, H, W, C), rng)
    w = short_mantissa((R, S, C, D), rng)
    dy = short_mantissa((N, P, Q, K), rng)
    xt = torch.from_numpy(x.astype(np.float64)).permute(0, 3, 1, 2)
    wt = torch.from_numpy(w.astype(np.float64)).reshape(R, S, K).permute(2, 0, 1).unsqueeze(1)  # K 1 R S
    dyt = torch.from_numpy(dy.astype(np.float64)).permute(0, 3, 1, 2)

    yref = F.conv2d(xt, wt, stride=st, padding=pd, dilation=dl, groups=C).permute(0, 2, 3, 1).numpy()
    assert yref.shape == (N, P, Q, K)
    y, sa = orc.dwconv2d_fwd("exact", 11, desc, x, w, np.arange(yref.size))
    assert close(y, yref.reshape(-1), sa)

    dxref = torch.nn.grad.conv2d_input((N, C, H, W), wt, dyt, stride=st, padding=pd, dilation=dl,
                                       groups=C).permute(0, 2, 3, 1).numpy()
    dx, sa = orc.dwconv2d_bwd_data("exact", 11, desc, dy, w, np.arange(dxref.size))
    assert close(dx, dxref.reshape(-1), sa)

    dwref = torch.nn.grad.conv2d_weight(xt, (K, 1, R, S), dyt, stride=st, padding=pd, dilation=dl,
                                        groups=C)                                           # K 1 R S
    dwref = dwref[:, 0].permute(1, 2, 0).numpy()                                            # R S K = R S C D
    dw, sa = orc.dwconv2d_bwd_filter("exact", 11, desc, x, dy, np.arange(dwref.size))
    assert close(dw, dwref.reshape(-1), sa)


def test_dwconv_single_channel_equals_conv(orc):
    """With one input channel the depthwise sums are the ordinary Conv2D sums
    (K = D output channels), Mitchell products included."""
    rng = np.random.default_rng(41)
    N, H, W, D, R, S = 2, 6, 5, 3, 3, 2
    desc = orc.conv_desc(N, H, W, 1, D, R, S, (2, 1), (1, 1), (1, 2))
    P, Q = orc.conv_out_hw(desc)
    x = rng.standard_normal((N, H, W, 1)).astype(np.float32)
    w = rng.standard_normal((R, S, 1, D)).astype(np.float32)
    dy = rng.standard_normal((N, P, Q, D)).astype(np.float32)
    for dwf, cf, a, b, size in ((orc.dwconv2d_fwd, orc.conv2d_fwd, x, w, N * P * Q * D),
                                (orc.dwconv2d_bwd_data, orc.conv2d_bwd_data, dy, w, N * H * W),
                                (orc.dwconv2d_bwd_filter, orc.conv2d_bwd_filter, x, dy, R * S * D)):
        got, sa = dwf("mitchell", 7, desc, a, b, np.arange(size))
        ref, sr = cf("mitchell", 7, desc, a, b, np.arange(size))
        assert np.array_equal(got, ref) and np.array_equal(sa, sr)


def test_dwconv_channels_are_independent(orc):
    """Each output channel of a depthwise convolution equals a one-channel
    convolution of its own input channel with its own filter slice."""
    rng = np.random.default_rng(42)
    N, H, W, C, D, R, S = 1, 5, 6, 3, 2, 3, 3
    desc = orc.conv_desc(N, H, W, C, C * D, R, S, (1, 1), (1, 1), (1, 1))
    P, Q = orc.conv_out_hw(desc)
    x = rng.standard_normal((N, H, W, C)).astype(np.float32)
    w = rng.standard_normal((R, S, C, D)).astype(np.float32)
    y, _ = orc.dwconv2d_fwd("mitchell", 7, desc, x, w, np.arange(N * P * Q * C * D))
    y = y.reshape(N, P, Q, C, D)
    d1 = orc.conv_desc(N, H, W, 1, D, R, S, (1, 1), (1, 1), (1, 1))
    for c in range(C):
        ref, _ = orc.conv2d_fwd("mitchell", 7, d1, x[..., c:c + 1], w[:, :, c:c + 1, :], np.arange(N * P * Q * D))
        assert np.array_equal(y[..., c, :].reshape(-1), ref)


def test_dwconv_rejects_channels_not_dividing(orc):
    desc = orc.conv_desc(1, 4, 4, 3, 4, 3, 3, (1, 1), (1, 1), (1, 1))
    with pytest.raises(ValueError):
        orc.dwconv2d_fwd("exact", 7, desc, np.zeros((1, 4, 4, 3), np.float32),
                         np.zeros((3, 3, 3, 1), np.float32), np.arange(4))
