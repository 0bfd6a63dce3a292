"""The autograd layers (AMDense, AMConv2d, AMAttention): forward outputs and
the gradients torch's autograd delivers, checked against the oracle element
by element.  A contraction that reads an earlier one's result (attention's
P V, the gradients through the softmax) is checked on the GPU's own copy of
that result, computed here through the same ABI calls."""
import numpy as np
import pytest

from gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def host(t):
    return t.detach().cpu().numpy()


def test_am_dense_forward_and_gradients(amd, orc, luts):
    import torch
    from approximate_multiplier_dnn_gb300.layers import AMDense
    g = torch.Generator().manual_seed(3)
    lut = luts("mitchell", 7)
    layer = AMDense(784, 100, lut, bias=False, generator=g)
    X = torch.randn((256, 784), generator=g).cuda().requires_grad_()
    y = layer(X)
    dy = torch.randn((256, 100), generator=g).cuda() * 0.01
    y.backward(dy)
    torch.cuda.synchronize()
    x, W, d = host(X), host(layer.weight), host(dy)
    ref, sa = orc.gemm("mitchell", 7, x, W)
    assert_close(host(y), ref, sa, "y")
    ref, sa = orc.gemm("mitchell", 7, d, W, transB=True)
    assert_close(host(X.grad), ref, sa, "dX")
    ref, sa = orc.gemm("mitchell", 7, x, d, transA=True)
    assert_close(host(layer.weight.grad), ref, sa, "dW")


def test_am_dense_bias_and_chain(amd, orc, luts):
    """Bias adds exactly after the approximate product; a two-layer chain's
    input gradient flows through both layers' approximate contractions."""
    import torch
    from approximate_multiplier_dnn_gb300.layers import AMDense, am_dense
    g = torch.Generator().manual_seed(4)
    lut = luts("exact", 7)
    l1 = AMDense(64, 48, lut, bias=True, generator=g)
    l2 = AMDense(48, 10, lut, bias=False, generator=g)
    with torch.no_grad():
        l1.bias.copy_(torch.randn(48, generator=g).cuda())
    X = torch.randn((32, 64), generator=g).cuda().requires_grad_()
    h = l1(X)
    h.retain_grad()
    assert torch.equal(h.detach(), am_dense(X.detach(), l1.weight.detach(), lut) + l1.bias.detach())
    out = l2(h)
    dout = torch.randn((32, 10), generator=g).cuda()
    out.backward(dout)
    torch.cuda.synchronize()
    # dh = dout W2^T (approximate); dX = dh W1^T on the gradient the layer received
    ref, sa = orc.gemm("exact", 7, host(dout), host(l2.weight), transB=True)
    assert_close(host(h.grad), ref, sa, "dh")
    ref, sa = orc.gemm("exact", 7, host(h.grad), host(l1.weight), transB=True)
    assert_close(host(X.grad), ref, sa, "dX")
    assert np.allclose(host(l1.bias.grad), host(h.grad).sum(0), rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("geom", [dict(N=4, H=12, W=12, C=16, K=24, R=3, S=3, stride=1, pad=1, dil=1),
                                  dict(N=2, H=11, W=9, C=8, K=16, R=3, S=2, stride=2, pad=1, dil=2)])
def test_am_conv2d_forward_and_gradients(amd, orc, luts, geom):
    import torch
    from approximate_multiplier_dnn_gb300.layers import AMConv2d
    g = torch.Generator().manual_seed(5)
    lut = luts("mitchell", 7)
    G = geom
    layer = AMConv2d(G["C"], G["K"], (G["R"], G["S"]), lut, stride=G["stride"], padding=G["pad"],
                     dilation=G["dil"], bias=False, generator=g)
    X = torch.randn((G["N"], G["H"], G["W"], G["C"]), generator=g).cuda().requires_grad_()
    y = layer(X)
    dy = torch.randn(tuple(y.shape), generator=g).cuda() * 0.01
    y.backward(dy)
    torch.cuda.synchronize()
    st, pd, dl = (G["stride"],) * 2, (G["pad"],) * 2, (G["dil"],) * 2
    desc = orc.conv_desc(G["N"], G["H"], G["W"], G["C"], G["K"], G["R"], G["S"], st, pd, dl)
    x, w, d = host(X), host(layer.weight), host(dy)
    ref, sa = orc.conv2d_fwd("mitchell", 7, desc, x, w, np.arange(y.numel()))
    assert_close(host(y).reshape(-1), ref, sa, "y")
    ref, sa = orc.conv2d_bwd_data("mitchell", 7, desc, d, w, np.arange(X.numel()))
    assert_close(host(X.grad).reshape(-1), ref, sa, "dX")
    ref, sa = orc.conv2d_bwd_filter("mitchell", 7, desc, x, d, np.arange(w.size))
    assert_close(host(layer.weight.grad).reshape(-1), ref, sa, "dW")


@pytest.mark.parametrize("geom", [
    dict(N=2, H=9, W=70, C=20, D=1, R=3, S=3, stride=1, pad=1, dil=1),    # tiled kernel
    dict(N=2, H=10, W=9, C=6, D=2, R=3, S=3, stride=2, pad=1, dil=1),     # direct kernel, multiplier 2
])
def test_am_depthwise_conv2d_forward_and_gradients(amd, orc, luts, geom):
    """AMDepthwiseConv2d: output and both autograd gradients against the
    oracle's depthwise sums; the bias is added exactly."""
    import torch
    from approximate_multiplier_dnn_gb300.layers import AMDepthwiseConv2d, am_depthwise_conv2d
    g = torch.Generator().manual_seed(6)
    lut = luts("mitchell", 7)
    G = geom
    layer = AMDepthwiseConv2d(G["C"], (G["R"], G["S"]), lut, depth_multiplier=G["D"], stride=G["stride"],
                              padding=G["pad"], dilation=G["dil"], bias=True, generator=g)
    with torch.no_grad():
        layer.bias.copy_(torch.randn(layer.bias.shape, generator=g).cuda())
    X = torch.randn((G["N"], G["H"], G["W"], G["C"]), generator=g).cuda().requires_grad_()
    y = layer(X)
    dy = torch.randn(tuple(y.shape), generator=g).cuda() * 0.01
    y.backward(dy)
    torch.cuda.synchronize()
    st, pd, dl = (G["stride"],) * 2, (G["pad"],) * 2, (G["dil"],) * 2
    K = G["C"] * G["D"]
    desc = orc.conv_desc(G["N"], G["H"], G["W"], G["C"], K, G["R"], G["S"], st, pd, dl)
    x, w, d = host(X), host(layer.weight), host(dy)
    y0 = am_depthwise_conv2d(X.detach(), layer.weight.detach(), lut, G["stride"], G["pad"], G["dil"])
    assert torch.equal(y.detach(), y0 + layer.bias.detach())
    ref, sa = orc.dwconv2d_fwd("mitchell", 7, desc, x, w, np.arange(y.numel()))
    assert_close(host(y0).reshape(-1), ref, sa, "y")
    ref, sa = orc.dwconv2d_bwd_data("mitchell", 7, desc, d, w, np.arange(X.numel()))
    assert_close(host(X.grad).reshape(-1), ref, sa, "dX")
    ref, sa = orc.dwconv2d_bwd_filter("mitchell", 7, desc, x, d, np.arange(w.size))
    assert_close(host(layer.weight.grad).reshape(-1), ref, sa, "dW")
    assert np.allclose(host(layer.bias.grad), d.reshape(-1, K).sum(0), rtol=1e-5, atol=1e-6)


def test_softmax_rows_backward_kernel(amd, orc):
    import torch
    rng = np.random.default_rng(8)
    S = rng.standard_normal((300, 77)).astype(np.float32)
    dP = rng.standard_normal((300, 77)).astype(np.float32)
    P = orc.softmax_rows(S).astype(np.float32)
    dPd, Pd = torch.from_numpy(dP).cuda(), torch.from_numpy(P).cuda()
    dS = torch.empty_like(dPd)
    amd.amsim_softmax_rows_backward(Pd, dPd, dS, 300, 77)
    torch.cuda.synchronize()
    ref = orc.softmax_rows_backward(P, dP)
    # fp32: one dot product of 77 terms and a product per element
    bound = 1e-6 * (np.abs(P) * (np.abs(dP) + (np.abs(P) * np.abs(dP)).sum(1, keepdims=True)) + 1e-30)
    assert np.all(np.abs(host(dS) - ref) <= bound * 8)


def test_am_attention_forward_and_gradients(amd, orc, luts):
    import torch
    from approximate_multiplier_dnn_gb300.layers import am_attention
    g = torch.Generator().manual_seed(6)
    lut = luts("mitchell", 7)
    b, h, s, d = 2, 3, 64, 32
    scale = 1.0 / np.sqrt(d)
    Q, K, V = (torch.randn((b, h, s, d), generator=g).cuda().requires_grad_() for _ in range(3))
    O = am_attention(Q, K, V, lut)
    dO = torch.randn((b, h, s, d), generator=g).cuda() * 0.1
    O.backward(dO)
    torch.cuda.synchronize()
    # the GPU's own intermediates, through the same calls (and scratch sizes,
    # hence the same plans and summation orders) the layer uses
    ws = amd.workspace(amd.amsim_gemm_workspace_size("N", "T", s, s, d, b * h, lut))
    Sg = torch.empty((b * h, s, s), device="cuda")
    amd.amsim_gemm_strided_batched("N", "T", s, s, d, scale, Q.detach(), d, s * d, K.detach(), d, s * d, 0.0, Sg,
                                   s, s * s, b * h, lut, ws=ws)
    Pg = torch.empty_like(Sg)
    amd.amsim_softmax_rows(Sg, Pg, b * h * s, s)
    dPg = torch.empty_like(Sg)
    amd.amsim_gemm_strided_batched("N", "T", s, s, d, 1.0, dO, d, s * d, V.detach(), d, s * d, 0.0, dPg, s, s * s,
                                   b * h, lut, ws=ws)
    dSg = torch.empty_like(Sg)
    amd.amsim_softmax_rows_backward(Pg, dPg, dSg, b * h * s, s)
    torch.cuda.synchronize()
    q, k, v, do = (host(t).reshape(b * h, s, d) for t in (Q, K, V, dO))
    P, dS = host(Pg), host(dSg)
    o, dq, dk, dv = (host(t).reshape(b * h, s, d) for t in (O, Q.grad, K.grad, V.grad))
    for i in range(b * h):
        ref, sa = orc.attention_scores("mitchell", 7, q[i], k[i], scale)
        assert_close(host(Sg)[i], ref, scale * sa, "S")
        ref, sa = orc.gemm("mitchell", 7, P[i], v[i])
        assert_close(o[i], ref, sa, "O")
        ref, sa = orc.gemm("mitchell", 7, P[i], do[i], transA=True)
        assert_close(dv[i], ref, sa, "dV")
        ref, sa = orc.gemm("mitchell", 7, dS[i], k[i], alpha=scale)
        assert_close(dq[i], ref, scale * sa, "dQ")
        ref, sa = orc.gemm("mitchell", 7, dS[i], q[i], transA=True, alpha=scale)
        assert_close(dk[i], ref, scale * sa, "dK")
