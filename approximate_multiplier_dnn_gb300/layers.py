"""Drop-in torch layers whose contractions -- the forward pass and both
gradients -- run through the LUT-simulated approximate multiplier, as the
AMDENSE and AMCONV2D layers of ApproxTrain (Sec. IV) do, plus attention built
from two approximate contractions around an exact softmax.

Each layer is a torch.autograd.Function over the C ABI: the approximate
contractions, the softmax and its gradient run in this library's kernels; bias
additions are ordinary (exact) torch additions, as they are not products.

Layouts: Dense weights are [in, out] (y = x w); Conv2D tensors are NHWC with
RSCK filters (TF's HWIO), stride/padding/dilation as in ApproxTrain's Conv2D;
depthwise filters are R x S x C x D (TF's depthwise layout, multiplier D);
attention takes Q, K, V as [batch, heads, seq, dim].

Operand order of every contraction (which operand indexes the LUT's rows;
it matters only for an asymmetric user LUT): Dense forward (x, w), input
gradient (dy, w), weight gradient (x, dy); Conv2D likewise (x, w), (dy, w),
(x, dy), and the same for depthwise; attention S = (q, k), O = (p, v), dV = (p, dO), dP = (dO, v),
dQ = (dS, k), dK = (dS, q).
"""
from __future__ import annotations

import math

import torch

from . import (ConvDesc, amsim_conv2d_bwd_data, amsim_conv2d_bwd_filter, amsim_conv2d_fwd, amsim_conv2d_out_hw,
               amsim_conv2d_workspace_size, amsim_dwconv2d_bwd_data, amsim_dwconv2d_bwd_filter, amsim_dwconv2d_fwd,
               amsim_dwconv2d_workspace_size, amsim_gemm, amsim_gemm_strided_batched, amsim_gemm_workspace_size,
               amsim_softmax_rows, amsim_softmax_rows_backward, workspace)


def _f32(t: torch.Tensor) -> torch.Tensor:
    if t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError("approximate layers take fp32 CUDA tensors")
    return t.contiguous()


def _gemm(tA: str, tB: str, A: torch.Tensor, B: torch.Tensor, m: int, n: int, k: int, lut, alpha=1.0):
    """C[m, n] = alpha op(A) op(B) for contiguous row-major A and B."""
    C = torch.empty((m, n), dtype=torch.float32, device=A.device)
    ws = workspace(amsim_gemm_workspace_size(tA, tB, m, n, k, 1, lut), A.device)
    amsim_gemm(tA, tB, m, n, k, alpha, A, max(1, A.shape[1]), B, max(1, B.shape[1]), 0.0, C, max(1, n), lut,
               ws=ws)
    return C


def _bgemm(tA: str, tB: str, A: torch.Tensor, B: torch.Tensor, m: int, n: int, k: int, lut, alpha=1.0):
    """C[b] = alpha op(A[b]) op(B[b]) over the leading batch dimension."""
    batch = A.shape[0]
    C = torch.empty((batch, m, n), dtype=torch.float32, device=A.device)
    ws = workspace(amsim_gemm_workspace_size(tA, tB, m, n, k, batch, lut), A.device)
    amsim_gemm_strided_batched(tA, tB, m, n, k, alpha, A, A.shape[2], A.shape[1] * A.shape[2], B, B.shape[2],
                               B.shape[1] * B.shape[2], 0.0, C, n, m * n, batch, lut, ws=ws)
    return C


# ------------------------------------------------------------------ Dense
class _DenseFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, lut):
        x, w = _f32(x), _f32(w)
        rows, fin = x.shape
        fout = w.shape[1]
        ctx.save_for_backward(x, w)
        ctx.lut = lut
        return _gemm("N", "N", x, w, rows, fout, fin, lut)

    @staticmethod
    def backward(ctx, dy):
        x, w = ctx.saved_tensors
        dy = _f32(dy)
        rows, fin = x.shape
        fout = w.shape[1]
        dx = _gemm("N", "T", dy, w, rows, fin, fout, ctx.lut) if ctx.needs_input_grad[0] else None
        dw = _gemm("T", "N", x, dy, fin, fout, rows, ctx.lut) if ctx.needs_input_grad[1] else None
        return dx, dw, None


def am_dense(x: torch.Tensor, w: torch.Tensor, lut) -> torch.Tensor:
    """y = x w with approximate products (x [rows, in], w [in, out])."""
    return _DenseFn.apply(x, w, lut)


class AMDense(torch.nn.Module):
    """Fully connected layer y = x W (+ b) whose forward and backward
    contractions use the approximate multiplier (ApproxTrain's AMDENSE)."""

    def __init__(self, in_features: int, out_features: int, lut, bias: bool = True, device="cuda",
                 generator: torch.Generator | None = None):
        super().__init__()
        self.lut = lut
        bound = math.sqrt(6.0 / (in_features + out_features))          # Glorot uniform
        w = (torch.rand((in_features, out_features), generator=generator) * 2.0 - 1.0) * bound
        self.weight = torch.nn.Parameter(w.to(device))
        self.bias = torch.nn.Parameter(torch.zeros(out_features, device=device)) if bias else None

    def forward(self, x):
        y = am_dense(x, self.weight, self.lut)
        return y + self.bias if self.bias is not None else y


# ------------------------------------------------------------------ Conv2D
def _pair(v):
    return (v, v) if isinstance(v, int) else tuple(v)


class _Conv2dFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, lut, stride, padding, dilation):
        x, w = _f32(x), _f32(w)
        N, H, W, C = x.shape
        R, S, C2, K = w.shape
        if C2 != C:
            raise ValueError("filter channels differ from the input's")
        desc = ConvDesc.make(N, H, W, C, K, R, S, stride, padding, dilation)
        P, Q = amsim_conv2d_out_hw(desc)
        y = torch.empty((N, P, Q, K), dtype=torch.float32, device=x.device)
        amsim_conv2d_fwd(desc, x, w, y, lut, ws=workspace(amsim_conv2d_workspace_size(desc, 0, lut), x.device))
        ctx.save_for_backward(x, w)
        ctx.lut, ctx.desc = lut, desc
        return y

    @staticmethod
    def backward(ctx, dy):
        x, w = ctx.saved_tensors
        dy = _f32(dy)
        desc, lut = ctx.desc, ctx.lut
        dx = dw = None
        if ctx.needs_input_grad[0]:
            dx = torch.empty_like(x)
            amsim_conv2d_bwd_data(desc, dy, w, dx, lut,
                                  ws=workspace(amsim_conv2d_workspace_size(desc, 1, lut), x.device))
        if ctx.needs_input_grad[1]:
            dw = torch.empty_like(w)
            amsim_conv2d_bwd_filter(desc, x, dy, dw, lut,
                                    ws=workspace(amsim_conv2d_workspace_size(desc, 2, lut), x.device))
        return dx, dw, None, None, None, None


def am_conv2d(x, w, lut, stride=1, padding=0, dilation=1):
    """y = conv2d(x, w) with approximate products (x NHWC, w RSCK, y NPQK)."""
    return _Conv2dFn.apply(x, w, lut, _pair(stride), _pair(padding), _pair(dilation))


class AMConv2d(torch.nn.Module):
    """2-D convolution (cross-correlation) whose forward pass and both
    gradients use the approximate multiplier (ApproxTrain's AMCONV2D).
    NHWC input, RSCK filters."""

    def __init__(self, in_channels: int, out_channels: int, kernel_size, lut, stride=1, padding=0, dilation=1,
                 bias: bool = True, device="cuda", generator: torch.Generator | None = None):
        super().__init__()
        self.lut = lut
        R, S = _pair(kernel_size)
        self.stride, self.padding, self.dilation = _pair(stride), _pair(padding), _pair(dilation)
        std = math.sqrt(2.0 / (R * S * in_channels))                   # He normal
        w = torch.randn((R, S, in_channels, out_channels), generator=generator) * std
        self.weight = torch.nn.Parameter(w.to(device))
        self.bias = torch.nn.Parameter(torch.zeros(out_channels, device=device)) if bias else None

    def forward(self, x):
        y = _Conv2dFn.apply(x, self.weight, self.lut, self.stride, self.padding, self.dilation)
        return y + self.bias if self.bias is not None else y


# ------------------------------------------------------------------ depthwise Conv2D
class _DepthwiseConv2dFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, w, lut, stride, padding, dilation):
        x, w = _f32(x), _f32(w)
        N, H, W, C = x.shape
        R, S, C2, D = w.shape
        if C2 != C:
            raise ValueError("filter channels differ from the input's")
        desc = ConvDesc.make(N, H, W, C, C * D, R, S, stride, padding, dilation)
        P, Q = amsim_conv2d_out_hw(desc)
        y = torch.empty((N, P, Q, C * D), dtype=torch.float32, device=x.device)
        amsim_dwconv2d_fwd(desc, x, w, y, lut)
        ctx.save_for_backward(x, w)
        ctx.lut, ctx.desc = lut, desc
        return y

    @staticmethod
    def backward(ctx, dy):
        x, w = ctx.saved_tensors
        dy = _f32(dy)
        desc, lut = ctx.desc, ctx.lut
        dx = dw = None
        if ctx.needs_input_grad[0]:
            dx = torch.empty_like(x)
            amsim_dwconv2d_bwd_data(desc, dy, w, dx, lut)
        if ctx.needs_input_grad[1]:
            dw = torch.empty_like(w)
            amsim_dwconv2d_bwd_filter(desc, x, dy, dw, lut,
                                      ws=workspace(amsim_dwconv2d_workspace_size(desc, 2, lut), x.device))
        return dx, dw, None, None, None, None


def am_depthwise_conv2d(x, w, lut, stride=1, padding=0, dilation=1):
    """Depthwise y = conv2d(x, w) per channel with approximate products (x NHWC,
    w R x S x C x D for a channel multiplier D, y NPQ(C*D), output channel
    c*D + d from input channel c)."""
    return _DepthwiseConv2dFn.apply(x, w, lut, _pair(stride), _pair(padding), _pair(dilation))


class AMDepthwiseConv2d(torch.nn.Module):
    """Depthwise 2-D convolution (one filter group per input channel, channel
    multiplier D) whose forward pass and both gradients use the approximate
    multiplier; depthwise convolution is one of the layer types ApproxTrain
    simulates (Sec. III, Table I).  NHWC input, R x S x C x D filters."""

    def __init__(self, channels: int, kernel_size, lut, depth_multiplier: int = 1, stride=1, padding=0,
                 dilation=1, bias: bool = True, device="cuda", generator: torch.Generator | None = None):
        super().__init__()
        self.lut = lut
        R, S = _pair(kernel_size)
        self.stride, self.padding, self.dilation = _pair(stride), _pair(padding), _pair(dilation)
        std = math.sqrt(2.0 / (R * S))                                  # He normal over a channel's taps
        w = torch.randn((R, S, channels, depth_multiplier), generator=generator) * std
        self.weight = torch.nn.Parameter(w.to(device))
        self.bias = (torch.nn.Parameter(torch.zeros(channels * depth_multiplier, device=device)) if bias
                     else None)

    def forward(self, x):
        y = _DepthwiseConv2dFn.apply(x, self.weight, self.lut, self.stride, self.padding, self.dilation)
        return y + self.bias if self.bias is not None else y


# ------------------------------------------------------------------ attention
class _AttentionFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, lut, scale):
        q, k, v = _f32(q), _f32(k), _f32(v)
        b, h, s, d = q.shape
        t = k.shape[2]
        qf, kf, vf = q.reshape(b * h, s, d), k.reshape(b * h, t, d), v.reshape(b * h, t, d)
        S = _bgemm("N", "T", qf, kf, s, t, d, lut, alpha=scale)
        P = torch.empty_like(S)
        amsim_softmax_rows(S, P, b * h * s, t)
        O = _bgemm("N", "N", P, vf, s, d, t, lut)
        ctx.save_for_backward(qf, kf, vf, P)
        ctx.lut, ctx.scale, ctx.shape = lut, scale, (b, h, s, t, d)
        return O.reshape(b, h, s, d)

    @staticmethod
    def backward(ctx, dO):
        qf, kf, vf, P = ctx.saved_tensors
        b, h, s, t, d = ctx.shape
        lut, scale = ctx.lut, ctx.scale
        dOf = _f32(dO).reshape(b * h, s, d)
        dV = _bgemm("T", "N", P, dOf, t, d, s, lut)                   # P^T dO
        dP = _bgemm("N", "T", dOf, vf, s, t, d, lut)                  # dO V^T
        dS = torch.empty_like(dP)
        amsim_softmax_rows_backward(P, dP, dS, b * h * s, t)
        dQ = _bgemm("N", "N", dS, kf, s, d, t, lut, alpha=scale)      # scale dS K
        dK = _bgemm("T", "N", dS, qf, t, d, s, lut, alpha=scale)      # scale dS^T Q
        return dQ.reshape(b, h, s, d), dK.reshape(b, h, t, d), dV.reshape(b, h, t, d), None, None


def am_attention(q, k, v, lut, scale: float | None = None):
    """softmax(scale q k^T) v per (batch, head), contractions approximate,
    softmax exact; scale defaults to 1/sqrt(dim)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    return _AttentionFn.apply(q, k, v, lut, float(scale))


class AMAttention(torch.nn.Module):
    """Scaled dot-product attention over [batch, heads, seq, dim] tensors
    with approximate contractions (no projections)."""

    def __init__(self, lut, scale: float | None = None):
        super().__init__()
        self.lut, self.scale = lut, scale

    def forward(self, q, k, v):
        return am_attention(q, k, v, self.lut, self.scale)
