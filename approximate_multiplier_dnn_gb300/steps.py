"""The five layer workloads as sequences of library calls (device tensors in,
device tensors out).  Each ``run()`` is one pass of the workload's contractions
through the C ABI on one stream; the benchmark, the smoke check and the
full-size parity tests all drive these same objects, so they time and check
the same launch configuration.

Operand order of every contraction follows the layer's data flow:
Dense forward (x, w); preceding-layer gradient (dy, w); weight gradient
(x, dy); conv likewise; attention (q, k) then (p, v).
"""
from __future__ import annotations

from . import (ConvDesc, GemmProblem, amsim_mul, amsim_conv2d_bwd_data, amsim_conv2d_bwd_filter, amsim_conv2d_fwd,
               amsim_conv2d_out_hw, amsim_conv2d_workspace_size, amsim_gemm, amsim_gemm_grouped,
               amsim_gemm_grouped_workspace_size, amsim_gemm_phased, amsim_gemm_phased_workspace_size,
               amsim_gemm_strided_batched, amsim_gemm_workspace_size,
               amsim_dwconv2d_bwd_data, amsim_dwconv2d_bwd_filter, amsim_dwconv2d_fwd, amsim_dwconv2d_workspace_size,
               amsim_softmax_rows, workspace)


def _dev(t, device):
    import torch
    if isinstance(t, torch.Tensor):
        return t.to(device)
    return torch.from_numpy(t).to(device)


class GemmCall:
    """One row-major GEMM C = alpha op(A) op(B) + beta C on device tensors."""

    def __init__(self, A, B, C, transA=False, transB=False, alpha=1.0, beta=0.0):
        self.A, self.B, self.C = A, B, C
        self.tA, self.tB = ("T" if transA else "N"), ("T" if transB else "N")
        self.m = A.shape[1] if transA else A.shape[0]
        self.k = A.shape[0] if transA else A.shape[1]
        self.n = B.shape[0] if transB else B.shape[1]
        self.alpha, self.beta = alpha, beta

    @property
    def macs(self) -> int:
        return self.m * self.n * self.k

    def ws_bytes(self, lut) -> int:
        return amsim_gemm_workspace_size(self.tA, self.tB, self.m, self.n, self.k, 1, lut)

    def __call__(self, lut, ws, stream=None):
        amsim_gemm(self.tA, self.tB, self.m, self.n, self.k, self.alpha, self.A, max(1, self.A.shape[1]),
                   self.B, max(1, self.B.shape[1]), self.beta, self.C, max(1, self.n), lut, ws=ws,
                   stream=stream)

    def native(self):
        """The same contraction with torch fp32 (cuBLAS) into a scratch output."""
        import torch
        a = self.A.t() if self.tA == "T" else self.A
        b = self.B.t() if self.tB == "T" else self.B
        out = torch.empty((self.m, self.n), dtype=torch.float32, device=self.A.device)
        return lambda: torch.matmul(a, b, out=out)

    def problem(self) -> GemmProblem:
        return GemmProblem.make(self.tA, self.tB, self.m, self.n, self.k, self.alpha, self.A,
                                max(1, self.A.shape[1]), self.B, max(1, self.B.shape[1]), self.beta, self.C,
                                max(1, self.n))


class GemmGroup:
    """Independent GEMMs issued as one grouped launch."""

    def __init__(self, calls):
        self.calls = list(calls)
        import ctypes
        self.arr = (GemmProblem * len(self.calls))(*[c.problem() for c in self.calls])

    @property
    def macs(self) -> int:
        return sum(c.macs for c in self.calls)

    def ws_bytes(self, lut) -> int:
        return amsim_gemm_grouped_workspace_size(self.arr, lut)

    def __call__(self, lut, ws, stream=None):
        amsim_gemm_grouped(self.arr, lut, ws=ws, stream=stream)


class PhasedGemms:
    """Ordered phases of GEMMs issued as one phased call: phase i reads
    outputs of phases before after[i] only."""

    def __init__(self, phases):
        self.names = [nm for nm, _, _ in phases]
        self.calls = [c for _, cl, _ in phases for c in cl]
        self.first, n = [], 0
        for _, cl, _ in phases:
            self.first.append(n)
            n += len(cl)
        self.after = [a for _, _, a in phases]
        self.arr = (GemmProblem * len(self.calls))(*[c.problem() for c in self.calls])

    @property
    def macs(self) -> int:
        return sum(c.macs for c in self.calls)

    def ws_bytes(self, lut) -> int:
        return amsim_gemm_phased_workspace_size(self.arr, self.first, self.after, lut)

    def __call__(self, lut, ws, stream=None):
        amsim_gemm_phased(self.arr, self.first, self.after, lut, ws=ws, stream=stream)


class MLPStep:
    """3-layer MLP (784-1000-500-10, batch 256): forward Y_l = X_l W_l, then
    for every layer dX_l = dY_l W_l^T and dW_l = X_l^T dY_l (pure linear
    layers; X_{l+1} = Y_l; dY_l synthetic per layer).  The nine GEMMs run as
    one phased call (one launch) whose five phases follow the data
    dependences, with independent work between each forward GEMM and the
    GEMMs that read its output, so that no SM waits at a phase boundary:
    {Y1}, {dX1, dX2}, {Y2} (reads Y1), {dW1, dW2} (dW2 reads Y1),
    {Y3, dW3, dX3} (Y3 and dW3 read Y2).  Every phase copies its operand tiles
    in place (the 10-wide operands, whose leading dimension is not a multiple
    of 4 elements, with plain asynchronous loads)."""

    def __init__(self, data: dict, lut, device="cuda"):
        import torch
        self.lut = lut
        d = {k: _dev(v, device) for k, v in data.items()}
        self.inputs = d
        f32 = dict(dtype=torch.float32, device=device)
        X = d["X"]
        self.Y, self.dX, self.dW = [], [], []
        fwd, xin = [], X
        for l in range(3):
            W = d[f"W{l + 1}"]
            Y = torch.empty((X.shape[0], W.shape[1]), **f32)
            fwd.append(GemmCall(xin, W, Y))
            self.Y.append(Y)
            xin = Y
        xs = [X, self.Y[0], self.Y[1]]
        dxc, dwc = [], []
        for l in range(3):
            W, dY = d[f"W{l + 1}"], d[f"dY{l + 1}"]
            dX = torch.empty((dY.shape[0], W.shape[0]), **f32)
            dW = torch.empty_like(W)
            dxc.append(GemmCall(dY, W, dX, transB=True))
            dwc.append(GemmCall(xs[l], dY, dW, transA=True))
            self.dX.append(dX)
            self.dW.append(dW)
        self.calls = fwd + [c for pair in zip(dxc, dwc) for c in pair]
        # (name, calls, number of leading phases that must be complete first)
        self.phased = PhasedGemms([("fwd1", [fwd[0]], 0),
                                   ("dX1+dX2", [dxc[0], dxc[1]], 0),
                                   ("fwd2", [fwd[1]], 1),
                                   ("dW1+dW2", [dwc[0], dwc[1]], 1),
                                   ("fwd3+dW3+dX3", [fwd[2], dwc[2], dxc[2]], 3)])
        self.ws = workspace(self.phased.ws_bytes(lut), device)

    @property
    def macs(self) -> int:
        return sum(c.macs for c in self.calls)

    def outputs(self) -> list:
        return self.Y + self.dX + self.dW

    def parts(self, stream=None):
        """(name, zero-argument launcher, approximate MACs, kernel launches) per ABI call."""
        return [("+".join(self.phased.names), lambda: self.phased(self.lut, self.ws, stream), self.phased.macs, 1)]

    def run(self, stream=None):
        self.phased(self.lut, self.ws, stream)

    def native(self):
        fns = [c.native() for c in self.calls]
        return lambda: [f() for f in fns]


class LayersMLPStep:
    """The MLP 784-1000-500-10 (batch 256) through the autograd layers: three
    approximate Dense layers (no bias) run forward and backward by torch's
    autograd -- nine separate approximate GEMM calls, the backward chained
    through the layers (a layer's dY is the next layer's dX), from a
    synthetic dY3.  Same MAC count as MLPStep; the gradients accumulate into
    buffers that are cleared each step."""

    def __init__(self, data: dict, lut, device="cuda"):
        import torch
        self.lut = lut
        d = {k: _dev(v, device) for k, v in data.items()}
        self.inputs = {k: d[k] for k in ("X", "W1", "W2", "W3", "dY3")}
        self.X = d["X"].requires_grad_()
        self.W = [d[f"W{l + 1}"].requires_grad_() for l in range(3)]
        self.dY = d["dY3"]
        for t in [self.X] + self.W:
            t.grad = torch.zeros_like(t)
        self.Y = None

    @property
    def macs(self) -> int:
        n, dims = self.X.shape[0], [self.X.shape[1]] + [w.shape[1] for w in self.W]
        return 3 * sum(n * dims[i] * dims[i + 1] for i in range(3))

    def outputs(self) -> list:
        return [self.X.grad] + [w.grad for w in self.W]

    def run(self, stream=None):
        import torch
        from .layers import am_dense
        ctx = torch.cuda.stream(stream) if stream is not None else torch.cuda.stream(torch.cuda.current_stream())
        with ctx:
            for t in [self.X] + self.W:
                t.grad.zero_()
            h = self.X
            for w in self.W:
                h = am_dense(h, w, self.lut)
            h.backward(self.dY)

    def parts(self, stream=None):
        return [("fwd+bwd through AMDense layers", lambda: self.run(stream), self.macs, 9)]

    def native(self):
        import torch
        X, W = self.X.detach().clone().requires_grad_(), [w.detach().clone().requires_grad_() for w in self.W]

        def f():
            h = X
            for w in W:
                h = h @ w
            h.backward(self.dY)
        return f


class ConvStep:
    """Conv2D forward, preceding-layer gradient and weight gradient of one
    NHWC layer (implicit GEMMs)."""

    def __init__(self, data: dict, geom: dict, lut, device="cuda", passes=(0, 1, 2)):
        import torch
        self.lut = lut
        g = geom
        self.desc = ConvDesc.make(g["N"], g["H"], g["W"], g["C"], g["K"], g["R"], g["S"], g["stride"], g["pad"],
                                  g["dil"])
        self.P, self.Q = amsim_conv2d_out_hw(self.desc)
        self.x = _dev(data["x"], device)
        self.w = _dev(data["w"], device)
        self.dy = _dev(data["dy"], device) if "dy" in data else None
        self.passes = tuple(passes)
        f32 = dict(dtype=torch.float32, device=device)
        self.y = torch.empty((g["N"], self.P, self.Q, g["K"]), **f32)
        self.dx = torch.empty_like(self.x) if 1 in self.passes else None
        self.dw = torch.empty_like(self.w) if 2 in self.passes else None
        self.g = g
        self.ws = workspace(max(amsim_conv2d_workspace_size(self.desc, p, lut) for p in self.passes), device)

    @property
    def macs(self) -> int:
        g = self.g
        return len(self.passes) * g["N"] * self.P * self.Q * g["K"] * g["R"] * g["S"] * g["C"]

    def outputs(self) -> list:
        return [t for t in (self.y, self.dx, self.dw) if t is not None]

    def parts(self, stream=None):
        g = self.g
        per = g["N"] * self.P * self.Q * g["K"] * g["R"] * g["S"] * g["C"]
        fns = {0: ("fwd", lambda: amsim_conv2d_fwd(self.desc, self.x, self.w, self.y, self.lut, ws=self.ws,
                                                   stream=stream)),
               1: ("bwd_data", lambda: amsim_conv2d_bwd_data(self.desc, self.dy, self.w, self.dx, self.lut,
                                                             ws=self.ws, stream=stream)),
               2: ("bwd_filter", lambda: amsim_conv2d_bwd_filter(self.desc, self.x, self.dy, self.dw, self.lut,
                                                                 ws=self.ws, stream=stream))}
        return [(fns[p][0], fns[p][1], per, 1 + (amsim_conv2d_workspace_size(self.desc, p, self.lut) > 0))
                for p in self.passes]

    def native(self):
        """The same passes with torch fp32 (cuDNN): NHWC tensors as channels-last views."""
        import torch
        import torch.nn.functional as F
        from torch.nn import grad as nng
        g = self.g
        st, pd, dl = (g["stride"][0], g["stride"][1]), (g["pad"][0], g["pad"][1]), (g["dil"][0], g["dil"][1])
        x = self.x.permute(0, 3, 1, 2)                       # N C H W view of NHWC
        w = self.w.permute(3, 2, 0, 1).contiguous()          # K C R S from R S C K
        dy = self.dy.permute(0, 3, 1, 2) if self.dy is not None else None
        fns = []
        if 0 in self.passes:
            fns.append(lambda: F.conv2d(x, w, stride=st, padding=pd, dilation=dl))
        if 1 in self.passes:
            fns.append(lambda: nng.conv2d_input(x.shape, w, dy, stride=st, padding=pd, dilation=dl))
        if 2 in self.passes:
            fns.append(lambda: nng.conv2d_weight(x, w.shape, dy, stride=st, padding=pd, dilation=dl))
        return lambda: [f() for f in fns]

    def run(self, stream=None):
        if 0 in self.passes:
            amsim_conv2d_fwd(self.desc, self.x, self.w, self.y, self.lut, ws=self.ws, stream=stream)
        if 1 in self.passes:
            amsim_conv2d_bwd_data(self.desc, self.dy, self.w, self.dx, self.lut, ws=self.ws, stream=stream)
        if 2 in self.passes:
            amsim_conv2d_bwd_filter(self.desc, self.x, self.dy, self.dw, self.lut, ws=self.ws, stream=stream)


class DwConvStep:
    """Depthwise Conv2D forward, preceding-layer gradient and weight gradient
    of one NHWC layer with a channel multiplier D (K = C*D output channels)."""

    def __init__(self, data: dict, geom: dict, lut, device="cuda", passes=(0, 1, 2)):
        import torch
        self.lut = lut
        g = geom
        self.desc = ConvDesc.make(g["N"], g["H"], g["W"], g["C"], g["C"] * g["D"], g["R"], g["S"], g["stride"],
                                  g["pad"], g["dil"])
        self.P, self.Q = amsim_conv2d_out_hw(self.desc)
        self.x = _dev(data["x"], device)
        self.w = _dev(data["w"], device)
        self.dy = _dev(data["dy"], device) if "dy" in data else None
        self.passes = tuple(passes)
        f32 = dict(dtype=torch.float32, device=device)
        self.y = torch.empty((g["N"], self.P, self.Q, g["C"] * g["D"]), **f32) if 0 in self.passes else None
        self.dx = torch.empty_like(self.x) if 1 in self.passes else None
        self.dw = torch.empty_like(self.w) if 2 in self.passes else None
        self.g = g
        self.ws = workspace(max(amsim_dwconv2d_workspace_size(self.desc, p, lut) for p in self.passes), device)

    @property
    def per_pass(self) -> int:
        g = self.g
        return g["N"] * self.P * self.Q * g["C"] * g["D"] * g["R"] * g["S"]

    @property
    def macs(self) -> int:
        return len(self.passes) * self.per_pass

    def pass_bytes(self, p) -> int:
        """Compulsory DRAM bytes of pass p: it reads its two operands once and
        writes its output once (4 bytes per element); the three passes touch
        the same three tensors (x, w, y) or their gradients."""
        g = self.g
        nx = g["N"] * g["H"] * g["W"] * g["C"]
        ny = g["N"] * self.P * self.Q * g["C"] * g["D"]
        nw = g["R"] * g["S"] * g["C"] * g["D"]
        return 4 * (nx + ny + nw)

    def kernel_name(self, p) -> str:
        """The library kernel pass p takes for this geometry (for labelling
        measurements; the library decides, see amsim_last_path)."""
        g = self.g
        base = (g["D"] == 1 and g["R"] == 3 and g["S"] == 3 and tuple(g["dil"]) == (1, 1) and g["C"] % 4 == 0)
        five = (g["D"] == 1 and g["R"] == 5 and g["S"] == 5 and tuple(g["dil"]) == (1, 1) and g["C"] % 4 == 0)
        if (base or five) and tuple(g["stride"]) == (1, 1):
            return "dw_tile_kernel"
        if base and tuple(g["stride"]) == (2, 2):
            if p != 1:
                return "dw_s2_kernel"
            if tuple(g["pad"]) == (1, 1):
                return "dw_s2d_kernel"
        return "dw_direct_kernel"

    def outputs(self) -> list:
        return [t for t in (self.y, self.dx, self.dw) if t is not None]

    def _call(self, p, stream):
        if p == 0:
            amsim_dwconv2d_fwd(self.desc, self.x, self.w, self.y, self.lut, ws=self.ws, stream=stream)
        elif p == 1:
            amsim_dwconv2d_bwd_data(self.desc, self.dy, self.w, self.dx, self.lut, ws=self.ws, stream=stream)
        else:
            amsim_dwconv2d_bwd_filter(self.desc, self.x, self.dy, self.dw, self.lut, ws=self.ws, stream=stream)

    def parts(self, stream=None):
        names = {0: "fwd", 1: "bwd_data", 2: "bwd_filter"}
        return [(names[p], (lambda p=p: self._call(p, stream)), self.per_pass,
                 1 + (amsim_dwconv2d_workspace_size(self.desc, p, self.lut) > 0)) for p in self.passes]

    def run(self, stream=None):
        for p in self.passes:
            self._call(p, stream)

    def native(self):
        """The same passes with torch fp32 (cuDNN grouped convolution, one group
        per input channel) on channels-last views."""
        import torch.nn.functional as F
        from torch.nn import grad as nng
        g = self.g
        st, pd, dl = tuple(g["stride"]), tuple(g["pad"]), tuple(g["dil"])
        K = g["C"] * g["D"]
        x = self.x.permute(0, 3, 1, 2)                                   # N C H W view of NHWC
        w = self.w.reshape(g["R"], g["S"], K).permute(2, 0, 1).unsqueeze(1).contiguous()   # K 1 R S
        dy = self.dy.permute(0, 3, 1, 2) if self.dy is not None else None
        fns = []
        if 0 in self.passes:
            fns.append(lambda: F.conv2d(x, w, stride=st, padding=pd, dilation=dl, groups=g["C"]))
        if 1 in self.passes:
            fns.append(lambda: nng.conv2d_input(x.shape, w, dy, stride=st, padding=pd, dilation=dl, groups=g["C"]))
        if 2 in self.passes:
            fns.append(lambda: nng.conv2d_weight(x, w.shape, dy, stride=st, padding=pd, dilation=dl,
                                                 groups=g["C"]))
        return lambda: [f() for f in fns]


class SquareGemmStep:
    def __init__(self, data: dict, lut, device="cuda"):
        import torch
        self.lut = lut
        self.A = _dev(data["A"], device)
        self.B = _dev(data["B"], device)
        self.C = torch.empty((self.A.shape[0], self.B.shape[1]), dtype=torch.float32, device=device)
        self.call = GemmCall(self.A, self.B, self.C)
        self.ws = workspace(self.call.ws_bytes(lut), device)

    @property
    def macs(self) -> int:
        return self.call.macs

    def outputs(self) -> list:
        return [self.C]

    def parts(self, stream=None):
        return [("gemm", lambda: self.call(self.lut, self.ws, stream), self.call.macs,
                 1 + (self.call.ws_bytes(self.lut) > 0))]

    def run(self, stream=None):
        self.call(self.lut, self.ws, stream)

    def native(self):
        return self.call.native()


class AttentionStep:
    """S = Q K^T / sqrt(d) (batched over batch*heads), exact fp32 row softmax,
    O = P V (batched).  Q, K, V: (batch, heads, seq, dim)."""

    def __init__(self, data: dict, lut, device="cuda"):
        import torch
        self.lut = lut
        self.Q = _dev(data["Q"], device)
        self.K = _dev(data["K"], device)
        self.V = _dev(data["V"], device)
        b, h, s, dd = self.Q.shape
        self.bh, self.s, self.d = b * h, s, dd
        f32 = dict(dtype=torch.float32, device=device)
        self.S = torch.empty((b, h, s, s), **f32)
        self.P = torch.empty((b, h, s, s), **f32)
        self.O = torch.empty((b, h, s, dd), **f32)
        self.scale = 1.0 / float(dd) ** 0.5
        n1 = amsim_gemm_workspace_size("N", "T", s, s, dd, self.bh, lut)
        n2 = amsim_gemm_workspace_size("N", "N", s, dd, s, self.bh, lut)
        self.ws = workspace(max(n1, n2), device)

    @property
    def macs(self) -> int:
        return 2 * self.bh * self.s * self.s * self.d

    def outputs(self) -> list:
        return [self.O]

    def parts(self, stream=None):
        s, d, bh = self.s, self.d, self.bh
        n1 = amsim_gemm_workspace_size("N", "T", s, s, d, bh, self.lut) > 0
        n2 = amsim_gemm_workspace_size("N", "N", s, d, s, bh, self.lut) > 0
        return [
            ("scores", lambda: amsim_gemm_strided_batched("N", "T", s, s, d, self.scale, self.Q, d, s * d, self.K, d,
                                                          s * d, 0.0, self.S, s, s * s, bh, self.lut, ws=self.ws,
                                                          stream=stream), bh * s * s * d, 1 + n1),
            ("softmax", lambda: amsim_softmax_rows(self.S, self.P, bh * s, s, stream=stream), 0, 1),
            ("pv", lambda: amsim_gemm_strided_batched("N", "N", s, d, s, 1.0, self.P, s, s * s, self.V, d, s * d,
                                                      0.0, self.O, d, s * d, bh, self.lut, ws=self.ws,
                                                      stream=stream), bh * s * s * d, 1 + n2),
        ]

    def run(self, stream=None):
        s, d, bh = self.s, self.d, self.bh
        amsim_gemm_strided_batched("N", "T", s, s, d, self.scale, self.Q, d, s * d, self.K, d, s * d, 0.0, self.S,
                                   s, s * s, bh, self.lut, ws=self.ws, stream=stream)
        amsim_softmax_rows(self.S, self.P, bh * s, s, stream=stream)
        amsim_gemm_strided_batched("N", "N", s, d, s, 1.0, self.P, s, s * s, self.V, d, s * d, 0.0, self.O, d,
                                   s * d, bh, self.lut, ws=self.ws, stream=stream)

    def native(self):
        """S = Q K^T / sqrt(d), row softmax, O = P V with torch fp32 (cuBLAS)."""
        import torch
        b, h, s, d = self.Q.shape
        q, k, v = (t.reshape(b * h, s, d) for t in (self.Q, self.K, self.V))

        def f():
            sc = torch.bmm(q, k.transpose(1, 2)) * self.scale
            return torch.bmm(torch.softmax(sc, dim=-1), v)
        return f


class MulStep:
    """Elementwise AMSim products c = AMSim(a, b) over n pairs."""

    def __init__(self, data: dict, lut, device="cuda"):
        import torch
        self.lut = lut
        self.a = _dev(data["a"], device)
        self.b = _dev(data["b"], device)
        self.c = torch.empty_like(self.a)

    @property
    def macs(self) -> int:
        return self.a.numel()

    def outputs(self) -> list:
        return [self.c]

    def parts(self, stream=None):
        return [("mul", lambda: amsim_mul(self.a, self.b, self.c, self.a.numel(), self.lut, stream=stream),
                 0, 1)]

    def run(self, stream=None):
        amsim_mul(self.a, self.b, self.c, self.a.numel(), self.lut, stream=stream)

    def native(self):
        import torch
        c = torch.empty_like(self.c)
        return lambda: torch.mul(self.a, self.b, out=c)
