"""The five layer workloads at full size, run through the same step objects
the benchmark times, checked against the CPU oracle on seeded samples of
their outputs (each sampled output computed in full by the oracle).
Chained contractions (MLP layers, attention P V) are checked on the GPU's
own inputs to that contraction, so 1-ulp differences upstream cannot flip a
truncated mantissa downstream."""
import numpy as np
import pytest

from gpu_helpers import assert_close
from approximate_multiplier_dnn_gb300 import steps
from approximate_multiplier_dnn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def host(t):
    return t.detach().cpu().numpy()


def test_mlp_784_1000_500_10(amd, orc, luts):
    import torch
    data = wl.mlp()
    st = steps.MLPStep(data, luts("mitchell", 7))
    st.run()
    torch.cuda.synchronize()
    assert st.macs == 989_952_000
    rng = np.random.default_rng(0)
    xs = [data["X"], host(st.Y[0]), host(st.Y[1])]
    for l in range(3):
        W, dY = data[f"W{l + 1}"], data[f"dY{l + 1}"]
        rows = rng.choice(xs[l].shape[0], 16, replace=False)
        ref, sa = orc.gemm("mitchell", 7, xs[l], W, rows=rows)
        assert_close(host(st.Y[l])[rows], ref, sa, f"Y{l + 1}")
        ref, sa = orc.gemm("mitchell", 7, dY, W, transB=True, rows=rows)
        assert_close(host(st.dX[l])[rows], ref, sa, f"dX{l + 1}")
        wrows = rng.choice(W.shape[0], 16, replace=False)
        ref, sa = orc.gemm("mitchell", 7, xs[l], dY, transA=True, rows=wrows)
        assert_close(host(st.dW[l])[wrows], ref, sa, f"dW{l + 1}")


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
def test_conv3x3_128x32x32x64(amd, orc, luts, kind):
    import torch
    g = wl.CONV3X3
    data = wl.conv3x3()
    st = steps.ConvStep(data, g, luts(kind, 7))
    st.run()
    torch.cuda.synchronize()
    assert st.macs == 3 * 4_831_838_208
    desc = orc.conv_desc(g["N"], g["H"], g["W"], g["C"], g["K"], g["R"], g["S"], g["stride"], g["pad"], g["dil"])
    rng = np.random.default_rng(1)
    pts = rng.choice(st.y.numel(), 2000, replace=False)
    ref, sa = orc.conv2d_fwd(kind, 7, desc, data["x"], data["w"], pts)
    assert_close(host(st.y).reshape(-1)[pts], ref, sa, "fwd")
    pts = rng.choice(st.dx.numel(), 2000, replace=False)
    ref, sa = orc.conv2d_bwd_data(kind, 7, desc, data["dy"], data["w"], pts)
    assert_close(host(st.dx).reshape(-1)[pts], ref, sa, "bwd_data")
    pts = np.concatenate([rng.choice(st.dw.numel(), 60, replace=False), [0, st.dw.numel() - 1]])
    ref, sa = orc.conv2d_bwd_filter(kind, 7, desc, data["x"], data["dy"], pts)
    assert_close(host(st.dw).reshape(-1)[pts], ref, sa, "bwd_filter")


@pytest.mark.parametrize("M", [4, 5, 6, 7, 8, 9, 10, 11])
def test_square_gemm_4096_mantissa_sweep(amd, orc, luts, M):
    import torch
    data = wl.square_gemm(4096)
    st = steps.SquareGemmStep(data, luts("mitchell", M))
    st.run()
    torch.cuda.synchronize()
    rng = np.random.default_rng(M)
    rows = rng.choice(4096, 6, replace=False)
    ref, sa = orc.gemm("mitchell", M, data["A"], data["B"], rows=rows)
    assert_close(host(st.C)[rows], ref, sa, f"4096^3 M={M}")


def test_attention_32x16x512x64(amd, orc, luts):
    import torch
    data = wl.attention()
    st = steps.AttentionStep(data, luts("mitchell", 7))
    st.run()
    torch.cuda.synchronize()
    S, P, O = host(st.S), host(st.P), host(st.O)
    rng = np.random.default_rng(2)
    for _ in range(6):
        b, h = rng.integers(0, 32), rng.integers(0, 16)
        rows = rng.choice(512, 8, replace=False)
        q, k, v = data["Q"][b, h], data["K"][b, h], data["V"][b, h]
        ref, sa = orc.attention_scores("mitchell", 7, q, k, 0.125, rows=rows)
        assert_close(S[b, h][rows], ref, 0.125 * sa, "S")
        pref = orc.softmax_rows(S[b, h][rows])
        assert np.allclose(P[b, h][rows], pref, rtol=2e-6, atol=1e-9)
        ref, sa = orc.attention_output("mitchell", 7, P[b, h], v, rows=rows)
        assert_close(O[b, h][rows], ref, sa, "O")


def test_conv1x1_64x56x56x256(amd, orc, luts):
    import torch
    g = wl.CONV1X1
    data = wl.conv1x1()
    st = steps.ConvStep(data, g, luts("mitchell", 7), passes=(0,))
    st.run()
    torch.cuda.synchronize()
    desc = orc.conv_desc(g["N"], g["H"], g["W"], g["C"], g["K"], g["R"], g["S"], g["stride"], g["pad"], g["dil"])
    rng = np.random.default_rng(3)
    pts = rng.choice(st.y.numel(), 3000, replace=False)
    ref, sa = orc.conv2d_fwd("mitchell", 7, desc, data["x"], data["w"], pts)
    assert_close(host(st.y).reshape(-1)[pts], ref, sa, "1x1 fwd")
