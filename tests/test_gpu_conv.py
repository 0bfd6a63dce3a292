"""Implicit-GEMM Conv2D on the GPU against the CPU oracle's direct sums
(ApproxTrain Sec. VI-B: Algorithm 3 forward; Algorithm 4 weight gradient and
preceding-layer gradient): strides, padding, dilation, non-square shapes, both
multiplier kinds, guard canaries, split-K on the weight gradient."""
import numpy as np
import pytest

from gpu_helpers import assert_close, guarded, guards_intact, to_dev

pytestmark = pytest.mark.gpu

GEOMS = [
    # N, H, W, C, K, R, S, stride, pad, dil
    (2, 7, 6, 3, 4, 3, 3, (1, 1), (1, 1), (1, 1)),
    (1, 9, 8, 2, 5, 3, 2, (2, 1), (1, 0), (1, 1)),
    (2, 8, 9, 3, 2, 3, 3, (1, 2), (2, 2), (2, 1)),
    (1, 5, 5, 4, 3, 1, 1, (1, 1), (0, 0), (1, 1)),
    (1, 10, 7, 2, 3, 2, 3, (3, 2), (1, 2), (1, 2)),
    (3, 12, 11, 20, 70, 3, 3, (1, 1), (1, 1), (1, 1)),
    (2, 16, 16, 64, 64, 3, 3, (2, 2), (1, 1), (1, 1)),
    (1, 6, 40, 33, 9, 5, 1, (1, 1), (2, 0), (1, 1)),
    (2, 20, 17, 40, 300, 1, 1, (1, 1), (0, 0), (1, 1)),   # pointwise: dense operands
    (1, 9, 9, 8, 12, 1, 1, (2, 2), (0, 0), (1, 1)),       # strided 1x1: gather
]


def run_conv(amd, lut, which, desc, t0, t1, out_shape):
    import torch
    buf, out = guarded(out_shape)
    d0, d1 = to_dev(t0), to_dev(t1)
    nb = amd.amsim_conv2d_workspace_size(desc, which, lut)
    ws = amd.workspace(nb)
    fn = (amd.amsim_conv2d_fwd, amd.amsim_conv2d_bwd_data, amd.amsim_conv2d_bwd_filter)[which]
    fn(desc, d0, d1, out, lut, ws=ws)
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside the output"
    return out.cpu().numpy()


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
@pytest.mark.parametrize("g", GEOMS)
def test_conv_three_passes(amd, orc, luts, g, kind):
    N, H, W, C, K, R, S, st, pd, dl = g
    rng = np.random.default_rng(sum(g[:7]) + (kind == "exact"))
    desc = amd.ConvDesc.make(N, H, W, C, K, R, S, st, pd, dl)
    odesc = orc.conv_desc(N, H, W, C, K, R, S, st, pd, dl)
    P, Q = orc.conv_out_hw(odesc)
    assert amd.amsim_conv2d_out_hw(desc) == (P, Q)
    x = rng.standard_normal((N, H, W, C)).astype(np.float32)
    w = rng.standard_normal((R, S, C, K)).astype(np.float32)
    dy = rng.standard_normal((N, P, Q, K)).astype(np.float32)
    lut = luts(kind, 7)

    y = run_conv(amd, lut, 0, desc, x, w, (N, P, Q, K))
    ref, sa = orc.conv2d_fwd(kind, 7, odesc, x, w, np.arange(y.size))
    assert_close(y.reshape(-1), ref, sa, f"fwd {g}")

    dx = run_conv(amd, lut, 1, desc, dy, w, (N, H, W, C))
    ref, sa = orc.conv2d_bwd_data(kind, 7, odesc, dy, w, np.arange(dx.size))
    assert_close(dx.reshape(-1), ref, sa, f"bwd_data {g}")

    dw = run_conv(amd, lut, 2, desc, x, dy, (R, S, C, K))
    ref, sa = orc.conv2d_bwd_filter(kind, 7, odesc, x, dy, np.arange(dw.size))
    assert_close(dw.reshape(-1), ref, sa, f"bwd_filter {g}")


def test_conv_errors(amd, luts):
    import torch
    lut = luts("mitchell", 7)
    x = torch.zeros(16, device="cuda")
    with pytest.raises(amd.AmsimError):
        amd.amsim_conv2d_fwd(amd.ConvDesc.make(1, 2, 2, 1, 1, 5, 5), x, x, x, lut)
    with pytest.raises(amd.AmsimError):
        amd.amsim_conv2d_fwd(amd.ConvDesc.make(1, 4, 4, 1, 1, 3, 3, stride=(0, 1)), x, x, x, lut)
    with pytest.raises(amd.AmsimError):
        amd.amsim_conv2d_bwd_data(amd.ConvDesc.make(1, 4, 4, 1, 1, 3, 3), None, x, x, lut)
