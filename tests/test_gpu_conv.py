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

# Unit-stride geometries whose passes take the tensor-box layouts (shifted
# activation copies for the forward and data-gradient passes, 64-channel
# blocks for the filter gradient) when the scratch holds the planes.
TMA_GEOMS = [
    (1, 32, 32, 64, 32, 3, 3, (1, 1), (1, 1), (1, 1)),    # all three passes
    (2, 16, 16, 32, 48, 3, 3, (1, 1), (1, 1), (1, 1)),    # forward and data gradient
    (2, 16, 16, 16, 16, 3, 5, (1, 1), (2, 2), (2, 1)),    # dilated rows, 3 x 5 filter
    (1, 8, 20, 64, 16, 3, 3, (1, 1), (1, 0), (1, 2)),     # filter gradient, dilated columns
]


def run_conv(amd, lut, which, desc, t0, t1, out_shape, scratch=True):
    import torch
    buf, out = guarded(out_shape)
    d0, d1 = to_dev(t0), to_dev(t1)
    nb = amd.amsim_conv2d_workspace_size(desc, which, lut)
    ws = amd.workspace(nb) if scratch else None
    fn = (amd.amsim_conv2d_fwd, amd.amsim_conv2d_bwd_data, amd.amsim_conv2d_bwd_filter)[which]
    fn(desc, d0, d1, out, lut, ws=ws)
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside the output"
    return out.cpu().numpy()


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
@pytest.mark.parametrize("g", GEOMS + TMA_GEOMS)
def test_conv_three_passes(amd, orc, luts, g, kind):
    check_three_passes(amd, orc, luts, g, kind, True)


@pytest.mark.parametrize("g", TMA_GEOMS)
def test_conv_three_passes_without_scratch(amd, orc, luts, g):
    """The same geometries through the gathering kernel (no scratch for planes)."""
    check_three_passes(amd, orc, luts, g, "mitchell", False)


def check_three_passes(amd, orc, luts, g, kind, scratch):
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

    y = run_conv(amd, lut, 0, desc, x, w, (N, P, Q, K), scratch)
    ref, sa = orc.conv2d_fwd(kind, 7, odesc, x, w, np.arange(y.size))
    assert_close(y.reshape(-1), ref, sa, f"fwd {g}")

    dx = run_conv(amd, lut, 1, desc, dy, w, (N, H, W, C), scratch)
    ref, sa = orc.conv2d_bwd_data(kind, 7, odesc, dy, w, np.arange(dx.size))
    assert_close(dx.reshape(-1), ref, sa, f"bwd_data {g}")

    dw = run_conv(amd, lut, 2, desc, x, dy, (R, S, C, K), scratch)
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


def test_tma_layout_is_used_when_scratch_allows(amd, luts):
    """A unit-stride geometry asks for plane scratch on every pass and, given
    it, takes the tensor-box layouts (a predecode launch, then the GEMM);
    without scratch the gathering kernel runs alone."""
    import torch
    N, H, W, C, K, R, S = 1, 32, 32, 64, 32, 3, 3
    desc = amd.ConvDesc.make(N, H, W, C, K, R, S, (1, 1), (1, 1), (1, 1))
    lut = luts("mitchell", 7)
    x = torch.zeros((N, H, W, C), device="cuda")
    w = torch.zeros((R, S, C, K), device="cuda")
    dy = torch.zeros((N, H, W, K), device="cuda")
    outs = [torch.empty((N, H, W, K), device="cuda"), torch.empty((N, H, W, C), device="cuda"),
            torch.empty((R, S, C, K), device="cuda")]
    args = [(x, w), (dy, w), (x, dy)]
    fns = (amd.amsim_conv2d_fwd, amd.amsim_conv2d_bwd_data, amd.amsim_conv2d_bwd_filter)
    for which in range(3):
        nb = amd.amsim_conv2d_workspace_size(desc, which, lut)
        assert nb >= 2 * 4 * N * H * W * min(C, K), f"pass {which}: no plane scratch requested"
        for scratch in (True, False):
            ws = amd.workspace(nb) if scratch else None
            torch.cuda.synchronize()
            n0 = amd.amsim_kernel_launches()
            fns[which](desc, *args[which], outs[which], lut, ws=ws)
            torch.cuda.synchronize()
            path, launches = amd.amsim_last_path(), amd.amsim_kernel_launches() - n0
            if scratch:
                assert path & amd.AMSIM_PATH_PLANES and path & amd.AMSIM_PATH_CONV_BOXES, (which, path)
                # the predecode pass and the GEMM (and the fixup kernel without a cooperative launch)
                assert launches == (3 if path & amd.AMSIM_PATH_FIXUP else 2), (which, path, launches)
            else:
                assert path & amd.AMSIM_PATH_INKERNEL_DECODE and not path & amd.AMSIM_PATH_PLANES, (which, path)
                assert launches == 1, (which, launches)
