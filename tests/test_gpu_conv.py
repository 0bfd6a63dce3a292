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

# Unit-stride geometries whose passes read their operands in place as tensor
# boxes (whole output rows of the activation at each filter tap for the
# forward and data-gradient passes, 64-channel blocks for the filter gradient).
TMA_GEOMS = [
    (1, 32, 32, 64, 32, 3, 3, (1, 1), (1, 1), (1, 1)),    # all three passes
    (2, 16, 16, 32, 48, 3, 3, (1, 1), (1, 1), (1, 1)),    # forward and data gradient
    (2, 16, 16, 16, 16, 3, 5, (1, 1), (2, 2), (2, 1)),    # dilated rows, 3 x 5 filter
    (1, 8, 20, 64, 16, 3, 3, (1, 1), (1, 0), (1, 2)),     # filter gradient, dilated columns
    (1, 16, 16, 128, 32, 3, 3, (1, 1), (1, 1), (1, 1)),   # filter gradient's R*S*C = 1152: a 128-column tail
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
    """The same geometries without scratch: no split reduction."""
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


def test_tensor_boxes_and_gather_fallback(amd, orc, luts):
    """A unit-stride geometry reads its operands in place as tensor boxes, with
    or without scratch (one launch, or a fixup kernel after a non-cooperative
    split); operands that are not 16-byte aligned fall back to the gathering
    kernel.  Both match the oracle."""
    import torch
    N, H, W, C, K, R, S = 1, 32, 32, 64, 32, 3, 3
    desc = amd.ConvDesc.make(N, H, W, C, K, R, S, (1, 1), (1, 1), (1, 1))
    odesc = orc.conv_desc(N, H, W, C, K, R, S, (1, 1), (1, 1), (1, 1))
    lut = luts("mitchell", 7)
    rng = np.random.default_rng(99)
    x = rng.standard_normal((N, H, W, C)).astype(np.float32)
    w = rng.standard_normal((R, S, C, K)).astype(np.float32)
    dy = rng.standard_normal((N, H, W, K)).astype(np.float32)
    fns = (amd.amsim_conv2d_fwd, amd.amsim_conv2d_bwd_data, amd.amsim_conv2d_bwd_filter)
    refs = (orc.conv2d_fwd, orc.conv2d_bwd_data, orc.conv2d_bwd_filter)
    args = [(x, w), (dy, w), (x, dy)]
    shapes = [(N, H, W, K), (N, H, W, C), (R, S, C, K)]

    def dev(a, shift):
        # a device copy starting `shift` floats into its buffer (shift 1: 4-byte aligned only)
        buf = torch.empty(a.size + 4, dtype=torch.float32, device="cuda")
        view = buf[shift:shift + a.size].view(*a.shape)
        view.copy_(torch.from_numpy(a).cuda())
        return view

    for which in range(3):
        nb = amd.amsim_conv2d_workspace_size(desc, which, lut)
        ref, sa = refs[which]("mitchell", 7, odesc, *args[which], np.arange(int(np.prod(shapes[which]))))
        for shift, scratch in ((0, True), (0, False), (1, True)):
            a0, a1 = dev(args[which][0], shift), dev(args[which][1], shift)
            out = torch.empty(shapes[which], dtype=torch.float32, device="cuda")
            ws = amd.workspace(nb) if scratch else None
            torch.cuda.synchronize()
            n0 = amd.amsim_kernel_launches()
            fns[which](desc, a0, a1, out, lut, ws=ws)
            torch.cuda.synchronize()
            path, launches = amd.amsim_last_path(), amd.amsim_kernel_launches() - n0
            if shift == 0:
                assert path & amd.AMSIM_PATH_RAW_TILES and path & amd.AMSIM_PATH_CONV_BOXES, (which, path)
                assert launches == (2 if path & amd.AMSIM_PATH_FIXUP else 1), (which, path, launches)
            else:
                assert path & amd.AMSIM_PATH_INKERNEL_DECODE and not path & amd.AMSIM_PATH_CONV_BOXES, (which, path)
            assert_close(out.cpu().numpy().reshape(-1), ref, sa, f"pass {which} shift {shift} scratch {scratch}")
