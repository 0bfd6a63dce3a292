"""Depthwise Conv2D on the GPU against the CPU oracle's direct sums (depthwise
convolution is one of the layer types of ApproxTrain's Table I, Sec. III;
every product per Sec. V-B, Algorithm 2): the tiled kernel (3x3, unit stride
and dilation, one filter per channel) and the direct kernel (channel
multipliers, strides, dilation, other filter sizes, unaligned tensors), both
multiplier kinds, several mantissa widths, special operands, the weight
gradient with and without scratch, and the MobileNet-style 64x56x56x128 layer
at full size on sampled outputs."""
import numpy as np
import pytest

from gpu_helpers import assert_close, bits, guarded, guards_intact, to_dev

pytestmark = pytest.mark.gpu

# N, H, W, C, D, R, S, stride, pad, dil
TILED = [
    (2, 9, 70, 20, 1, 3, 3, (1, 1), (1, 1), (1, 1)),    # ragged row, column and channel tiles
    (1, 16, 16, 32, 1, 3, 3, (1, 1), (0, 0), (1, 1)),   # no padding: P, Q = H - 2, W - 2
    (2, 8, 8, 8, 1, 3, 3, (1, 1), (2, 2), (1, 1)),      # padding 2
    (1, 5, 12, 4, 1, 3, 3, (1, 1), (3, 1), (1, 1)),     # padding beyond the filter reach
    (3, 17, 65, 48, 1, 3, 3, (1, 1), (1, 1), (1, 1)),   # 65 columns: a one-column second tile
    (3, 1, 1, 8, 1, 3, 3, (1, 1), (1, 1), (1, 1)),      # 1x1 image: only the centre tap meets data
    (2, 3, 130, 4, 1, 3, 3, (1, 1), (0, 0), (1, 1)),    # one output row, exactly two 64-column tiles
    (2, 14, 14, 32, 1, 3, 3, (1, 1), (1, 1), (1, 1)),   # 16 x 32 tiles (two 8-row blocks per warp)
    (1, 32, 16, 8, 1, 3, 3, (1, 1), (1, 1), (1, 1)),    # 32 x 16 tiles
    (1, 64, 8, 4, 1, 3, 3, (1, 1), (1, 1), (1, 1)),     # 64 x 8 tiles
    (2, 7, 7, 16, 1, 3, 3, (1, 1), (1, 1), (1, 1)),     # 7 x 7: the last MobileNet resolution
]
# 5x5 filters at unit stride: the tiled kernel with 8-channel tiles
TILED5 = [
    (2, 12, 70, 16, 1, 5, 5, (1, 1), (2, 2), (1, 1)),   # ragged row and column tiles
    (1, 14, 14, 8, 1, 5, 5, (1, 1), (2, 2), (1, 1)),    # 16 x 32 tiles
    (2, 9, 9, 12, 1, 5, 5, (1, 1), (0, 0), (1, 1)),     # no padding, 12 channels
    (1, 7, 40, 20, 1, 5, 5, (1, 1), (4, 1), (1, 1)),    # padding past the filter's reach in rows
]

DIRECT = [
    (2, 7, 6, 3, 1, 3, 3, (1, 1), (1, 1), (1, 1)),      # 3 channels: not a multiple of 4
    (1, 9, 8, 2, 3, 3, 2, (2, 1), (1, 0), (1, 1)),      # multiplier 3, stride 2
    (2, 8, 9, 4, 2, 3, 3, (1, 2), (2, 2), (2, 1)),      # multiplier 2, dilation
    (1, 10, 7, 3, 1, 5, 3, (3, 2), (2, 2), (1, 2)),
    (1, 5, 5, 5, 1, 1, 1, (1, 1), (0, 0), (1, 1)),      # pointwise
    (1, 12, 40, 8, 4, 3, 3, (1, 1), (1, 1), (1, 1)),    # 3x3 unit stride with multiplier 4
]

# 3x3 stride 2: the stride-2 tiled kernels (the data gradient's for padding 1
# only; other paddings take the direct kernel for that pass)
STRIDE2 = [
    (2, 16, 16, 32, 1, 3, 3, (2, 2), (1, 1), (1, 1)),   # the stride-2 MobileNet layer shape
    (1, 33, 130, 16, 1, 3, 3, (2, 2), (1, 1), (1, 1)),  # 17 x 65 outputs: ragged row and column tiles
    (2, 14, 14, 12, 1, 3, 3, (2, 2), (1, 1), (1, 1)),   # 12 channels: a half channel block
    (1, 17, 17, 8, 1, 3, 3, (2, 2), (0, 0), (1, 1)),    # no padding
    (1, 18, 130, 20, 1, 3, 3, (2, 2), (1, 1), (1, 1)),  # even height, 130 columns, 20 channels
]

PASSES = ("fwd", "bwd_data", "bwd_filter")


def dims(orc, g):
    N, H, W, C, D, R, S, st, pd, dl = g
    desc = orc.conv_desc(N, H, W, C, C * D, R, S, st, pd, dl)
    P, Q = orc.conv_out_hw(desc)
    return desc, P, Q


def operands(orc, g, rng):
    N, H, W, C, D, R, S, *_ = g
    _, P, Q = dims(orc, g)
    x = rng.standard_normal((N, H, W, C)).astype(np.float32)
    w = rng.standard_normal((R, S, C, D)).astype(np.float32)
    dy = rng.standard_normal((N, P, Q, C * D)).astype(np.float32)
    return x, w, dy


def out_shape(g, P, Q, which):
    N, H, W, C, D, R, S, *_ = g
    return ((N, P, Q, C * D), (N, H, W, C), (R, S, C, D))[which]


def run_dw(amd, lut, which, g, t0, t1, shape, scratch=True):
    import torch
    N, H, W, C, D, R, S, st, pd, dl = g
    desc = amd.ConvDesc.make(N, H, W, C, C * D, R, S, st, pd, dl)
    buf, out = guarded(shape)
    d0, d1 = to_dev(t0), to_dev(t1)
    nb = amd.amsim_dwconv2d_workspace_size(desc, which, lut)
    ws = amd.workspace(nb) if (scratch and nb) else None
    fn = (amd.amsim_dwconv2d_fwd, amd.amsim_dwconv2d_bwd_data, amd.amsim_dwconv2d_bwd_filter)[which]
    fn(desc, d0, d1, out, lut, ws=ws)
    torch.cuda.synchronize()
    path = amd.amsim_last_path()
    assert guards_intact(buf), "write outside the output"
    return out.cpu().numpy(), path


def oracle_pass(orc, kind, M, which, desc, t0, t1, n):
    fn = (orc.dwconv2d_fwd, orc.dwconv2d_bwd_data, orc.dwconv2d_bwd_filter)[which]
    return fn(kind, M, desc, t0, t1, np.arange(n))


def check_passes(amd, orc, lut, kind, M, g, x, w, dy, expect_path, scratch=True):
    """expect_path: one AMSIM_PATH_* bit for every pass, or a bit per pass."""
    desc, P, Q = dims(orc, g)
    args = ((x, w), (dy, w), (x, dy))
    expect = tuple(expect_path) if isinstance(expect_path, (tuple, list)) else (expect_path,) * 3
    for which in range(3):
        shape = out_shape(g, P, Q, which)
        got, path = run_dw(amd, lut, which, g, *args[which], shape, scratch)
        assert path & expect[which], (PASSES[which], g, path)
        ref, sa = oracle_pass(orc, kind, M, which, desc, *args[which], got.size)
        assert_close(got.reshape(-1), ref, sa, f"{PASSES[which]} {g} {kind} M={M}")


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
@pytest.mark.parametrize("g", TILED)
def test_dwconv_tiled_kernel(amd, orc, luts, g, kind):
    rng = np.random.default_rng(sum(g[:7]) + 7 * (kind == "exact"))
    x, w, dy = operands(orc, g, rng)
    check_passes(amd, orc, luts(kind, 7), kind, 7, g, x, w, dy, amd.AMSIM_PATH_DW_TILES)


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
@pytest.mark.parametrize("g", TILED5)
def test_dwconv_tiled_kernel_5x5(amd, orc, luts, g, kind):
    rng = np.random.default_rng(31 + sum(g[:7]) + 7 * (kind == "exact"))
    x, w, dy = operands(orc, g, rng)
    check_passes(amd, orc, luts(kind, 7), kind, 7, g, x, w, dy, amd.AMSIM_PATH_DW_TILES)


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
@pytest.mark.parametrize("g", DIRECT)
def test_dwconv_direct_kernel(amd, orc, luts, g, kind):
    rng = np.random.default_rng(3 + sum(g[:7]) + 7 * (kind == "exact"))
    x, w, dy = operands(orc, g, rng)
    check_passes(amd, orc, luts(kind, 7), kind, 7, g, x, w, dy, amd.AMSIM_PATH_DW_DIRECT)


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
@pytest.mark.parametrize("g", STRIDE2)
def test_dwconv_stride2_kernel(amd, orc, luts, g, kind):
    rng = np.random.default_rng(5 + sum(g[:7]) + 7 * (kind == "exact"))
    x, w, dy = operands(orc, g, rng)
    check_passes(amd, orc, luts(kind, 7), kind, 7, g, x, w, dy, stride2_paths(amd, g))


def stride2_paths(amd, g):
    t, d = amd.AMSIM_PATH_DW_TILES, amd.AMSIM_PATH_DW_DIRECT
    return (t, t if g[8] == (1, 1) else d, t)


@pytest.mark.parametrize("M,path", [(1, "tiles"), (4, "tiles"), (8, "direct"), (11, "direct")])
def test_dwconv_mantissa_widths(amd, orc, luts, M, path):
    """Narrow tables (8-bit, staged) and wide ones (16-bit 128 KB at M=8, 32-bit
    16 MB at M=11: read through the cache by the direct kernel)."""
    g = (1, 10, 20, 8, 1, 3, 3, (1, 1), (1, 1), (1, 1))
    rng = np.random.default_rng(40 + M)
    x, w, dy = operands(orc, g, rng)
    bit = amd.AMSIM_PATH_DW_TILES if path == "tiles" else amd.AMSIM_PATH_DW_DIRECT
    check_passes(amd, orc, luts("mitchell", M), "mitchell", M, g, x, w, dy, bit)


def sprinkle(a, rng, frac=0.03):
    """Replace a fraction of the entries by zeros, denormals, infinities, NaN
    and huge values (|x| >= 2^64: products may overflow)."""
    flat = a.reshape(-1).view(np.uint32).copy()
    n = flat.size
    specials = [0x00000000, 0x80000000, 0x00012345, 0x80400000, 0x7F800000, 0xFF800000, 0x7FC00000,
                0x60000000, 0xE1234567, 0x7E800000]
    idx = rng.choice(n, size=max(len(specials), int(frac * n)), replace=False)
    for j, i in enumerate(idx):
        flat[i] = specials[j % len(specials)]
    return flat.view(np.float32).reshape(a.shape)


@pytest.mark.parametrize("g", [TILED[0], TILED[1], TILED5[0], TILED5[2], DIRECT[1], STRIDE2[0], STRIDE2[3]])
def test_dwconv_special_operands(amd, orc, luts, g):
    """Zeros, denormals, infinities, NaN and overflowing products in every
    operand: the NaN pattern and infinities match exactly, the rest within the
    tolerance.  In the unpadded geometry the last activation columns are
    infinite: the weight gradient must not pair them with positions past the
    output gradient's edge."""
    rng = np.random.default_rng(77 + sum(g[:7]))
    x, w, dy = operands(orc, g, rng)
    x, w, dy = sprinkle(x, rng), sprinkle(w, rng, 0.05), sprinkle(dy, rng)
    if g[8] == (0, 0):
        x[0, 3, -1, :] = np.inf
        x[0, 4, -2, 1] = -np.inf
    t, d = amd.AMSIM_PATH_DW_TILES, amd.AMSIM_PATH_DW_DIRECT
    bit = t if (g in TILED or g in TILED5) else stride2_paths(amd, g) if g in STRIDE2 else d
    check_passes(amd, orc, luts("mitchell", 7), "mitchell", 7, g, x, w, dy, bit)


def test_dwconv_filter_gradient_scratch_and_determinism(amd, orc, luts):
    """The weight gradient with scratch (shares added by a second kernel) and
    without (one share per channel block): both match the oracle, and each is
    bit-identical across runs."""
    lut = luts("mitchell", 7)
    for g in (TILED[4], (4, 32, 32, 8, 2, 3, 3, (2, 2), (1, 1), (1, 1))):
        rng = np.random.default_rng(5)
        x, w, dy = operands(orc, g, rng)
        desc, P, Q = dims(orc, g)
        shape = out_shape(g, P, Q, 2)
        ref, sa = orc.dwconv2d_bwd_filter("mitchell", 7, desc, x, dy, np.arange(int(np.prod(shape))))
        for scratch in (True, False):
            a, path = run_dw(amd, lut, 2, g, x, dy, shape, scratch)
            b, _ = run_dw(amd, lut, 2, g, x, dy, shape, scratch)
            assert np.array_equal(bits(a), bits(b)), (g, scratch)
            assert bool(path & amd.AMSIM_PATH_STREAMK) == scratch, (g, scratch, path)
            assert_close(a.reshape(-1), ref, sa, f"bwd_filter {g} scratch={scratch}")


def test_dwconv_unaligned_tensors_take_direct_kernel(amd, orc, luts):
    """A tiled geometry whose tensors start 4 bytes off a 16-byte boundary runs
    on the direct kernel, with the same results within the tolerance."""
    import torch
    g = TILED[0]
    N, H, W, C, D, R, S, st, pd, dl = g
    desc = amd.ConvDesc.make(N, H, W, C, C * D, R, S, st, pd, dl)
    odesc, P, Q = dims(orc, g)
    lut = luts("mitchell", 7)
    rng = np.random.default_rng(9)
    x, w, dy = operands(orc, g, rng)

    def dev(a):
        buf = torch.empty(a.size + 4, dtype=torch.float32, device="cuda")
        v = buf[1:1 + a.size].view(*a.shape)
        v.copy_(torch.from_numpy(a).cuda())
        return v

    fns = (amd.amsim_dwconv2d_fwd, amd.amsim_dwconv2d_bwd_data, amd.amsim_dwconv2d_bwd_filter)
    args = ((x, w), (dy, w), (x, dy))
    for which in range(3):
        shape = out_shape(g, P, Q, which)
        out = dev(np.zeros(shape, np.float32))
        nb = amd.amsim_dwconv2d_workspace_size(desc, which, lut)
        fns[which](desc, dev(args[which][0]), dev(args[which][1]), out, lut,
                   ws=amd.workspace(nb) if nb else None)
        torch.cuda.synchronize()
        assert amd.amsim_last_path() & amd.AMSIM_PATH_DW_DIRECT
        ref, sa = oracle_pass(orc, "mitchell", 7, which, odesc, *args[which], out.numel())
        assert_close(out.cpu().numpy().reshape(-1), ref, sa, f"unaligned {PASSES[which]}")


def test_dwconv_empty_batch_and_errors(amd, luts):
    import torch
    lut = luts("mitchell", 7)
    # N == 0: nothing to compute forward; the weight gradient is all +0
    desc = amd.ConvDesc.make(0, 8, 8, 4, 4, 3, 3, (1, 1), (1, 1), (1, 1))
    dw = torch.full((3, 3, 4, 1), 5.0, device="cuda")
    amd.amsim_dwconv2d_fwd(desc, None, None, dw, lut)
    amd.amsim_dwconv2d_bwd_filter(desc, None, None, dw, lut)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dw.cpu().numpy()), np.zeros(36, np.uint32).reshape(3, 3, 4, 1))
    x = torch.zeros(1024, device="cuda")
    with pytest.raises(amd.AmsimError):      # K not a multiple of C
        amd.amsim_dwconv2d_fwd(amd.ConvDesc.make(1, 8, 8, 4, 6, 3, 3), x, x, x, lut)
    with pytest.raises(amd.AmsimError):      # filter larger than the padded input
        amd.amsim_dwconv2d_fwd(amd.ConvDesc.make(1, 2, 2, 4, 4, 5, 5), x, x, x, lut)
    with pytest.raises(amd.AmsimError):      # null operand
        amd.amsim_dwconv2d_bwd_data(amd.ConvDesc.make(1, 8, 8, 4, 4, 3, 3), None, x, x, lut)


def test_dwconv_mobilenet_layer_full_size(amd, orc, luts):
    """The 64x56x56x128 3x3 depthwise layer (stride 1, padding 1, Mitchell
    M=7) at full size, in the launch configuration the benchmark times:
    sampled outputs of the three passes against the oracle."""
    from approximate_multiplier_dnn_gb300 import steps
    from approximate_multiplier_dnn_gb300 import workloads as wl
    lut = luts("mitchell", 7)
    data = wl.dwconv3x3()
    geom = wl.DWCONV3X3
    st = steps.DwConvStep(data, geom, lut)
    st.run()
    import torch
    torch.cuda.synchronize()
    desc = orc.conv_desc(geom["N"], geom["H"], geom["W"], geom["C"], geom["C"] * geom["D"], geom["R"],
                         geom["S"], geom["stride"], geom["pad"], geom["dil"])
    rng = np.random.default_rng(0)
    y, dx, dw = st.y.cpu().numpy().reshape(-1), st.dx.cpu().numpy().reshape(-1), st.dw.cpu().numpy().reshape(-1)
    pts = np.unique(np.concatenate([rng.integers(0, y.size, 3000), [0, y.size - 1]]))
    ref, sa = orc.dwconv2d_fwd("mitchell", 7, desc, data["x"], data["w"], pts)
    assert_close(y[pts], ref, sa, "full-size fwd")
    pts = np.unique(np.concatenate([rng.integers(0, dx.size, 3000), [0, dx.size - 1]]))
    ref, sa = orc.dwconv2d_bwd_data("mitchell", 7, desc, data["dy"], data["w"], pts)
    assert_close(dx[pts], ref, sa, "full-size bwd_data")
    pts = np.unique(np.concatenate([rng.integers(0, dw.size, 96), [0, dw.size - 1]]))
    ref, sa = orc.dwconv2d_bwd_filter("mitchell", 7, desc, data["x"], data["dy"], pts)
    assert_close(dw[pts], ref, sa, "full-size bwd_filter")


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_dwconv_closed_form_equals_table(amd, orc, kind):
    """Closed-form products (amsim_lut_set_closed_form) in the tiled kernels
    (3x3 and 5x5 at stride 1, and the three stride-2 kernels) give the table path's
    results bit for bit, on ordinary operands and on tiles with special or
    tiny (nonzero, below 2^-63) values, which take the slow computation; and
    they stay within the oracle's tolerance."""
    lut_t = amd.Lut.build(kind, 7)
    lut_c = amd.Lut.build(kind, 7).set_closed_form(True)
    try:
        for g in (TILED[0], TILED[1], TILED[4], TILED5[0], TILED5[1], STRIDE2[0], STRIDE2[1], STRIDE2[4]):
            for specials in (False, True, "tiny"):
                rng = np.random.default_rng(11 + sum(g[:7]) + (specials is True) + 2 * (specials == "tiny"))
                x, w, dy = operands(orc, g, rng)
                if specials is True:
                    x, w, dy = sprinkle(x, rng), sprinkle(w, rng, 0.05), sprinkle(dy, rng)
                if specials:
                    # nonzero magnitudes below 2^-63: the slow products of the closed form
                    x.reshape(-1)[::97] = np.float32(3e-20)
                    dy.reshape(-1)[::89] = np.float32(-5e-21)
                desc, P, Q = dims(orc, g)
                args = ((x, w), (dy, w), (x, dy))
                for which in range(3):
                    shape = out_shape(g, P, Q, which)
                    a, pa = run_dw(amd, lut_t, which, g, *args[which], shape)
                    b, pb = run_dw(amd, lut_c, which, g, *args[which], shape)
                    assert pa & amd.AMSIM_PATH_DW_TILES and not pa & amd.AMSIM_PATH_CLOSED_FORM, pa
                    assert pb & amd.AMSIM_PATH_DW_TILES and pb & amd.AMSIM_PATH_CLOSED_FORM, pb
                    ba, bb = bits(a), bits(b)
                    both_nan = np.isnan(a) & np.isnan(b)
                    assert np.array_equal(ba[~both_nan], bb[~both_nan]), (kind, g, specials, PASSES[which])
                    assert np.array_equal(np.isnan(a), np.isnan(b))
                    ref, sa = oracle_pass(orc, kind, 7, which, desc, *args[which], b.size)
                    got = b.reshape(-1)
                    if specials is True and g[5] == 5:
                        # 25 products near the top of the fp32 range: a partial sum may overflow to an
                        # infinity in one summation order and not in another, then meet the opposite
                        # infinity (a NaN in one order only).  Outputs finite on both sides are still
                        # held to the oracle; the "tiny" case checks the slow products of 5x5 tiles
                        # against it in full.
                        fin = np.isfinite(ref) & np.isfinite(got)
                        assert_close(got[fin], ref[fin], sa[fin], f"closed form {kind} {PASSES[which]} {g} (finite)")
                        continue
                    assert_close(got, ref, sa, f"closed form {kind} {PASSES[which]} {g}")
    finally:
        lut_t.close()
        lut_c.close()
