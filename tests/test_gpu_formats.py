"""(1, e, m) multipliers with fewer exponent bits than fp32 (ApproxTrain Sec.
V-B, last paragraph: e from 1 to 8 given an exponent casting function) on the
GPU against the oracle, which carries the same reading of the cast (IEEE-style
bias 2^(e-1) - 1, operands below the format's range become zeros and above it
infinities, Algorithm 2 with that bias, the product returned as fp32).

Elementwise products are compared bit for bit; contractions (GEMM in every
transpose, batched, grouped and phased calls, Conv2D's three passes,
depthwise Conv2D's three passes) within the contraction tolerance.  Operand
magnitudes span several binades past both ends of each format's range, so
the cast's zeros and infinities, Algorithm 2's zero test and its overflow
(with and without the carry) all occur."""
import numpy as np
import pytest

from gpu_helpers import assert_close, bits, to_dev

pytestmark = pytest.mark.gpu


def spread(rng, shape, E):
    """N(0,1) values scaled by 2^u, u uniform over the format's exponent range
    widened by a few binades on each side."""
    B = (1 << (E - 1)) - 1
    lo, hi = -B - 3, B + 3
    u = rng.integers(lo, hi + 1, size=shape)
    return (rng.standard_normal(shape) * np.exp2(u)).astype(np.float32)


@pytest.fixture(scope="module")
def fmt_lut(amd):
    cache = {}

    def get(kind, M, E):
        key = (kind, M)
        if key not in cache:
            cache[key] = amd.Lut.build(kind, M)
        lut = cache[key]
        lut.set_exponent_bits(E)
        return lut
    yield get
    for v in cache.values():
        v.close()


@pytest.mark.parametrize("E", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("kind,M", [("mitchell", 7), ("exact", 7), ("exact", 10)])
def test_elementwise_bit_exact(amd, orc, fmt_lut, E, kind, M):
    import torch
    lut = fmt_lut(kind, M, E)
    rng = np.random.default_rng(10 * E + M)
    n = 1 << 17
    a = spread(rng, n, E)
    b = spread(rng, n, E)
    u = rng.integers(0, 1 << 32, size=(2, 4096), dtype=np.uint64).astype(np.uint32).view(np.float32)
    a[:4096], b[:4096] = u[0], u[1]                 # any bit pattern: NaN, Inf, denormals
    c = torch.empty(n, dtype=torch.float32, device="cuda")
    amd.amsim_mul(to_dev(a), to_dev(b), c, n, lut)
    torch.cuda.synchronize()
    want = orc.mul(kind, M, a, b, ebits=E)
    assert np.array_equal(bits(c.cpu().numpy()), bits(want))
    if E < 8:
        w = want.astype(np.float64)
        assert (w == 0).sum() > 1000 and np.isinf(w).sum() > 1000


@pytest.mark.parametrize("E", [2, 4, 5, 7])
@pytest.mark.parametrize("trans", ["NN", "NT", "TN", "TT"])
def test_gemm_each_transpose(amd, orc, fmt_lut, E, trans):
    import torch
    lut = fmt_lut("mitchell", 7, E)
    rng = np.random.default_rng(E * 7 + len(trans))
    m, n, k = 130, 300, 75
    A = spread(rng, (m, k), E) * np.float32(2.0 ** -3)
    B = spread(rng, (k, n), E) * np.float32(2.0 ** -3)
    tA, tB = trans[0] == "T", trans[1] == "T"
    Ad = A.T.copy() if tA else A
    Bd = B.T.copy() if tB else B
    C = amd.gemm(to_dev(Ad), to_dev(Bd), lut, transA=tA, transB=tB)
    torch.cuda.synchronize()
    path = amd.amsim_last_path()
    assert path & (amd.AMSIM_PATH_INKERNEL_DECODE | amd.AMSIM_PATH_SINGLE_ROLE), path
    assert not path & (amd.AMSIM_PATH_RAW_TILES | amd.AMSIM_PATH_PLANES), path
    ref, sa = orc.gemm("mitchell", 7, Ad, Bd, transA=tA, transB=tB, ebits=E)
    assert_close(C.cpu().numpy(), ref, sa, f"E={E} {trans}")


def test_gemm_large_stream_k_and_no_scratch(amd, orc, fmt_lut):
    """A multi-wave problem (stream-K partial sums) and the same without scratch."""
    import torch
    E = 5
    lut = fmt_lut("exact", 10, E)
    rng = np.random.default_rng(3)
    m, n, k = 700, 900, 1000
    A = spread(rng, (m, k), E) * np.float32(2.0 ** -4)
    B = spread(rng, (k, n), E) * np.float32(2.0 ** -4)
    rows = np.array([0, 1, 350, 699])
    ref, sa = orc.gemm("exact", 10, A, B, rows=rows, ebits=E)
    dA, dB = to_dev(A), to_dev(B)
    for ws_kind in ("auto", "none"):
        C = torch.empty((m, n), dtype=torch.float32, device="cuda")
        nb = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut) if ws_kind == "auto" else 0
        amd.amsim_gemm("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, C, n, lut,
                       ws=amd.workspace(nb) if nb else None, ws_bytes=nb)
        torch.cuda.synchronize()
        assert_close(C.cpu().numpy()[rows], ref, sa, f"E=5 {ws_kind}")


def test_batched_grouped_and_phased(amd, orc, fmt_lut):
    import torch
    from approximate_multiplier_dnn_gb300 import GemmProblem
    E = 4
    lut = fmt_lut("mitchell", 7, E)
    rng = np.random.default_rng(4)
    bt, m, n, k = 3, 64, 80, 48
    Q = spread(rng, (bt, m, k), E) * np.float32(0.125)
    K = spread(rng, (bt, n, k), E) * np.float32(0.125)
    S = torch.empty((bt, m, n), dtype=torch.float32, device="cuda")
    nb = amd.amsim_gemm_workspace_size("N", "T", m, n, k, bt, lut)
    dQ, dK = to_dev(Q), to_dev(K)
    amd.amsim_gemm_strided_batched("N", "T", m, n, k, 0.5, dQ, k, m * k, dK, k, n * k, 0.0, S, n, m * n, bt, lut,
                                   ws=amd.workspace(nb))
    torch.cuda.synchronize()
    for b in range(bt):
        ref, sa = orc.gemm("mitchell", 7, Q[b], K[b], transB=True, alpha=0.5, ebits=E)
        assert_close(S.cpu().numpy()[b], ref, 0.5 * sa, f"batched {b}")
    # phased: two phases, the second reading the first's output (runs phase by phase)
    X = spread(rng, (200, 150), E) * np.float32(0.25)
    W1 = spread(rng, (150, 120), E) * np.float32(0.25)
    W2 = spread(rng, (120, 90), E) * np.float32(0.25)
    dX, dW1, dW2 = to_dev(X), to_dev(W1), to_dev(W2)
    Y1 = torch.empty((200, 120), device="cuda")
    Y2 = torch.empty((200, 90), device="cuda")
    probs = [GemmProblem.make("N", "N", 200, 120, 150, 1.0, dX, 150, dW1, 120, 0.0, Y1, 120),
             GemmProblem.make("N", "N", 200, 90, 120, 1.0, Y1, 120, dW2, 90, 0.0, Y2, 90)]
    ws = amd.workspace(amd.amsim_gemm_phased_workspace_size(probs, [0, 1], [0, 1], lut))
    amd.amsim_gemm_phased(probs, [0, 1], [0, 1], lut, ws=ws)
    torch.cuda.synchronize()
    assert not amd.amsim_last_path() & amd.AMSIM_PATH_PHASED
    y1 = Y1.cpu().numpy()
    ref, sa = orc.gemm("mitchell", 7, X, W1, ebits=E)
    assert_close(y1, ref, sa, "phased Y1")
    ref, sa = orc.gemm("mitchell", 7, y1, W2, ebits=E)
    assert_close(Y2.cpu().numpy(), ref, sa, "phased Y2")


@pytest.mark.parametrize("E", [3, 5])
def test_conv_all_passes(amd, orc, fmt_lut, E):
    import torch
    lut = fmt_lut("exact", 7, E)
    rng = np.random.default_rng(E)
    N, H, W, C, K, R, S = 2, 9, 10, 16, 24, 3, 3
    desc = amd.ConvDesc.make(N, H, W, C, K, R, S, (1, 1), (1, 1), (1, 1))
    od = orc.conv_desc(N, H, W, C, K, R, S, (1, 1), (1, 1), (1, 1))
    P, Q = amd.amsim_conv2d_out_hw(desc)
    x = spread(rng, (N, H, W, C), E) * np.float32(0.25)
    w = spread(rng, (R, S, C, K), E) * np.float32(0.25)
    dy = spread(rng, (N, P, Q, K), E) * np.float32(0.25)
    outs = [torch.empty(s, dtype=torch.float32, device="cuda") for s in ((N, P, Q, K), (N, H, W, C), (R, S, C, K))]
    fns = (amd.amsim_conv2d_fwd, amd.amsim_conv2d_bwd_data, amd.amsim_conv2d_bwd_filter)
    args = ((x, w), (dy, w), (x, dy))
    for which in range(3):
        nb = amd.amsim_conv2d_workspace_size(desc, which, lut)
        a0, a1 = to_dev(args[which][0]), to_dev(args[which][1])
        fns[which](desc, a0, a1, outs[which], lut, ws=amd.workspace(nb))
        torch.cuda.synchronize()
        assert not amd.amsim_last_path() & amd.AMSIM_PATH_RAW_TILES
    for which, fn in enumerate((orc.conv2d_fwd, orc.conv2d_bwd_data, orc.conv2d_bwd_filter)):
        got = outs[which].cpu().numpy().reshape(-1)
        ref, sa = fn("exact", 7, od, args[which][0], args[which][1], np.arange(got.size), ebits=E)
        assert_close(got, ref, sa, f"conv E={E} pass {which}")


@pytest.mark.parametrize("E", [4, 6])
def test_depthwise_all_passes(amd, orc, fmt_lut, E):
    import torch
    lut = fmt_lut("mitchell", 7, E)
    rng = np.random.default_rng(30 + E)
    N, H, W, C, R, S = 2, 11, 12, 32, 3, 3
    desc = amd.ConvDesc.make(N, H, W, C, C, R, S, (1, 1), (1, 1), (1, 1))
    od = orc.conv_desc(N, H, W, C, C, R, S, (1, 1), (1, 1), (1, 1))
    x = spread(rng, (N, H, W, C), E) * np.float32(0.5)
    w = spread(rng, (R, S, C, 1), E) * np.float32(0.5)
    w[0, 0, 3, 0] = np.float32(2.0 ** 60)          # finite in fp32, infinite in the format (padded taps -> NaN)
    dy = spread(rng, (N, H, W, C), E) * np.float32(0.5)
    outs = [torch.empty(s, dtype=torch.float32, device="cuda") for s in ((N, H, W, C), (N, H, W, C), (R, S, C, 1))]
    fns = (amd.amsim_dwconv2d_fwd, amd.amsim_dwconv2d_bwd_data, amd.amsim_dwconv2d_bwd_filter)
    args = ((x, w), (dy, w), (x, dy))
    for which in range(3):
        nb = amd.amsim_dwconv2d_workspace_size(desc, which, lut)
        a0, a1 = to_dev(args[which][0]), to_dev(args[which][1])
        fns[which](desc, a0, a1, outs[which], lut, ws=amd.workspace(nb) if nb else None, ws_bytes=nb)
        torch.cuda.synchronize()
        assert amd.amsim_last_path() & amd.AMSIM_PATH_DW_DIRECT, amd.amsim_last_path()
    for which, fn in enumerate((orc.dwconv2d_fwd, orc.dwconv2d_bwd_data, orc.dwconv2d_bwd_filter)):
        got = outs[which].cpu().numpy().reshape(-1)
        ref, sa = fn("mitchell", 7, od, args[which][0], args[which][1], np.arange(got.size), ebits=E)
        assert_close(got, ref, sa, f"depthwise E={E} pass {which}")


def test_exponent_setting_rules(amd, luts):
    lut = amd.Lut.build("mitchell", 7)
    try:
        L = amd.lib()
        assert L.amsim_lut_set_exponent_bits(lut.handle, 0) == amd.AMSIM_EUNSUPPORTED
        assert L.amsim_lut_set_exponent_bits(lut.handle, 9) == amd.AMSIM_EUNSUPPORTED
        lut.set_closed_form(True)
        assert L.amsim_lut_set_exponent_bits(lut.handle, 5) == amd.AMSIM_EUNSUPPORTED
        lut.set_closed_form(False)
        lut.set_exponent_bits(5)
        assert L.amsim_lut_set_closed_form(lut.handle, 1) == amd.AMSIM_EUNSUPPORTED
        lut.set_exponent_bits(8)
        lut.set_closed_form(True)
    finally:
        lut.close()
    assert amd.lib().amsim_lut_set_exponent_bits(None, 5) == amd.AMSIM_EINVAL
