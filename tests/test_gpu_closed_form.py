"""Closed-form products (amsim_lut_set_closed_form): the raw-tile kernel
computes Mitchell's and the exact product's mantissa factor in registers
instead of reading the table.  The closed forms equal the table's entries bit
for bit (pinned on the CPU against the oracle's tables), and the kernel's
summation order does not depend on where a product value comes from, so every
output must equal the table path's bit for bit on the same plan -- and match
the oracle like any other output."""
import numpy as np
import pytest

from gpu_helpers import REL, assert_close, bits, guarded, guards_intact, to_dev
from approximate_multiplier_dnn_gb300 import GemmProblem

pytestmark = pytest.mark.gpu


def rnd(rng, shape):
    return rng.standard_normal(shape).astype(np.float32)


def host(t):
    return t.detach().cpu().numpy()


@pytest.fixture(scope="module")
def cf(amd):
    """Closed-form handles, one per (kind, M), apart from the table handles."""
    cache = {}

    def get(kind, M):
        if (kind, M) not in cache:
            cache[(kind, M)] = amd.Lut.build(kind, M).set_closed_form(True)
        return cache[(kind, M)]

    yield get
    for v in cache.values():
        v.close()


def same_bits(a, b, what):
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    assert np.array_equal(na, nb), f"{what}: NaN pattern differs"
    diff = bits(np.where(na, 0, a)) != bits(np.where(nb, 0, b))
    assert not diff.any(), f"{what}: {diff.sum()} of {a.size} elements differ"


def gemm(amd, lut, A, B, m, n, k, ta=False, tb=False, alpha=1.0, beta=0.0, C0=None, lda=None, ldb=None,
         use_ws=True):
    import torch
    lda = lda or A.shape[1]
    ldb = ldb or B.shape[1]
    Cb, C = guarded((m, n), np.zeros((m, n), np.float32) if C0 is None else C0)
    tA, tB = ("T" if ta else "N"), ("T" if tb else "N")
    ws = amd.workspace(amd.amsim_gemm_workspace_size(tA, tB, m, n, k, 1, lut)) if use_ws else None
    amd.amsim_gemm(tA, tB, m, n, k, alpha, A, lda, B, ldb, beta, C, n, lut, ws=ws)
    torch.cuda.synchronize()
    path = amd.amsim_last_path()
    assert guards_intact(Cb)
    return host(C), path


@pytest.mark.parametrize("kind,M", [("mitchell", 7), ("exact", 7), ("mitchell", 3), ("exact", 11),
                                    ("mitchell", 11), ("exact", 1)])
def test_closed_form_gemm_equals_table(amd, orc, luts, cf, kind, M):
    rng = np.random.default_rng(60 + M)
    m, n, k = 300, 520, 700
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    Ad, Bd = to_dev(A), to_dev(B)
    got_t, path_t = gemm(amd, luts(kind, M), Ad, Bd, m, n, k)
    got_c, path_c = gemm(amd, cf(kind, M), Ad, Bd, m, n, k)
    assert path_t & amd.AMSIM_PATH_RAW_TILES and not path_t & amd.AMSIM_PATH_CLOSED_FORM, path_t
    assert path_c & amd.AMSIM_PATH_RAW_TILES and path_c & amd.AMSIM_PATH_CLOSED_FORM, path_c
    same_bits(got_c, got_t, "C")
    ref, sa = orc.gemm(kind, M, A, B)
    assert_close(got_c, ref, sa, "C")


@pytest.mark.parametrize("ta,tb", [(True, False), (False, True), (True, True)])
def test_closed_form_transposes_alpha_beta_no_scratch(amd, orc, luts, cf, ta, tb):
    """Transposed operands, alpha/beta, and a launch without scratch (one CTA
    per tile, no stream-K) on a ragged shape."""
    rng = np.random.default_rng(70)
    m, n, k = 197, 333, 451
    A = rnd(rng, (k, m) if ta else (m, k))
    B = rnd(rng, (n, k) if tb else (k, n))
    C0 = rnd(rng, (m, n))
    Ad, Bd = to_dev(A), to_dev(B)
    for use_ws in (True, False):
        got_t, _ = gemm(amd, luts("mitchell", 7), Ad, Bd, m, n, k, ta, tb, 0.5, -1.25, C0, use_ws=use_ws)
        got_c, path = gemm(amd, cf("mitchell", 7), Ad, Bd, m, n, k, ta, tb, 0.5, -1.25, C0, use_ws=use_ws)
        assert path & amd.AMSIM_PATH_CLOSED_FORM, path
        same_bits(got_c, got_t, f"C ws={use_ws}")
    ref, sa = orc.gemm("mitchell", 7, A, B, transA=ta, transB=tb, alpha=0.5, beta=-1.25, C0=C0)
    # beta C0 is one rounding of an exact scaling, not a sum of products
    assert_close(got_c, ref, 0.5 * sa + 1.25 * np.abs(C0.astype(np.float64)) / REL * 2.0 ** -23 + 1e-30, "C")


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_closed_form_special_values(amd, orc, luts, cf, kind):
    """Zeros, denormals, infinities, NaN and operands of magnitude >= 2^64
    (the kernel's rounded-product stages) give the table's results."""
    rng = np.random.default_rng(71)
    m, n, k = 130, 260, 300
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    A[3, :40] = 0.0
    A[5, 7] = -0.0
    A[9, 10:20] = np.float32(1e-40)                 # denormal: counts as zero
    A[11, 3] = np.inf
    B[3, 17] = 0.0                                  # inf * 0 -> NaN in row 11, column 17
    A[20, 5] = np.nan
    A[40, 1] = np.float32(3e19)                     # >= 2^64
    B[1, 30] = np.float32(-2e19)                    # product overflows to -inf
    B[2, :] = np.float32(1e-39)
    # magnitudes at the fast stages' lower edge: 2^-63 x 2^-63 products are the
    # smallest normals; 2^-64 x 2^-64 ones fall below and are zero
    j = np.arange(k, dtype=np.float32)
    A[50, :] = np.ldexp(1.0 + (j % 8) / 8.0, -63).astype(np.float32)
    B[:, 60] = np.ldexp(1.0 + (j % 5) / 4.0, -63).astype(np.float32)
    A[60, :] = np.ldexp(1.0 + (j % 3) / 2.0, -64).astype(np.float32)
    B[:, 70] = np.float32(2.0 ** -64)
    # NaN with payloads (signalling, and negative quiet)
    A[70, 9] = np.array([0x7F800001], np.uint32).view(np.float32)[0]
    B[10, 80] = np.array([0xFFC00001], np.uint32).view(np.float32)[0]
    Ad, Bd = to_dev(A), to_dev(B)
    got_t, _ = gemm(amd, luts(kind, 7), Ad, Bd, m, n, k)
    got_c, path = gemm(amd, cf(kind, 7), Ad, Bd, m, n, k)
    assert path & amd.AMSIM_PATH_CLOSED_FORM, path
    same_bits(got_c, got_t, "C")
    ref, sa = orc.gemm(kind, 7, A, B)
    assert_close(got_c, ref, sa, "C")
    assert got_c[60, 70] == 0.0 and 0.0 < abs(got_c[50, 60]) < 1e-33
    assert np.isnan(got_c[70]).all() and np.isnan(got_c[:, 80]).all()


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_closed_form_conv2d_equals_table(amd, orc, luts, cf, kind):
    import torch
    rng = np.random.default_rng(72)
    # a geometry all three passes read as tensor boxes (whole output rows per
    # tile, channels in multiples of 16 and 64)
    N, H, W, C, K, R, S = 2, 16, 16, 64, 32, 3, 3
    desc = amd.ConvDesc.make(N, H, W, C, K, R, S, (1, 1), (1, 1), (1, 1))
    P, Q = amd.amsim_conv2d_out_hw(desc)
    x, w = rnd(rng, (N, H, W, C)), rnd(rng, (R, S, C, K)) * 0.1
    dy = rnd(rng, (N, P, Q, K))
    xd, wd, dyd = to_dev(x), to_dev(w), to_dev(dy)
    res = {}
    for name, lut in (("table", luts(kind, 7)), ("closed", cf(kind, 7))):
        y = torch.empty((N, P, Q, K), device="cuda")
        dx = torch.empty_like(xd)
        dw = torch.empty_like(wd)
        paths = []
        for mode, fn, args in ((0, amd.amsim_conv2d_fwd, (xd, wd, y)), (1, amd.amsim_conv2d_bwd_data, (dyd, wd, dx)),
                               (2, amd.amsim_conv2d_bwd_filter, (xd, dyd, dw))):
            ws = amd.workspace(amd.amsim_conv2d_workspace_size(desc, mode, lut))
            fn(desc, *args, lut, ws=ws)
            torch.cuda.synchronize()
            paths.append(amd.amsim_last_path())
        res[name] = (host(y), host(dx), host(dw), paths)
    for p in res["closed"][3]:
        assert p & amd.AMSIM_PATH_CLOSED_FORM and p & amd.AMSIM_PATH_CONV_BOXES, p
    for i, what in enumerate(("y", "dx", "dw")):
        same_bits(res["closed"][i], res["table"][i], what)
    od = orc.conv_desc(N, H, W, C, K, R, S, (1, 1), (1, 1), (1, 1))
    ref, sa = orc.conv2d_fwd(kind, 7, od, x, w, np.arange(N * P * Q * K))
    assert_close(res["closed"][0].reshape(-1), ref, sa, "y")
    ref, sa = orc.conv2d_bwd_data(kind, 7, od, dy, w, np.arange(x.size))
    assert_close(res["closed"][1].reshape(-1), ref, sa, "dx")
    ref, sa = orc.conv2d_bwd_filter(kind, 7, od, x, dy, np.arange(w.size))
    assert_close(res["closed"][2].reshape(-1), ref, sa, "dw")


def test_closed_form_phased(amd, orc, cf):
    """Phased launches compute closed-form products too; a phase reading the
    previous one's output is checked on the GPU's copy of it."""
    import torch
    rng = np.random.default_rng(73)
    lut = cf("mitchell", 7)
    m = 256
    X = rnd(rng, (m, 784))
    W1, W2 = (rnd(rng, (784, 1000)) / 28).astype(np.float32), (rnd(rng, (1000, 500)) / 32).astype(np.float32)
    E, F = rnd(rng, (300, 520)), rnd(rng, (520, 700))
    Xd, W1d, W2d, Ed, Fd = (to_dev(a) for a in (X, W1, W2, E, F))
    Y1b, Y1 = guarded((m, 1000), np.full((m, 1000), np.nan, np.float32))
    Db, D = guarded((300, 700), np.full((300, 700), np.nan, np.float32))
    Y2b, Y2 = guarded((m, 500), np.full((m, 500), np.nan, np.float32))
    probs = [GemmProblem.make("N", "N", m, 1000, 784, 1.0, Xd, 784, W1d, 1000, 0.0, Y1, 1000),
             GemmProblem.make("N", "N", 300, 700, 520, 1.0, Ed, 520, Fd, 700, 0.0, D, 700),
             GemmProblem.make("N", "N", m, 500, 1000, 1.0, Y1, 1000, W2d, 500, 0.0, Y2, 500)]
    first, after = [0, 2], [0, 1]
    ws = amd.workspace(amd.amsim_gemm_phased_workspace_size(probs, first, after, lut))
    amd.amsim_gemm_phased(probs, first, after, lut, ws=ws)
    torch.cuda.synchronize()
    path = amd.amsim_last_path()
    assert path & amd.AMSIM_PATH_PHASED and path & amd.AMSIM_PATH_CLOSED_FORM, path
    assert guards_intact(Y1b) and guards_intact(Db) and guards_intact(Y2b)
    y1 = host(Y1)
    for got, A, B, what in ((y1, X, W1, "Y1"), (host(D), E, F, "D"), (host(Y2), y1, W2, "Y2")):
        ref, sa = orc.gemm("mitchell", 7, A, B)
        assert_close(got, ref, sa, what)


def test_closed_form_other_paths_use_the_table(amd, orc, luts, cf):
    """An operand the raw-tile kernel cannot copy (a row stride that is not a
    multiple of 4 floats, too large for plain loads) takes another kernel path,
    which reads the table: same results, no closed-form path bit."""
    rng = np.random.default_rng(74)
    m, n, k = 600, 256, 700
    Afull = rnd(rng, (m, k + 1))
    B = rnd(rng, (k, n))
    Ad, Bd = to_dev(Afull), to_dev(B)
    got_t, _ = gemm(amd, luts("mitchell", 7), Ad, Bd, m, n, k, lda=k + 1)
    got_c, path = gemm(amd, cf("mitchell", 7), Ad, Bd, m, n, k, lda=k + 1)
    assert not path & amd.AMSIM_PATH_RAW_TILES and not path & amd.AMSIM_PATH_CLOSED_FORM, path
    same_bits(got_c, got_t, "C")
    ref, sa = orc.gemm("mitchell", 7, Afull[:, :k], B)
    assert_close(got_c, ref, sa, "C")


def test_closed_form_switch(amd, luts):
    """Only kind-built handles take the closed form; switching it off restores
    the table path."""
    import torch
    e = amd.amsim_lut_generate("mitchell", 5)
    user = amd.Lut.from_entries(e, 5)
    with pytest.raises(amd.AmsimError) as exc:
        user.set_closed_form(True)
    assert exc.value.status == amd.AMSIM_EUNSUPPORTED
    user.set_closed_form(False)
    h = amd.Lut.build("exact", 5)
    A = torch.randn((64, 96), device="cuda")
    B = torch.randn((96, 80), device="cuda")
    got = []
    for on in (True, False):
        h.set_closed_form(on)
        C, path = gemm(amd, h, A, B, 64, 80, 96)
        assert bool(path & amd.AMSIM_PATH_CLOSED_FORM) == on, path
        got.append(C)
    same_bits(got[0], got[1], "C")
    user.close()
    h.close()
