"""Tail tiles of the raw-tile kernel: a tile whose real lane columns all lie in
its first 128 (the last lane tile of an L extent such as a 3x3 filter
gradient's R*S*C = 576 = 2 x 256 + 64) is computed by all eight consumer warps
as eight blocks of 8 rows, instead of four warps of 16 rows with four idle:
four columns per lane, or two (lane * 2, lane * 2 + 1) when at most 64
columns are real.
Each output's products are still summed in the same order, so the results
are bit-identical to the in-kernel-decode kernel's regular layout; cut tiles
(stream-K, with shares cut by stage cost) reduce partial sums written in that
layout, checked against the oracle."""
import numpy as np
import pytest

from gpu_helpers import REL, assert_close, to_dev
from approximate_multiplier_dnn_gb300 import GemmProblem

pytestmark = pytest.mark.gpu


def rnd(rng, shape):
    return rng.standard_normal(shape).astype(np.float32)


def batched(amd, lut, A, lda, B, m, n, k, batch, ws=None):
    """C[b] = A[b] B[b] with A[b] m x k (leading dimension lda), B[b] k x n."""
    import torch
    C = torch.full((batch, m, n), float("nan"), dtype=torch.float32, device="cuda")
    amd.amsim_gemm_strided_batched("N", "N", m, n, k, 1.0, A, lda, A.shape[1] * lda, B, n, k * n, 0.0, C, n,
                                   m * n, batch, lut, ws=ws)
    torch.cuda.synchronize()
    return C.cpu().numpy(), amd.amsim_last_path()


@pytest.mark.parametrize("values", ["normal", "zeros"])
@pytest.mark.parametrize("n", [320, 260, 300, 340, 384])
def test_tail_layout_bit_identical_to_regular_layout(amd, luts, n, values):
    """One wave of whole tiles (no stream-K): 64 x n per batch entry, the
    second lane tile a tail (n - 256 <= 128 real columns; two columns per lane
    up to 64).  Aligned operands
    take the raw-tile kernel (tail layout); the same operands behind a leading
    dimension of k + 1 take the in-kernel-decode kernel (regular layout).
    With ReLU-like zeros the folded form reads the table's zero row."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    batch = max(sms // 2, 1)
    m, k = 64, 256
    rng = np.random.default_rng(n + (7 if values == "zeros" else 0))
    A = rnd(rng, (batch, m, k))
    B = rnd(rng, (batch, k, n))
    if values == "zeros":
        A[A < 0] = 0.0
        B[B < -0.3] = -0.0
    lut = luts("mitchell", 7)
    dA, dB = to_dev(A), to_dev(B)
    raw, path_raw = batched(amd, lut, dA, k, dB, m, n, k, batch)
    assert path_raw & amd.AMSIM_PATH_RAW_TILES and not path_raw & amd.AMSIM_PATH_STREAMK, path_raw
    wide = torch.zeros((batch, m, k + 1), dtype=torch.float32, device="cuda")
    wide[:, :, :k] = dA
    reg, path_reg = batched(amd, lut, wide, k + 1, dB, m, n, k, batch)
    assert path_reg & amd.AMSIM_PATH_INKERNEL_DECODE and not path_reg & amd.AMSIM_PATH_STREAMK, path_reg
    assert np.array_equal(raw.view(np.uint32), reg.view(np.uint32))


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
@pytest.mark.parametrize("m,n,k", [(64, 320, 20000), (50, 300, 9000), (64, 116, 30000), (64, 360, 20000)])
def test_tail_tiles_cut_by_stream_k(amd, orc, luts, kind, m, n, k):
    """Few tiles over a long reduction: stream-K cuts the tail tile among many
    CTAs, whose partial sums (tail layout) the fused reduction adds; U rows
    past the edge (m = 50) leave the last row block's warps idle."""
    import torch
    rng = np.random.default_rng(m + n + k)
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    lut = luts(kind, 7)
    nb = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut)
    C = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    amd.amsim_gemm("N", "N", m, n, k, 1.0, to_dev(A), k, to_dev(B), n, 0.0, C, n, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    taken = amd.amsim_last_path()
    assert taken & amd.AMSIM_PATH_RAW_TILES and taken & amd.AMSIM_PATH_STREAMK, taken
    got = C.cpu().numpy()
    rows = np.array([0, 7, 8, m // 2, m - 1])
    ref, sa = orc.gemm(kind, 7, A, B, rows=rows)
    assert_close(got[rows], ref, sa, f"stream-K tail {m}x{n}x{k} {kind}")


@pytest.mark.parametrize("n", [300, 360])
def test_tail_tiles_with_special_operands(amd, orc, luts, n):
    """Zeros, denormals, infinities, NaN and |x| >= 2^64 in a tail tile: the
    per-stage flags pick the rounding products in the tail layouts too."""
    import torch
    from approximate_multiplier_dnn_gb300 import workloads as wl
    m, k = 64, 256
    rng = np.random.default_rng(23)
    a, b = wl.special_values_mix(m * k + k * n, seed=24)
    A = a[:m * k].reshape(m, k).copy()
    B = b[m * k:].reshape(k, n).copy()
    A[:, :] = np.where(rng.random(A.shape) < 0.95, rng.standard_normal(A.shape), A).astype(np.float32)
    B[:, :] = np.where(rng.random(B.shape) < 0.95, rng.standard_normal(B.shape), B).astype(np.float32)
    for kind in ("mitchell", "exact"):
        lut = luts(kind, 7)
        C = torch.empty((m, n), dtype=torch.float32, device="cuda")
        amd.amsim_gemm("N", "N", m, n, k, 1.0, to_dev(A), k, to_dev(B), n, 0.0, C, n, lut)
        torch.cuda.synchronize()
        assert amd.amsim_last_path() & amd.AMSIM_PATH_RAW_TILES
        ref, sa = orc.gemm(kind, 7, A, B)
        assert_close(C.cpu().numpy(), ref, sa + 1e-30, f"tail specials {kind}")


def test_tail_tiles_in_a_phased_launch(amd, orc, luts):
    """A phased launch whose first phase is a 64 x 576 x 8192 GEMM (a 3x3
    filter gradient's shape: its third lane tile is a tail, cut among CTAs;
    phased launches compute it in the regular layout, with the cost model
    for that layout) and whose second reads its output: checked against the
    oracle, and two calls are bit-identical (the last part to arrive adds the
    parts in CTA order)."""
    import torch
    rng = np.random.default_rng(25)
    m, n, k = 64, 576, 8192
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    W2 = rnd(rng, (n, 72))
    lut = luts("mitchell", 7)
    dA, dB, dW2 = to_dev(A), to_dev(B), to_dev(W2)
    outs = []
    for _ in range(2):
        C1 = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        C2 = torch.full((m, 72), float("nan"), dtype=torch.float32, device="cuda")
        probs = [GemmProblem.make("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, C1, n),
                 GemmProblem.make("N", "N", m, 72, n, 1.0, C1, n, dW2, 72, 0.0, C2, 72)]
        first, after = [0, 1], [0, 1]
        nb = amd.amsim_gemm_phased_workspace_size(probs, first, after, lut)
        amd.amsim_gemm_phased(probs, first, after, lut, ws=amd.workspace(nb))
        torch.cuda.synchronize()
        assert amd.amsim_last_path() & amd.AMSIM_PATH_PHASED, amd.amsim_last_path()
        outs.append((C1.cpu().numpy(), C2.cpu().numpy()))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    c1, c2 = outs[0]
    rows = np.array([0, 9, 33, m - 1])
    ref, sa = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert_close(c1[rows], ref, sa, "phased tail C1")
    ref2, sa2 = orc.gemm("mitchell", 7, c1, W2, rows=rows)
    assert_close(c2[rows], ref2, sa2, "phased C2 (reads C1)")


@pytest.mark.parametrize("n", [300, 360])
@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_tail_tiles_with_closed_forms(amd, orc, luts, kind, n):
    """Closed-form products (computed in registers) in both tail layouts, cut
    by stream-K: bit-identical to the table's products, within the oracle's
    tolerance."""
    import torch
    rng = np.random.default_rng(26 + n)
    m, k = 64, 12000
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    dA, dB = to_dev(A), to_dev(B)
    outs = []
    cf = amd.Lut.build(kind, 7).set_closed_form(True)
    try:
        for lut in (luts(kind, 7), cf):
            nb = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut)
            C = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
            amd.amsim_gemm("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, C, n, lut, ws=amd.workspace(nb))
            torch.cuda.synchronize()
            taken = amd.amsim_last_path()
            assert taken & amd.AMSIM_PATH_RAW_TILES and taken & amd.AMSIM_PATH_STREAMK, taken
            outs.append(C.cpu().numpy())
        assert taken & amd.AMSIM_PATH_CLOSED_FORM, taken
    finally:
        cf.close()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    rows = np.array([0, 31, m - 1])
    ref, sa = orc.gemm(kind, 7, A, B, rows=rows)
    assert_close(outs[1][rows], ref, sa, f"closed form tail {kind} n={n}")


@pytest.mark.parametrize("ldc_pad", [0, 1])
@pytest.mark.parametrize("ta,tb", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("m,n", [(64, 300), (300, 64), (64, 360)])
def test_tail_tiles_transposes_alpha_beta(amd, orc, luts, m, n, ta, tb, ldc_pad):
    """Tail tiles through every store path: C along L (m = 64: U is A's rows),
    C along U (n = 64: the planner swaps the operands, so L is A's rows and
    stores run down C's columns), and an odd leading dimension of C (scalar
    stores); alpha and beta both applied."""
    import torch
    k = 500
    rng = np.random.default_rng(1000 * m + n + 2 * ta + tb + 7 * ldc_pad)
    A = rnd(rng, (k, m) if ta else (m, k))
    B = rnd(rng, (n, k) if tb else (k, n))
    ldc = n + ldc_pad
    C0 = rnd(rng, (m, ldc))
    lut = luts("mitchell", 7)
    C = to_dev(C0)
    alpha, beta = 0.5, -1.25
    amd.amsim_gemm("T" if ta else "N", "T" if tb else "N", m, n, k, alpha, to_dev(A), A.shape[1], to_dev(B),
                   B.shape[1], beta, C, ldc, lut)
    torch.cuda.synchronize()
    assert amd.amsim_last_path() & amd.AMSIM_PATH_RAW_TILES, amd.amsim_last_path()
    got = C.cpu().numpy()
    ref, sa = orc.gemm("mitchell", 7, A, B, transA=ta, transB=tb, alpha=alpha, beta=beta, C0=C0[:, :n].copy())
    scale = abs(alpha) * sa + abs(beta) * np.abs(C0[:, :n].astype(np.float64)) / REL * 2.0 ** -23
    assert_close(got[:, :n], ref, scale + 1e-30, f"tail {m}x{n} {ta}{tb} ldc+{ldc_pad}")
    if ldc_pad:
        assert np.array_equal(got[:, n:], C0[:, n:])      # the padding column is untouched


@pytest.mark.parametrize("n", [300, 360])
@pytest.mark.parametrize("kind,M", [("mitchell", 8), ("mitchell", 9), ("exact", 7), ("exact", 4)])
def test_tail_tiles_other_tables(amd, orc, luts, kind, M, n):
    """Tail layouts with 16-bit tables in shared memory (M = 8, the exact kind
    at M = 7) and with the table read from global memory (M = 9: offsets and
    scales in two arrays), cut by stream-K: within the oracle's tolerance."""
    import torch
    rng = np.random.default_rng(40 + M + n)
    m, k = 64, 9000
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    lut = luts(kind, M)
    nb = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut)
    C = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    amd.amsim_gemm("N", "N", m, n, k, 1.0, to_dev(A), k, to_dev(B), n, 0.0, C, n, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    taken = amd.amsim_last_path()
    assert taken & amd.AMSIM_PATH_RAW_TILES and taken & amd.AMSIM_PATH_STREAMK, taken
    rows = np.array([0, 17, m - 1])
    ref, sa = orc.gemm(kind, M, A, B, rows=rows)
    assert_close(C.cpu().numpy()[rows], ref, sa, f"tail {kind} M={M} n={n}")
