"""LUT-GEMM on the GPU against the CPU oracle (ApproxTrain Sec. VI-D GEMM
kernel, Sec. VI-C AMDENSE): all transpose combinations, ragged shapes that span
several CTA tiles, alpha/beta, split-K with and without scratch, special
operands, batched strided GEMMs, guard canaries and run-to-run determinism.
Tolerance: |gpu - oracle| <= 1e-5 * sum_k |AMSim product| per element."""
import numpy as np
import pytest

from gpu_helpers import REL, assert_close, guarded, guards_intact, to_dev

pytestmark = pytest.mark.gpu


def gpu_gemm(amd, lut, A, B, ta, tb, alpha=1.0, beta=0.0, C0=None, ws="auto", batch_strides=None):
    import torch
    m = A.shape[1] if ta else A.shape[0]
    k = A.shape[0] if ta else A.shape[1]
    n = B.shape[0] if tb else B.shape[1]
    dA, dB = to_dev(A), to_dev(B)
    buf, C = guarded((m, n), C0 if C0 is not None else np.zeros((m, n), np.float32))
    tA, tB = ("T" if ta else "N"), ("T" if tb else "N")
    if ws == "auto":
        nbytes = amd.amsim_gemm_workspace_size(tA, tB, m, n, k, 1, lut)
        wsb = amd.workspace(nbytes)
    else:
        wsb = ws
    amd.amsim_gemm(tA, tB, m, n, k, alpha, dA, max(1, A.shape[1]), dB, max(1, B.shape[1]), beta, C, max(1, n),
                   lut, ws=wsb)
    torch.cuda.synchronize()
    assert guards_intact(buf), "write outside C"
    return C.cpu().numpy()


def check(orc, kind, M, A, B, ta, tb, got, alpha=1.0, beta=0.0, C0=None, what=""):
    ref, sa = orc.gemm(kind, M, A, B, transA=ta, transB=tb, alpha=alpha, beta=beta, C0=C0)
    scale = abs(alpha) * sa
    if C0 is not None and beta != 0.0:
        scale = scale + abs(beta) * np.abs(C0.astype(np.float64)) / REL * 2.0 ** -23
    assert_close(got, ref, scale + 1e-30, what)


def rnd(rng, shape, kind="normal"):
    if kind == "normal":
        return rng.standard_normal(shape).astype(np.float32)
    return rng.uniform(-1, 1, size=shape).astype(np.float32)


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_small_gemm_workload(amd, orc, luts, kind):
    """64x128 by 128x64, U[-1,1], seed 0 (the small GEMM workload)."""
    from approximate_multiplier_dnn_gb300 import workloads as wl
    d = wl.gemm_small()
    got = gpu_gemm(amd, luts(kind, 7), d["A"], d["B"], False, False)
    check(orc, kind, 7, d["A"], d["B"], False, False, got, what=f"gemm64 {kind}")


SHAPES = [(1, 1, 1), (3, 17, 31), (33, 65, 129), (100, 300, 50), (257, 10, 500), (10, 257, 77),
          (130, 520, 40), (64, 256, 16), (65, 257, 17)]


@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
@pytest.mark.parametrize("shape", SHAPES)
def test_shapes_and_transposes(amd, orc, luts, shape, ta, tb):
    m, n, k = shape
    rng = np.random.default_rng(m * 10007 + n * 101 + k + 2 * ta + tb)
    A = rnd(rng, (k, m) if ta else (m, k))
    B = rnd(rng, (n, k) if tb else (k, n))
    got = gpu_gemm(amd, luts("mitchell", 7), A, B, ta, tb)
    check(orc, "mitchell", 7, A, B, ta, tb, got, what=f"{shape} {ta}{tb}")


@pytest.mark.parametrize("M", [4, 7, 8, 11])
@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_widths_and_residency(amd, orc, luts, kind, M):
    """8/16/32-bit narrowed tables; shared-memory and global-memory residency."""
    rng = np.random.default_rng(M)
    A = rnd(rng, (70, 90), "uniform")
    B = rnd(rng, (90, 300), "uniform")
    got = gpu_gemm(amd, luts(kind, M), A, B, False, False)
    check(orc, kind, M, A, B, False, False, got, what=f"{kind} M={M}")


def test_alpha_beta(amd, orc, luts):
    rng = np.random.default_rng(5)
    A, B = rnd(rng, (50, 70)), rnd(rng, (70, 90))
    C0 = rnd(rng, (50, 90))
    got = gpu_gemm(amd, luts("mitchell", 7), A, B, False, False, alpha=0.125, beta=-1.5, C0=C0)
    check(orc, "mitchell", 7, A, B, False, False, got, alpha=0.125, beta=-1.5, C0=C0, what="alpha/beta")


def test_k_zero_gives_beta_c(amd, luts):
    rng = np.random.default_rng(6)
    C0 = rnd(rng, (5, 7))
    got = gpu_gemm(amd, luts("mitchell", 7), np.zeros((5, 0), np.float32), np.zeros((0, 7), np.float32),
                   False, False, alpha=1.0, beta=2.0, C0=C0)
    assert np.array_equal(got, (2.0 * C0).astype(np.float32))


@pytest.mark.parametrize("with_ws", [True, False])
def test_split_k(amd, orc, luts, with_ws):
    """Few output tiles and a long reduction: split across CTAs when scratch is
    given (fixed-order reduction), a single pass otherwise."""
    rng = np.random.default_rng(7)
    A, B = rnd(rng, (60, 4000)), rnd(rng, (4000, 70))
    lut = luts("mitchell", 7)
    assert amd.amsim_gemm_workspace_size("N", "N", 60, 70, 4000, 1, lut) > 0
    got = gpu_gemm(amd, lut, A, B, False, False, ws="auto" if with_ws else None)
    check(orc, "mitchell", 7, A, B, False, False, got, what=f"split-k ws={with_ws}")


def test_special_operands(amd, orc, luts):
    """Zeros, denormals, infinities, NaNs and huge values (|x| >= 2^64, the
    slower exact-overflow path) inside the operands."""
    from approximate_multiplier_dnn_gb300 import workloads as wl
    rng = np.random.default_rng(8)
    a, b = wl.special_values_mix(40 * 96 + 96 * 50, seed=9)
    A = a[:40 * 96].reshape(40, 96).copy()
    B = b[40 * 96:40 * 96 + 96 * 50].reshape(96, 50).copy()
    # keep most rows/columns finite so most outputs are finite
    A[:, :] = np.where(rng.random(A.shape) < 0.9, rng.standard_normal(A.shape), A).astype(np.float32)
    B[:, :] = np.where(rng.random(B.shape) < 0.9, rng.standard_normal(B.shape), B).astype(np.float32)
    for kind in ("mitchell", "exact"):
        got = gpu_gemm(amd, luts(kind, 7), A, B, False, False)
        check(orc, kind, 7, A, B, False, False, got, what=f"specials {kind}")


def test_huge_values_overflow_to_inf(amd, orc, luts):
    """Products whose exponent reaches 255 through the LUT carry give infinity."""
    A = np.full((4, 8), np.float32(1.5 * 2.0 ** 127))
    B = np.full((8, 4), np.float32(1.5))
    got = gpu_gemm(amd, luts("mitchell", 7), A, B, False, False)
    ref, _ = orc.gemm("mitchell", 7, A, B)
    assert np.all(np.isinf(ref)) and np.array_equal(got, ref)


def test_batched_strided_attention_like(amd, orc, luts):
    import torch
    rng = np.random.default_rng(10)
    batch, s, d = 3, 70, 64
    Q = rnd(rng, (batch, s, d))
    K = rnd(rng, (batch, s, d))
    lut = luts("mitchell", 7)
    dQ, dK = to_dev(Q), to_dev(K)
    buf, S = guarded((batch, s, s))
    nb = amd.amsim_gemm_workspace_size("N", "T", s, s, d, batch, lut)
    amd.amsim_gemm_strided_batched("N", "T", s, s, d, 0.125, dQ, d, s * d, dK, d, s * d, 0.0, S, s, s * s, batch,
                                   lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    assert guards_intact(buf)
    got = S.cpu().numpy()
    for b in range(batch):
        ref, sa = orc.gemm("mitchell", 7, Q[b], K[b], transB=True, alpha=0.125)
        assert_close(got[b], ref, 0.125 * sa, f"batch {b}")


def test_deterministic(amd, luts):
    rng = np.random.default_rng(11)
    A, B = rnd(rng, (300, 500)), rnd(rng, (500, 200))
    lut = luts("mitchell", 7)
    g1 = gpu_gemm(amd, lut, A, B, False, False)
    g2 = gpu_gemm(amd, lut, A, B, False, False)
    assert np.array_equal(g1.view(np.uint32), g2.view(np.uint32))


def test_argument_errors(amd, luts):
    import torch
    lut = luts("mitchell", 7)
    x = torch.zeros(64, device="cuda")
    with pytest.raises(amd.AmsimError) as e:
        amd.amsim_gemm("N", "N", 4, 4, 4, 1.0, x, 3, x, 4, 0.0, x, 4, lut)    # lda < k
    assert e.value.status == amd.AMSIM_EINVAL
    with pytest.raises(amd.AmsimError):
        amd.amsim_gemm("X", "N", 4, 4, 4, 1.0, x, 4, x, 4, 0.0, x, 4, lut)
    with pytest.raises(amd.AmsimError):
        amd.amsim_gemm("N", "N", -1, 4, 4, 1.0, x, 4, x, 4, 0.0, x, 4, lut)
    with pytest.raises(amd.AmsimError):
        amd.amsim_gemm("N", "N", 4, 4, 4, 1.0, None, 4, x, 4, 0.0, x, 4, lut)


def test_grouped_matches_oracle_and_single_calls(amd, orc, luts):
    """Several GEMMs of different shapes, transposes and batch in one grouped
    launch (stream-K across problems), each checked against the oracle."""
    import torch
    lut = luts("mitchell", 7)
    rng = np.random.default_rng(20)
    specs = [(256, 1000, 300, False, False, 1), (256, 784, 100, False, True, 1), (78, 100, 256, True, False, 1),
             (5, 7, 9, False, False, 3), (33, 17, 1000, False, True, 2), (1, 1, 1, False, False, 1)]
    host, probs, outs = [], [], []
    for (m, n, k, ta, tb, batch) in specs:
        A = rnd(rng, (batch,) + ((k, m) if ta else (m, k)))
        B = rnd(rng, (batch,) + ((n, k) if tb else (k, n)))
        dA, dB = to_dev(A), to_dev(B)
        C = torch.zeros((batch, m, n), dtype=torch.float32, device="cuda")
        probs.append(amd.GemmProblem.make("T" if ta else "N", "T" if tb else "N", m, n, k, 1.0, dA, A.shape[2], dB,
                                          B.shape[2], 0.0, C, n, A[0].size, B[0].size, m * n, batch))
        host.append((A, B, ta, tb))
        outs.append((C, dA, dB))
    nb = amd.amsim_gemm_grouped_workspace_size(probs, lut)
    amd.amsim_gemm_grouped(probs, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    for (A, B, ta, tb), (C, _, _) in zip(host, outs):
        got = C.cpu().numpy()
        for b in range(A.shape[0]):
            ref, sa = orc.gemm("mitchell", 7, A[b], B[b], transA=ta, transB=tb)
            assert_close(got[b], ref, sa, f"grouped {A.shape}x{B.shape}")
    # the same group without scratch (data-parallel tiles) agrees within tolerance
    outs2 = []
    probs2 = []
    for p, (C, dA, dB) in zip(probs, outs):
        C2 = torch.zeros_like(C)
        q = amd.GemmProblem.make(p.transA.decode(), p.transB.decode(), p.m, p.n, p.k, 1.0, dA, p.lda, dB, p.ldb, 0.0,
                                 C2, p.ldc, p.strideA, p.strideB, p.strideC, p.batch)
        probs2.append(q)
        outs2.append(C2)
    amd.amsim_gemm_grouped(probs2, lut)
    torch.cuda.synchronize()
    for (A, B, ta, tb), C2 in zip(host, outs2):
        got = C2.cpu().numpy()
        for b in range(A.shape[0]):
            ref, sa = orc.gemm("mitchell", 7, A[b], B[b], transA=ta, transB=tb)
            assert_close(got[b], ref, sa, "grouped without scratch")


@pytest.mark.parametrize("shape", [(300, 500, 2000), (64, 256, 4096), (700, 90, 333), (2, 3, 5000)])
def test_stream_k_shapes(amd, orc, luts, shape):
    """Shapes whose tiles leave SMs idle run stream-K (partial tiles added by
    the fixup kernel in CTA order): parity and bit-identical repeats."""
    m, n, k = shape
    rng = np.random.default_rng(sum(shape))
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    lut = luts("mitchell", 7)
    assert amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut) > 0
    g1 = gpu_gemm(amd, lut, A, B, False, False)
    g2 = gpu_gemm(amd, lut, A, B, False, False)
    assert np.array_equal(g1.view(np.uint32), g2.view(np.uint32))
    rows = np.unique(np.random.default_rng(1).integers(0, m, size=min(m, 40)))
    ref, sa = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert_close(g1[rows], ref, sa, f"stream-k {shape}")


def _path_ws(amd, lut, path, tA, tB, m, n, k, batch=1):
    """Scratch selecting one kernel path: 'planes' (the full size: operands
    predecoded once into planes, copied by TMA), 'in_kernel' (one byte short:
    operands decoded inside the GEMM, stream-K kept) or 'none'."""
    full = amd.amsim_gemm_workspace_size(tA, tB, m, n, k, batch, lut)
    if path == "planes":
        return amd.workspace(full)
    if path == "in_kernel":
        return amd.workspace(max(full - 1, 1))
    return None


PATH_SHAPES = [(33, 65, 129), (257, 10, 500), (300, 500, 2000), (65, 257, 17), (2, 3, 5000), (513, 600, 999)]

# elements of unaligned operands the raw-tile kernel loads plainly (above it a
# launch uses planes or the in-kernel decode)
DIRECT_ELEMS = 256 * 1024


@pytest.mark.parametrize("path", ["planes", "in_kernel", "none"])
@pytest.mark.parametrize("shape", PATH_SHAPES)
def test_each_kernel_path(amd, orc, luts, shape, path):
    m, n, k = shape
    rng = np.random.default_rng(31 * m + 7 * n + k)
    A, B = rnd(rng, (m, k)), rnd(rng, (n, k))
    lut = luts("mitchell", 7)
    got = gpu_gemm(amd, lut, A, B, False, True, ws=_path_ws(amd, lut, path, "N", "T", m, n, k))
    taken = amd.amsim_last_path()
    # operands with copy-engine strides (k a multiple of 4 here) are copied in
    # place and decoded in shared memory on any scratch, and so are small
    # unaligned ones (loaded plainly); larger unaligned ones need planes
    raw = k % 4 == 0 or (m + n) * k <= DIRECT_ELEMS
    if raw:
        assert taken & amd.AMSIM_PATH_RAW_TILES, taken
    elif path == "planes":
        assert taken & amd.AMSIM_PATH_PLANES, taken
    else:
        assert not taken & (amd.AMSIM_PATH_PLANES | amd.AMSIM_PATH_RAW_TILES), taken
        assert taken & (amd.AMSIM_PATH_INKERNEL_DECODE | amd.AMSIM_PATH_SINGLE_ROLE), taken
    if path == "none":
        assert not taken & amd.AMSIM_PATH_STREAMK, taken
    check(orc, "mitchell", 7, A, B, False, True, got, what=f"{shape} path={path}")


@pytest.mark.parametrize("path", ["planes", "in_kernel", "none"])
def test_special_operands_each_path(amd, orc, luts, path):
    """Zeros, denormals, infinities, NaNs and |x| >= 2^64 through every path;
    the predecoded path flags the whole problem for the rounding slow path."""
    from approximate_multiplier_dnn_gb300 import workloads as wl
    rng = np.random.default_rng(12)
    a, b = wl.special_values_mix(70 * 130 + 130 * 90, seed=13)
    A = a[:70 * 130].reshape(70, 130).copy()
    B = b[70 * 130:70 * 130 + 130 * 90].reshape(130, 90).copy()
    A[:, :] = np.where(rng.random(A.shape) < 0.93, rng.standard_normal(A.shape), A).astype(np.float32)
    B[:, :] = np.where(rng.random(B.shape) < 0.93, rng.standard_normal(B.shape), B).astype(np.float32)
    for kind in ("mitchell", "exact"):
        lut = luts(kind, 7)
        got = gpu_gemm(amd, lut, A, B, False, False, ws=_path_ws(amd, lut, path, "N", "N", 70, 90, 130))
        check(orc, kind, 7, A, B, False, False, got, what=f"specials {kind} path={path}")


@pytest.mark.parametrize("kind,M,small", [("mitchell", 7, False), ("exact", 7, False), ("mitchell", 8, False),
                                          ("mitchell", 9, False), ("mitchell", 7, True)])
def test_special_operands_on_planes(amd, orc, luts, kind, M, small):
    """Zeros, denormals, infinities, NaNs and |x| >= 2^64 through the
    predecoded planes: packed operand words (M = 7 wide tiles, M = 8 narrow
    tiles) and two planes (M = 9, table in global memory).  Operands too large
    and unaligned for plain loads (k = 1301) force the planes.  small: nonzero
    magnitudes below 2^-63 instead of the huge ones (the zero test of
    Algorithm 2, no folded form)."""
    from approximate_multiplier_dnn_gb300 import workloads as wl
    rng = np.random.default_rng(40 + M)
    m, n, k = 300, 260, 1301
    a, b = wl.special_values_mix(m * k + k * n, seed=41)
    A = a[:m * k].reshape(m, k).copy()
    B = b[m * k:m * k + k * n].reshape(k, n).copy()
    A[:, :] = np.where(rng.random(A.shape) < 0.97, rng.standard_normal(A.shape), A).astype(np.float32)
    B[:, :] = np.where(rng.random(B.shape) < 0.97, rng.standard_normal(B.shape), B).astype(np.float32)
    if small:
        for X in (A, B):
            big = ~np.isfinite(X) | (np.abs(X) >= 2.0 ** 64)
            X[big] = np.float32(3e-20)
    lut = luts(kind, M)
    got = gpu_gemm(amd, lut, A, B, False, False)
    bits = amd.amsim_last_path()
    assert bits & amd.AMSIM_PATH_PLANES, bits
    check(orc, kind, M, A, B, False, False, got, what=f"planes specials {kind} M={M} small={small}")


@pytest.mark.parametrize("k", [150, 152])
@pytest.mark.parametrize("path", ["planes", "none"])
def test_batched_broadcast_operand(amd, orc, luts, path, k):
    """strideB = 0: one B serves every batch (one plane, one copied tensor for
    k = 152, or plain loads of one tensor for k = 150, for all batches)."""
    import torch
    rng = np.random.default_rng(14)
    batch, m, n = 5, 70, 90
    A = rnd(rng, (batch, m, k))
    B = rnd(rng, (k, n))
    lut = luts("mitchell", 7)
    buf, C = guarded((batch, m, n))
    full = amd.amsim_gemm_workspace_size("N", "N", m, n, k, batch, lut)
    ws = amd.workspace(full) if path == "planes" else None
    amd.amsim_gemm_strided_batched("N", "N", m, n, k, 1.0, to_dev(A), k, m * k, to_dev(B), n, 0, 0.0, C, n, m * n,
                                   batch, lut, ws=ws)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    got = C.cpu().numpy()
    for b in range(batch):
        ref, sa = orc.gemm("mitchell", 7, A[b], B)
        assert_close(got[b], ref, sa, f"batch {b} path={path}")


def test_paths_bit_identical_without_stream_k(amd, luts):
    """Shapes that fill whole waves run data-parallel; every output element is
    then summed in the same order on every path and tile shape, so the outputs
    are bit-identical: 64-row tiles with and without scratch at m = 64 x SMs,
    and the predecoded kernel's 128 x 256 tiles (one wave: 38 x 4 tiles on 152
    SMs) against the kernel without scratch."""
    import torch
    rng = np.random.default_rng(15)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    lut = luts("mitchell", 7)
    k = 100
    cases = [(64 * sms, 200, ("in_kernel", "none"), False)]
    if sms % 4 == 0:
        # n in (768, 1024]: four lane tiles; m / 128 * 4 = SMs; 0.0096 plane bytes per MAC takes the planes
        cases.append((128 * sms // 4, 1000, ("planes", "none"), False))
        # ReLU-like zeros in both operands: the folded form (zero uniform
        # operands through the table's zero row) on every path
        cases.append((128 * sms // 4, 1000, ("planes", "none"), True))
    for m, n, paths, zeros in cases:
        A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
        if zeros:
            A[A < 0] = 0.0
            B[B < -0.3] = -0.0
        outs, bits = [], []
        for p in paths:
            outs.append(gpu_gemm(amd, lut, A, B, False, False, ws=_path_ws(amd, lut, p, "N", "N", m, n, k)))
            bits.append(amd.amsim_last_path())
        assert not any(b & amd.AMSIM_PATH_STREAMK for b in bits), bits
        if paths[0] == "planes":
            assert bits[0] & amd.AMSIM_PATH_PLANES and bits[0] & amd.AMSIM_PATH_WIDE_TILES, bits
            assert not bits[1] & amd.AMSIM_PATH_WIDE_TILES, bits
        for o in outs[1:]:
            assert np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)), (m, n, paths)


@pytest.mark.parametrize("zeros", [False, True])
@pytest.mark.parametrize("kind,M,wide", [("mitchell", 7, True), ("exact", 7, True), ("mitchell", 8, False),
                                         ("mitchell", 9, True)])
def test_predecoded_tile_shape_by_table(amd, orc, luts, kind, M, wide, zeros):
    """The predecoded kernel takes the wide 128 x 256 tiles when their ring fits
    beside the table in shared memory (8- and 16-bit M = 7 tables) or when the
    table is read from global memory (M = 9), and the narrow tiles for the
    128 KB M = 8 table; 98 wide tiles on the SMs cut some tiles by stream-K.
    With ReLU-like zeros (and signed zeros, denormals) in both operands the
    uniform operand's zeros take the table's zero row."""
    rng = np.random.default_rng(16 + M)
    m = n = 1700
    k = 64
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    if zeros:
        A[A < 0.1] = 0.0
        B[B > 0.2] = -0.0
        A[::7, ::5] = np.float32(1e-40)
        B[::5, ::3] = np.float32(-3e-39)
    lut = luts(kind, M)
    got = gpu_gemm(amd, lut, A, B, False, False)
    bits = amd.amsim_last_path()
    assert bits & amd.AMSIM_PATH_PLANES, bits
    assert bool(bits & amd.AMSIM_PATH_WIDE_TILES) == wide, bits
    check(orc, kind, M, A, B, False, False, got, what=f"tile shape {kind} M={M}")


def test_workspace_counts_plane_bytes_per_element(amd, luts):
    """The scratch of a plane-path GEMM holds one 4-byte packed word per
    operand element when the table fits shared memory (M = 7) and an offset
    and a scale, 8 bytes, when it is read from global memory (M = 9); both
    use the wide tiles' stream-K slots, so the sizes differ by exactly the
    second plane: 4 x (m k + k n) bytes."""
    m = n = k = 4096
    w7 = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, luts("mitchell", 7))
    w9 = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, luts("mitchell", 9))
    assert w9 - w7 == 4 * (m * k + k * n), (w7, w9)
    assert w7 > 4 * (m * k + k * n), w7


def test_raw_or_planes_by_launch_size(amd, orc, luts):
    """Dense operands the copy engine can read take planes only for large
    launches whose elements many tiles reuse: a batched 512 x 512 x 64 GEMM
    (2^30 MACs, 0.031 plane bytes per MAC) takes planes, one MLP layer's
    256 x 1000 x 784 GEMM (0.039) raw tiles.  Both match the oracle (the large
    one on sampled batches)."""
    import torch
    rng = np.random.default_rng(23)
    lut = luts("mitchell", 7)
    batch, m, n, k = 64, 512, 512, 64
    A = rnd(rng, (batch, m, k))
    B = rnd(rng, (batch, n, k))
    nb = amd.amsim_gemm_workspace_size("N", "T", m, n, k, batch, lut)
    C = torch.empty((batch, m, n), device="cuda")
    amd.amsim_gemm_strided_batched("N", "T", m, n, k, 1.0, to_dev(A), k, m * k, to_dev(B), k, n * k, 0.0, C, n,
                                   m * n, batch, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    bits = amd.amsim_last_path()
    assert bits & amd.AMSIM_PATH_PLANES and not bits & amd.AMSIM_PATH_RAW_TILES, bits
    got = C.cpu().numpy()
    for b in (0, 37, 63):
        ref, sa = orc.gemm("mitchell", 7, A[b], B[b], transB=True)
        assert_close(got[b], ref, sa, f"batch {b}")
    m, n, k = 256, 1000, 784
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    got = gpu_gemm(amd, lut, A, B, False, False)
    bits = amd.amsim_last_path()
    assert bits & amd.AMSIM_PATH_RAW_TILES and not bits & amd.AMSIM_PATH_PLANES, bits
    check(orc, "mitchell", 7, A, B, False, False, got, what="mlp layer")


@pytest.mark.parametrize("zeros_in", ["A", "B", "both"])
def test_folded_scale_bit_identical_to_general_form(amd, orc, luts, zeros_in):
    """Stages whose uniform operands lie in [2^-63, 2^64) and whose lane
    operands do too or are zero fold the uniform scale into the rebuilt entry
    (raw-tile, plane and in-kernel-decode kernels, tables in shared memory);
    the closed form computes the same products in registers with the general
    order.  All add the same exact products in the same order, so outputs are
    bit-identical -- with ReLU-like zeros in either operand (zero uniform
    operands send their stages to the general form) and a few tiny ones (a
    product below the zero test: general form too)."""
    import torch
    rng = np.random.default_rng(16)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m, n, k = 64 * sms, 200, 100          # one 64 x 256 tile per SM: no stream-K on any path
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    if zeros_in in ("A", "both"):
        A[rng.random(A.shape) < 0.5] = 0.0
        A[0, 3] = np.float32(1e-25)
    if zeros_in in ("B", "both"):
        B[rng.random(B.shape) < 0.5] = 0.0
        B[7, 5] = np.float32(-3e-24)
    lut = luts("mitchell", 7)
    base = gpu_gemm(amd, lut, A, B, False, False)
    base_path = amd.amsim_last_path()
    assert base_path & (amd.AMSIM_PATH_RAW_TILES | amd.AMSIM_PATH_PLANES), base_path
    # the closed form on the same plan: no table, the general order
    cf = amd.Lut.build("mitchell", 7).set_closed_form(True)
    try:
        alu = gpu_gemm(amd, cf, A, B, False, False)
        assert amd.amsim_last_path() & amd.AMSIM_PATH_CLOSED_FORM
    finally:
        cf.close()
    assert np.array_equal(base.view(np.uint32), alu.view(np.uint32))
    # the same A with a leading dimension of k + 1 (not a multiple of 4 elements,
    # too large for plain loads): the in-kernel-decode kernel
    A1 = np.zeros((m, k + 1), np.float32)
    A1[:, :k] = A
    dA1, dB = to_dev(A1), to_dev(B)
    C = torch.empty((m, n), dtype=torch.float32, device="cuda")
    nb = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut)
    amd.amsim_gemm("N", "N", m, n, k, 1.0, dA1, k + 1, dB, n, 0.0, C, n, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    path = amd.amsim_last_path()
    assert path & (amd.AMSIM_PATH_INKERNEL_DECODE | amd.AMSIM_PATH_SINGLE_ROLE), path
    assert np.array_equal(base.view(np.uint32), C.cpu().numpy().view(np.uint32))
    rows = np.array([0, 7, m - 1])
    ref, sa = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert_close(base[rows], ref, sa, f"folded, zeros in {zeros_in}")


RAW_SHAPES = [(64, 256, 16), (300, 500, 2000), (130, 520, 40), (257, 10, 500), (5, 7, 4), (700, 90, 332)]
# (shape, transA, transB) whose leading dimensions are multiples of 4 elements
# (what selects this path): lda = m for a transposed A, else k; ldb = k for a
# transposed B, else n.
RAW_CASES = [(s, ta, tb) for s in RAW_SHAPES for ta in (False, True) for tb in (False, True)
             if (s[0] if ta else s[2]) % 4 == 0 and (s[2] if tb else s[1]) % 4 == 0]


@pytest.mark.parametrize("shape,ta,tb", RAW_CASES)
def test_raw_tile_path(amd, orc, luts, shape, ta, tb):
    """Operand tiles copied in place (rows or k innermost, so both the plain and
    the swizzled transposing decode run) and decoded in shared memory."""
    m, n, k = shape
    rng = np.random.default_rng(7 * m + 5 * n + k + 2 * ta + tb)
    A = rnd(rng, (k, m) if ta else (m, k))
    B = rnd(rng, (n, k) if tb else (k, n))
    lut = luts("mitchell", 7)
    got = gpu_gemm(amd, lut, A, B, ta, tb)
    assert amd.amsim_last_path() & amd.AMSIM_PATH_RAW_TILES, amd.amsim_last_path()
    check(orc, "mitchell", 7, A, B, ta, tb, got, what=f"raw {shape} {ta}{tb}")


def test_raw_tile_path_special_operands(amd, orc, luts):
    """Zeros, denormals, infinities, NaNs and |x| >= 2^64 through the in-place
    copies (the per-stage large-operand flag selects the rounding path)."""
    from approximate_multiplier_dnn_gb300 import workloads as wl
    rng = np.random.default_rng(16)
    a, b = wl.special_values_mix(72 * 128 + 128 * 96, seed=17)
    A = a[:72 * 128].reshape(72, 128).copy()
    B = b[72 * 128:72 * 128 + 128 * 96].reshape(128, 96).copy()
    A[:, :] = np.where(rng.random(A.shape) < 0.93, rng.standard_normal(A.shape), A).astype(np.float32)
    B[:, :] = np.where(rng.random(B.shape) < 0.93, rng.standard_normal(B.shape), B).astype(np.float32)
    for kind in ("mitchell", "exact"):
        got = gpu_gemm(amd, luts(kind, 7), A, B, False, False)
        assert amd.amsim_last_path() & amd.AMSIM_PATH_RAW_TILES
        check(orc, kind, 7, A, B, False, False, got, what=f"raw specials {kind}")


@pytest.mark.parametrize("ta", [False, True])
@pytest.mark.parametrize("tb", [False, True])
@pytest.mark.parametrize("shape", [(70, 90, 129), (64, 10, 500), (10, 256, 1000), (33, 7, 3)])
def test_unaligned_small_operands_load_plainly(amd, orc, luts, shape, ta, tb):
    """Small operands whose leading dimension is not a multiple of 4 elements
    (a 10-wide layer) are read by the raw-tile kernel with plain loads, alone
    or beside an operand copied in place, with no predecode launch."""
    m, n, k = shape
    rng = np.random.default_rng(19 * m + 3 * n + k + 2 * ta + tb)
    A = rnd(rng, (k, m) if ta else (m, k))
    B = rnd(rng, (n, k) if tb else (k, n))
    for kind in ("mitchell", "exact"):
        got = gpu_gemm(amd, luts(kind, 7), A, B, ta, tb)
        taken = amd.amsim_last_path()
        assert taken & amd.AMSIM_PATH_RAW_TILES and not taken & amd.AMSIM_PATH_PLANES, taken
        check(orc, kind, 7, A, B, ta, tb, got, what=f"plain loads {shape} {ta}{tb} {kind}")


def test_unaligned_special_operands_load_plainly(amd, orc, luts):
    """Zeros, denormals, infinities, NaNs and |x| >= 2^64 through the plain
    loads of the raw-tile kernel."""
    from approximate_multiplier_dnn_gb300 import workloads as wl
    rng = np.random.default_rng(20)
    a, b = wl.special_values_mix(70 * 130 + 130 * 90, seed=21)
    A = a[:70 * 130].reshape(70, 130).copy()
    B = b[70 * 130:70 * 130 + 130 * 90].reshape(130, 90).copy()
    A[:, :] = np.where(rng.random(A.shape) < 0.93, rng.standard_normal(A.shape), A).astype(np.float32)
    B[:, :] = np.where(rng.random(B.shape) < 0.93, rng.standard_normal(B.shape), B).astype(np.float32)
    for kind in ("mitchell", "exact"):
        got = gpu_gemm(amd, luts(kind, 7), A, B, False, False)
        assert amd.amsim_last_path() & amd.AMSIM_PATH_RAW_TILES
        check(orc, kind, 7, A, B, False, False, got, what=f"plain-load specials {kind}")


def test_misaligned_base_address_loads_plainly(amd, orc, luts):
    """An operand with a leading dimension that is a multiple of 4 elements
    but a base address off a 16-byte boundary is read with plain loads; the
    other operand is still copied in place."""
    import torch
    rng = np.random.default_rng(22)
    m, n, k = 96, 80, 200
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    lut = luts("mitchell", 7)
    store = torch.zeros(m * k + 1, dtype=torch.float32, device="cuda")
    dA = store[1:].view(m, k)
    dA.copy_(to_dev(A))
    buf, C = guarded((m, n))
    amd.amsim_gemm("N", "N", m, n, k, 1.0, dA, k, to_dev(B), n, 0.0, C, n, lut)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    assert amd.amsim_last_path() & amd.AMSIM_PATH_RAW_TILES, amd.amsim_last_path()
    check(orc, "mitchell", 7, A, B, False, False, C.cpu().numpy(), what="misaligned base")


def test_unaligned_large_operands_take_planes(amd, orc, luts):
    """Larger operands whose leading dimension is not a multiple of 4 elements
    cannot be copied in place: with scratch they go through planes instead."""
    rng = np.random.default_rng(18)
    A, B = rnd(rng, (600, 999)), rnd(rng, (999, 700))
    lut = luts("mitchell", 7)
    got = gpu_gemm(amd, lut, A, B, False, False)
    taken = amd.amsim_last_path()
    assert taken & amd.AMSIM_PATH_PLANES and not taken & amd.AMSIM_PATH_RAW_TILES, taken
    check(orc, "mitchell", 7, A, B, False, False, got, what="unaligned lda")
