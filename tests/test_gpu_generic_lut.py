"""User multiplier models on the GPU against the oracle (ApproxTrain Sec. V-A:
the designer supplies approx_mul in C/C++ and Algorithm 1 builds its table;
Sec. VI: tables are handed to the operator library at run time).

Tables come from amsim_lut_build_from_fn (one call) and from
amsim_lut_generate_from_fn + amsim_lut_build_from_entries; the oracle reads
the same entries through its own Algorithm 1 over the same Python model, so
the reference never comes from the library.  An asymmetric model makes the
operand order visible (the first operand's mantissa indexes the rows): GEMMs
whose operand roles the kernels swap (the transposed table), batched and
grouped calls, convolutions, and the elementwise product are each checked.
Operands carry zeros, denormals, infinities, NaN, products that overflow
through the table's carry and products that underflow, besides normal values.
"""
import numpy as np
import pytest

from gpu_helpers import assert_close, bits, to_dev

pytestmark = pytest.mark.gpu


def asym_model(M):
    """Exact product of a and of b with its lowest kept mantissa bit cleared."""
    clear = np.uint32(~(1 << (23 - M)) & 0xFFFFFFFF)

    def model(a, b):
        bb = (np.float32(b).view(np.uint32) & clear).view(np.float32)
        return float(np.float32(a) * bb)
    return model


def wide_model(a, b):
    """Exact product plus 2^-21: entries use their low mantissa bits, so the
    table cannot be narrowed (32-bit entries)."""
    return float(np.float32(np.float32(a) * np.float32(b)) + np.float32(2.0 ** -21))


MODELS = {
    "asym5": (5, asym_model(5)),
    "asym7": (7, asym_model(7)),
    "asym9": (9, asym_model(9)),     # table beyond shared memory: global/L2 path
    "wide6": (6, wide_model),
}


@pytest.fixture(scope="module", params=sorted(MODELS))
def user_lut(request, amd, orc):
    M, model = MODELS[request.param]
    ref = orc.lut_from_fn(model, M)                  # the oracle's own Algorithm 1
    lut = amd.Lut.from_fn(model, M)                  # one ABI call
    assert np.array_equal(lut.entries(), ref)
    yield request.param, M, ref, lut
    lut.close()


def test_two_call_build_matches_one_call(amd, orc):
    M = 5
    entries = amd.amsim_lut_generate_from_fn(asym_model(M), M)
    assert np.array_equal(entries, orc.lut_from_fn(asym_model(M), M))
    lut = amd.Lut.from_entries(entries, M)
    try:
        assert np.array_equal(lut.entries(), entries)
        assert lut.info()["M"] == M
    finally:
        lut.close()
    wide = amd.Lut.from_fn(wide_model, 6)
    try:
        assert wide.info()["width_bits"] == 32
    finally:
        wide.close()


def normal_operands(rng, shape):
    return (rng.standard_normal(shape) + np.where(rng.random(shape) < 0.5, 1.5, -1.5)).astype(np.float32)


HUGE = np.float32(1.96875 * 2.0 ** 127)     # with a 1.96875 partner: e0 = 254 and a carry -> Inf
TINY = np.float32(1.5 * 2.0 ** -126)        # with a 0.765625 partner: e0 = 0 -> zero


def sprinkle(rng, A, B, count=6):
    """Put special operands at a few places of A (m x k) and B (k x n)."""
    m, k = A.shape
    n = B.shape[1]
    specials = [0.0, -0.0, np.float32(3e-39), np.inf, -np.inf, np.nan]
    for i in range(count):
        A[rng.integers(m), rng.integers(k)] = specials[i % len(specials)]
        B[rng.integers(k), rng.integers(n)] = specials[(i + 3) % len(specials)]
    r, kk, c = rng.integers(m), rng.integers(k), rng.integers(n)
    A[r, kk], B[kk, c] = HUGE, np.float32(1.96875)          # overflow through the carry
    r, kk, c = rng.integers(m), rng.integers(k), rng.integers(n)
    A[r, kk], B[kk, c] = TINY, np.float32(0.765625)         # underflow to zero
    return A, B


@pytest.mark.parametrize("shape", [(70, 300, 40), (300, 7, 33), (5, 600, 17), (128, 256, 64), (257, 130, 300)])
def test_user_gemm_both_orientations(amd, orc, user_lut, shape):
    import torch
    name, M, table, lut = user_lut
    m, n, k = shape
    rng = np.random.default_rng(sum(shape) + M)
    A, B = sprinkle(rng, normal_operands(rng, (m, k)), normal_operands(rng, (k, n)))
    C = amd.gemm(to_dev(A), to_dev(B), lut)
    torch.cuda.synchronize()
    ref, sa = orc.gemm(table, M, A, B)
    assert_close(C.cpu().numpy(), ref, sa, f"{name} {shape}")
    # the swapped product (rows index the first operand): B^T A^T
    Bt, At = B.T.copy(), A.T.copy()
    C2 = amd.gemm(to_dev(Bt), to_dev(At), lut).cpu().numpy()
    ref2, sa2 = orc.gemm(table, M, Bt, At)
    assert_close(C2, ref2, sa2, f"{name} swapped {shape}")
    if name.startswith("asym"):
        fin = np.isfinite(ref) & np.isfinite(ref2.T)
        assert not np.allclose(ref2.T[fin], ref[fin], rtol=1e-7, atol=0)


@pytest.mark.parametrize("trans", ["NT", "TN", "TT"])
def test_user_gemm_transposes(amd, orc, user_lut, trans):
    import torch
    name, M, table, lut = user_lut
    m, n, k = 96, 80, 150
    rng = np.random.default_rng(7 + M)
    A, B = sprinkle(rng, normal_operands(rng, (m, k)), normal_operands(rng, (k, n)))
    tA, tB = trans[0] == "T", trans[1] == "T"
    Ad = A.T.copy() if tA else A
    Bd = B.T.copy() if tB else B
    C = amd.gemm(to_dev(Ad), to_dev(Bd), lut, transA=tA, transB=tB)
    torch.cuda.synchronize()
    ref, sa = orc.gemm(table, M, Ad, Bd, transA=tA, transB=tB)
    assert_close(C.cpu().numpy(), ref, sa, f"{name} {trans}")


def test_user_batched_and_grouped(amd, orc, user_lut):
    import torch
    name, M, table, lut = user_lut
    rng = np.random.default_rng(5)
    # batched (attention-like: S = Q K^T) with specials
    bt, m, n, k = 3, 64, 48, 40
    Q = normal_operands(rng, (bt, m, k))
    K = normal_operands(rng, (bt, n, k))
    Q[1, 3, 7], K[2, 5, 9] = np.nan, np.inf
    S = torch.empty((bt, m, n), dtype=torch.float32, device="cuda")
    nb = amd.amsim_gemm_workspace_size("N", "T", m, n, k, bt, lut)
    amd.amsim_gemm_strided_batched("N", "T", m, n, k, 0.125, to_dev(Q), k, m * k, to_dev(K), k, n * k, 0.0,
                                   S, n, m * n, bt, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    got = S.cpu().numpy()
    for b in range(bt):
        ref, sa = orc.gemm(table, M, Q[b], K[b], transB=True, alpha=0.125)
        assert_close(got[b], ref, 0.125 * sa, f"{name} batched {b}")
    # grouped: three problems in one call (both LUT orientations are handled by the library)
    specs = [(200, 300, 50), (300, 9, 70), (8, 400, 30)]
    probs, outs, hosts = [], [], []
    for m, n, k in specs:
        A, B = sprinkle(rng, normal_operands(rng, (m, k)), normal_operands(rng, (k, n)), count=2)
        dA, dB = to_dev(A), to_dev(B)
        C = torch.zeros((m, n), dtype=torch.float32, device="cuda")
        probs.append(amd.GemmProblem.make("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, C, n))
        outs.append((C, dA, dB))
        hosts.append((A, B))
    nb = amd.amsim_gemm_grouped_workspace_size(probs, lut)
    amd.amsim_gemm_grouped(probs, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    for (A, B), (C, _, _) in zip(hosts, outs):
        ref, sa = orc.gemm(table, M, A, B)
        assert_close(C.cpu().numpy(), ref, sa, f"{name} grouped {A.shape}x{B.shape}")


def test_user_elementwise_bit_exact(amd, orc, user_lut):
    import torch
    name, M, table, lut = user_lut
    rng = np.random.default_rng(3)
    n = 1 << 16
    u = rng.integers(0, 1 << 32, size=(2, n), dtype=np.uint64).astype(np.uint32)
    a, b = u.view(np.float32)
    a = a.copy()
    b = b.copy()
    a[:4], b[:4] = HUGE, np.float32(1.96875)
    a[4:8], b[4:8] = TINY, np.float32(0.765625)
    c = torch.empty(n, dtype=torch.float32, device="cuda")
    amd.amsim_mul(to_dev(a), to_dev(b), c, n, lut)
    torch.cuda.synchronize()
    assert np.array_equal(bits(c.cpu().numpy()), bits(orc.mul(table, M, a, b)))


GEOMS = [
    dict(N=2, H=9, W=10, C=16, K=24, R=3, S=3, stride=(1, 1), pad=(1, 1), dil=(1, 1)),
    dict(N=1, H=11, W=8, C=8, K=12, R=3, S=2, stride=(2, 1), pad=(1, 0), dil=(1, 2)),
]


@pytest.mark.parametrize("g", range(len(GEOMS)))
def test_user_conv_all_passes(amd, orc, user_lut, g):
    import torch
    name, M, table, lut = user_lut
    geo = GEOMS[g]
    N, H, W, C, K, R, S = (geo[x] for x in ("N", "H", "W", "C", "K", "R", "S"))
    desc = amd.ConvDesc.make(N, H, W, C, K, R, S, geo["stride"], geo["pad"], geo["dil"])
    P, Q = amd.amsim_conv2d_out_hw(desc)
    od = orc.conv_desc(N, H, W, C, K, R, S, geo["stride"], geo["pad"], geo["dil"])
    rng = np.random.default_rng(20 + g)
    x = normal_operands(rng, (N, H, W, C))
    w = normal_operands(rng, (R, S, C, K))
    dy = normal_operands(rng, (N, P, Q, K))
    x[0, 1, 2, 3], w[1, 0, 2, 5], dy[0, 0, 1, 2] = np.inf, 0.0, np.nan
    y = torch.empty((N, P, Q, K), dtype=torch.float32, device="cuda")
    dx = torch.empty((N, H, W, C), dtype=torch.float32, device="cuda")
    dw = torch.empty((R, S, C, K), dtype=torch.float32, device="cuda")
    for which, fn, a0, a1, out in ((0, amd.amsim_conv2d_fwd, x, w, y), (1, amd.amsim_conv2d_bwd_data, dy, w, dx),
                                   (2, amd.amsim_conv2d_bwd_filter, x, dy, dw)):
        nb = amd.amsim_conv2d_workspace_size(desc, which, lut)
        fn(desc, to_dev(a0), to_dev(a1), out, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    for got, fn, a0, a1 in ((y, orc.conv2d_fwd, x, w), (dx, orc.conv2d_bwd_data, dy, w),
                            (dw, orc.conv2d_bwd_filter, x, dy)):
        gv = got.cpu().numpy().reshape(-1)
        ref, sa = fn(table, M, od, a0, a1, np.arange(gv.size))
        assert_close(gv, ref, sa, f"{name} conv {g} {fn.__name__}")
