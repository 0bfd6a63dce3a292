"""Arbitrary (here asymmetric) LUTs built from a user multiplier model through
Algorithm 1 (ApproxTrain Sec. V-A: the designer supplies approx_mul in C/C++;
LUTs are loaded at run time).  An asymmetric table makes the operand order
visible: the first operand's mantissa indexes the rows.  GEMMs whose operand
roles are swapped inside the kernel (the transposed table), batched GEMMs and a
grouped launch mixing both orientations are checked against a float64
reference that reads the same table (normal, finite operands only)."""
import numpy as np
import pytest

from gpu_helpers import assert_close, to_dev

pytestmark = pytest.mark.gpu

M = 5


def model(a, b):
    """Exact product of a and of b with its lowest kept mantissa bit cleared."""
    bb = np.float32(b).view(np.uint32) & np.uint32(~(1 << (23 - M)) & 0xFFFFFFFF)
    return float(np.float32(a) * bb.view(np.float32))


@pytest.fixture(scope="module")
def asym(amd):
    entries = amd.amsim_lut_generate_from_fn(model, M)
    t = entries.reshape(1 << M, 1 << M)
    assert not np.array_equal(t, t.T)
    lut = amd.Lut.from_entries(entries, M)
    yield entries, lut
    lut.close()


def products(entries, A, B):
    """AMSim products of normal operands from the table: [m, n, k] float64."""
    a = A.view(np.uint32).astype(np.int64)
    b = B.view(np.uint32).astype(np.int64)
    qa = (a & 0x7FFFFF) >> (23 - M)
    qb = (b & 0x7FFFFF) >> (23 - M)
    ea = (a >> 23) & 0xFF
    eb = (b >> 23) & 0xFF
    sa = a >> 31
    sb = b >> 31
    e = entries.astype(np.int64)[(qa[:, :, None] << M) | qb[None, :, :]]   # [m, k, n]
    carry = e >> 23
    mant = 1.0 + (e & 0x7FFFFF) / 2.0 ** 23
    v = np.ldexp(mant, (ea[:, :, None] + eb[None, :, :] - 254 + carry).astype(np.int32))
    sign = np.where((sa[:, :, None] ^ sb[None, :, :]) == 1, -1.0, 1.0)
    return np.transpose(sign * v, (0, 2, 1))


def reference(entries, A, B):
    p = products(entries, A, B)
    return p.sum(axis=2), np.abs(p).sum(axis=2)


def normal_operands(rng, shape):
    return (rng.standard_normal(shape) + np.where(rng.random(shape) < 0.5, 1.5, -1.5)).astype(np.float32)


@pytest.mark.parametrize("shape", [(70, 300, 40), (300, 7, 33), (5, 600, 17), (128, 256, 64)])
def test_asymmetric_gemm_both_orientations(amd, asym, shape):
    import torch
    entries, lut = asym
    m, n, k = shape
    rng = np.random.default_rng(sum(shape))
    A, B = normal_operands(rng, (m, k)), normal_operands(rng, (k, n))
    C = amd.gemm(to_dev(A), to_dev(B), lut)
    torch.cuda.synchronize()
    ref, sa = reference(entries, A, B)
    assert_close(C.cpu().numpy(), ref, sa, f"asym {shape}")
    # the swapped product differs (rows index the first operand)
    C2 = amd.gemm(to_dev(B.T.copy()), to_dev(A.T.copy()), lut).cpu().numpy()
    ref2, sa2 = reference(entries, B.T.copy(), A.T.copy())
    assert_close(C2, ref2, sa2, f"asym swapped {shape}")
    assert not np.allclose(C2.T, ref, rtol=1e-7, atol=0)


def test_asymmetric_grouped_mixed_orientations(amd, asym):
    """One grouped call holding problems of both orientations (the library
    splits it into one launch per orientation)."""
    import torch
    entries, lut = asym
    rng = np.random.default_rng(5)
    specs = [(200, 300, 50), (300, 9, 70), (8, 400, 30)]
    probs, outs, hosts = [], [], []
    for m, n, k in specs:
        A, B = normal_operands(rng, (m, k)), normal_operands(rng, (k, n))
        dA, dB = to_dev(A), to_dev(B)
        C = torch.zeros((m, n), dtype=torch.float32, device="cuda")
        probs.append(amd.GemmProblem.make("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, C, n))
        outs.append((C, dA, dB))
        hosts.append((A, B))
    nb = amd.amsim_gemm_grouped_workspace_size(probs, lut)
    amd.amsim_gemm_grouped(probs, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    for (A, B), (C, _, _) in zip(hosts, outs):
        ref, sa = reference(entries, A, B)
        assert_close(C.cpu().numpy(), ref, sa, f"grouped asym {A.shape}x{B.shape}")


def test_lut_info_and_roundtrip(amd, asym):
    entries, lut = asym
    assert np.array_equal(lut.entries(), entries)
    info = lut.info()
    assert info["M"] == M
