"""Pins of the oracle's user-multiplier path: Algorithm 1 over a caller's
approx_mul (ApproxTrain Sec. V-A: the designer supplies the C/C++ function and
a script builds the table) and Algorithm 2 over a stored table (Sec. V-B; the
tables are loaded at run time, Sec. VI).  Facts that do not come from the
oracle itself:

* a model that returns numpy's IEEE fp32 product of 1.p and 1.q (exact for
  M <= 11) yields the exact kind's table, and AMSim over that table equals the
  exact kind bit for bit on random, boundary and special operands; a model
  restating Mitchell's formula yields the Mitchell table;
* an asymmetric model's products, worked by hand
  (tests/golden/asym_model_values.txt);
* brute force at M = 2 over a random table: for normal operands whose
  exponent sum stays in range, AMSim equals sign * 2^(ea + eb + carry) *
  (1 + mantissa / 2^23) evaluated in float64, entry index (qa << M) | qb;
* Algorithm 1 rejects models whose carry is not 0 or 1, or whose product is
  negative;
* a GEMM over a table from the exact-product model equals the exact kind's
  GEMM, and over an asymmetric table equals a float64 sum of the brute-force
  products.
"""
import numpy as np
import pytest

from conftest import read_golden


def bits_f32(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


def f32_bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def exact_model(a, b):
    return float(np.float32(a) * np.float32(b))


def mitchell_model(a, b):
    x = float(np.float32(a)) - 1.0
    y = float(np.float32(b)) - 1.0
    return 1.0 + x + y if x + y < 1.0 else 2.0 * (x + y)


def asym_model(M):
    clear = np.uint32(~(1 << (23 - M)) & 0xFFFFFFFF)

    def model(a, b):
        bb = (np.float32(b).view(np.uint32) & clear).view(np.float32)
        return float(np.float32(a) * bb)
    return model


def _operands(rng, n):
    """Random fp32 patterns: any exponent, plus zeros, denormals, Inf, NaN."""
    u = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    kind = rng.integers(0, 16, size=n)
    u[kind == 0] &= np.uint32(0x80000000)                       # signed zero
    u[kind == 1] &= np.uint32(0x807FFFFF)                       # denormal
    u[kind == 2] = (u[kind == 2] & np.uint32(0x80000000)) | np.uint32(0x7F800000)   # Inf
    u[kind == 3] |= np.uint32(0x7F800001)                       # NaN
    e = rng.integers(100, 155, size=n).astype(np.uint32)        # mostly near 1.0
    mid = kind >= 8
    u[mid] = (u[mid] & np.uint32(0x807FFFFF)) | (e[mid] << np.uint32(23))
    return u


@pytest.mark.parametrize("M", [1, 2, 4, 7])
def test_exact_model_callback_gives_exact_kind(orc, M):
    t = orc.lut_from_fn(exact_model, M)
    assert np.array_equal(t, orc.lut("exact", M))
    rng = np.random.default_rng(40 + M)
    a, b = _operands(rng, 60_000), _operands(rng, 60_000)
    got = f32_bits(orc.mul(t, M, bits_f32(a), bits_f32(b)))
    want = f32_bits(orc.mul("exact", M, bits_f32(a), bits_f32(b)))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M", [3, 7, 10])
def test_mitchell_model_callback_gives_mitchell_kind(orc, M):
    assert np.array_equal(orc.lut_from_fn(mitchell_model, M), orc.lut("mitchell", M))


def test_asymmetric_model_hand_worked(orc):
    M = 5
    t = orc.lut_from_fn(asym_model(M), M)
    sq = t.reshape(1 << M, 1 << M)
    assert not np.array_equal(sq, sq.T)
    for a, b, want in read_golden("asym_model_values.txt"):
        got = orc.amsim_bits(t, M, int(a, 16), int(b, 16))
        assert got == int(want, 16), (a, b, hex(got), want)


def _random_table(rng, M):
    n = 1 << (2 * M)
    carry = rng.integers(0, 2, size=n).astype(np.uint32)
    mant = rng.integers(0, 1 << 23, size=n).astype(np.uint32)
    return (carry << np.uint32(23)) | mant


def _table_products(t, M, a, b):
    """sign * 2^(ea + eb - 254 + carry) * (1 + mant / 2^23) in float64 for normal
    operands, entry (qa << M) | qb."""
    a = a.astype(np.int64)
    b = b.astype(np.int64)
    qa = (a & 0x7FFFFF) >> (23 - M)
    qb = (b & 0x7FFFFF) >> (23 - M)
    e = t.astype(np.int64)[(qa << M) | qb]
    v = np.ldexp(1.0 + (e & 0x7FFFFF) / 2.0 ** 23, (((a >> 23) & 0xFF) + ((b >> 23) & 0xFF) - 254
                                                   + (e >> 23)).astype(np.int32))
    return np.where(((a >> 31) ^ (b >> 31)) == 1, -v, v)


def test_table_products_brute_force(orc):
    M = 2
    rng = np.random.default_rng(9)
    t = _random_table(rng, M)
    q = np.arange(1 << M, dtype=np.uint32)
    qa, qb = [x.reshape(-1) for x in np.meshgrid(q, q, indexing="ij")]
    reps = 500
    qa, qb = np.tile(qa, reps), np.tile(qb, reps)
    n = qa.size
    ea = rng.integers(64, 190, size=n).astype(np.uint32)      # e0 = ea + eb - 127 in [1, 251]
    eb = rng.integers(64, 190, size=n).astype(np.uint32)
    low = np.uint32((1 << (23 - M)) - 1)
    a = (rng.integers(0, 2, size=n).astype(np.uint32) << np.uint32(31)) | (ea << np.uint32(23)) | \
        (qa << np.uint32(23 - M)) | (rng.integers(0, 1 << 23, size=n).astype(np.uint32) & low)
    b = (rng.integers(0, 2, size=n).astype(np.uint32) << np.uint32(31)) | (eb << np.uint32(23)) | \
        (qb << np.uint32(23 - M)) | (rng.integers(0, 1 << 23, size=n).astype(np.uint32) & low)
    got = orc.mul(t, M, bits_f32(a), bits_f32(b)).astype(np.float64)
    assert np.array_equal(got, _table_products(t, M, a, b))


def test_algorithm1_rejects_models_outside_its_range(orc):
    with pytest.raises(ValueError):
        orc.lut_from_fn(lambda a, b: 0.5 * a * b, 3)        # product below 1: carry -1
    with pytest.raises(ValueError):
        orc.lut_from_fn(lambda a, b: 2.0 * a * b, 3)        # product of 1.q x 1.q reaches 4: carry 2
    with pytest.raises(ValueError):
        orc.lut_from_fn(lambda a, b: -a * b, 3)             # sign belongs to Algorithm 2
    assert orc.lut_from_fn(lambda a, b: a * b, 3).size == 64


@pytest.mark.parametrize("trans", [(False, False), (True, False), (False, True)])
def test_gemm_over_exact_model_table_equals_exact_kind(orc, trans):
    M = 6
    t = orc.lut_from_fn(exact_model, M)
    rng = np.random.default_rng(11)
    m, n, k = 9, 7, 33
    A = rng.standard_normal((k, m) if trans[0] else (m, k)).astype(np.float32)
    B = rng.standard_normal((n, k) if trans[1] else (k, n)).astype(np.float32)
    A.reshape(-1)[::13] = 0.0
    B.reshape(-1)[::97] = np.inf
    got, sa = orc.gemm(t, M, A, B, transA=trans[0], transB=trans[1])
    want, sa2 = orc.gemm("exact", M, A, B, transA=trans[0], transB=trans[1])
    assert np.array_equal(f32_bits(got), f32_bits(want))
    assert np.array_equal(sa, sa2, equal_nan=True)


def test_gemm_over_asymmetric_table_equals_float64_sum(orc):
    M = 5
    t = orc.lut_from_fn(asym_model(M), M)
    rng = np.random.default_rng(12)
    m, n, k = 6, 5, 40
    A = (rng.standard_normal((m, k)) + 2.0).astype(np.float32)
    B = (rng.standard_normal((k, n)) - 2.0).astype(np.float32)
    A[A == 0] = 1.0
    B[B == 0] = 1.0
    got, sa = orc.gemm(t, M, A, B)
    au = f32_bits(A)
    bu = f32_bits(B)
    prod = _table_products(t, M, au[:, :, None], bu[None, :, :])      # [m, k, n]
    assert np.array_equal(got.astype(np.float64), prod.sum(axis=1).astype(np.float32).astype(np.float64))
    assert np.allclose(sa, np.abs(prod).sum(axis=1), rtol=0, atol=0)
