"""Pins of the CPU oracle's scalar level (Algorithm 1 LUT generation and
Algorithm 2 AMSim of the ApproxTrain page, Sec. V-A and V-B) against facts that
do not come from the oracle itself:

* LUT byte sizes printed on the page (tests/golden/lut_sizes.txt);
* exact kind: carry/mantissa equal the integer normalisation of
  (2^M+p)(2^M+q), and AMSim equals numpy's IEEE fp32 product of the
  M-bit-truncated operands whenever the biased exponent sum is >= 1;
* Mitchell kind: hand-worked values (tests/golden/mitchell_hand_values.txt),
  Mitchell's log-domain construction (log2(1+x) ~ x, add, antilog), the error
  bound [-1/9, 0] with its minimum at x = y = 1/2, equality iff x = 0 or y = 0;
* special values and exponent boundaries worked by hand
  (tests/golden/special_values.txt).
"""
import numpy as np
import pytest

from conftest import read_golden

MASK32 = 0xFFFFFFFF


def f32_bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def bits_f32(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


# ------------------------------------------------------------------ LUT sizes
def test_lut_sizes_match_page(orc):
    for M, lo, hi in read_golden("lut_sizes.txt"):
        M, lo, hi = int(M), int(lo), int(hi)
        for kind in ("exact", "mitchell"):
            t = orc.lut(kind, M)
            assert t.dtype == np.uint32 and t.size == 1 << (2 * M)
            assert lo <= t.nbytes <= hi, (kind, M, t.nbytes)


def test_lut_rejects_bad_width(orc):
    with pytest.raises(ValueError):
        orc.lut("exact", 0)
    with pytest.raises(ValueError):
        orc.lut("mitchell", 12)


# ------------------------------------------------------------------ exact kind
@pytest.mark.parametrize("M", list(range(1, 12)))
def test_exact_lut_is_integer_normalisation(orc, M):
    """Carry and mantissa of (2^M+p)(2^M+q) / 2^(2M) by integer arithmetic."""
    t = orc.lut("exact", M).astype(np.int64)
    p = np.arange(1 << M, dtype=np.int64)
    N = ((1 << M) + p)[:, None] * ((1 << M) + p)[None, :]
    carry = (N >= (1 << (2 * M + 1))).astype(np.int64)
    lead = np.where(carry == 1, 1 << (2 * M + 1), 1 << (2 * M))
    shift = 23 - 2 * M - carry
    mant = (N - lead) << shift
    expect = (carry << 23) | mant
    assert np.array_equal(t, expect.reshape(-1))


def _truncate(bits, M):
    keep = np.uint32((0xFFFFFFFF << (23 - M)) & MASK32)
    return bits & keep


def _normal_operands(rng, n, M):
    """Random normal fp32 operands whose biased exponent sum e0 lies in [1, 300)."""
    ea = rng.integers(1, 255, size=n)
    lo = np.maximum(1, 128 - ea)
    hi = np.minimum(255, 427 - ea)
    eb = rng.integers(lo, hi)
    fa = rng.integers(0, 1 << 23, size=n)
    fb = rng.integers(0, 1 << 23, size=n)
    sa = rng.integers(0, 2, size=n)
    sb = rng.integers(0, 2, size=n)
    a = ((sa << 31) | (ea << 23) | fa).astype(np.uint32)
    b = ((sb << 31) | (eb << 23) | fb).astype(np.uint32)
    return a, b


@pytest.mark.parametrize("M", list(range(1, 8)))
def test_exact_equals_ieee_product_all_mantissa_pairs(orc, M):
    """Brute force over every mantissa pair, random signs/exponents with e0 >= 1."""
    rng = np.random.default_rng(100 + M)
    p = np.arange(1 << M, dtype=np.uint32)
    P, Q = np.meshgrid(p, p, indexing="ij")
    n = P.size
    a, b = _normal_operands(rng, n, M)
    a = (a & np.uint32(0xFF800000)) | (P.reshape(-1) << np.uint32(23 - M)) | (a & np.uint32((1 << (23 - M)) - 1))
    b = (b & np.uint32(0xFF800000)) | (Q.reshape(-1) << np.uint32(23 - M)) | (b & np.uint32((1 << (23 - M)) - 1))
    got = f32_bits(orc.mul("exact", M, bits_f32(a), bits_f32(b)))
    with np.errstate(over="ignore"):
        ref = f32_bits(bits_f32(_truncate(a, M)) * bits_f32(_truncate(b, M)))
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("M", [8, 9, 10, 11])
def test_exact_equals_ieee_product_sampled(orc, M):
    rng = np.random.default_rng(200 + M)
    a, b = _normal_operands(rng, 200_000, M)
    got = f32_bits(orc.mul("exact", M, bits_f32(a), bits_f32(b)))
    with np.errstate(over="ignore"):
        ref = f32_bits(bits_f32(_truncate(a, M)) * bits_f32(_truncate(b, M)))
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ Mitchell
def test_mitchell_hand_values(orc):
    for M, a, b, mit, ex in read_golden("mitchell_hand_values.txt"):
        M = int(M)
        a, b, mit, ex = (np.float32(float(v)) for v in (a, b, mit, ex))
        assert orc.mul("mitchell", M, [a], [b])[0] == mit, (a, b)
        assert orc.mul("mitchell", M, [b], [a])[0] == mit, (b, a)
        assert orc.mul("exact", M, [a], [b])[0] == ex, (a, b)


@pytest.mark.parametrize("M", list(range(1, 12)))
def test_mitchell_lut_is_log_domain_construction(orc, M):
    """Mitchell: log2(2^k(1+x)) ~ k + x; add the two logs L; antilog
    2^floor(L) * (1 + frac(L)).  With k = 0 for both mantissas, floor(L) is the
    carry and frac(L) the mantissa.  Integer form: L * 2^M = p + q."""
    t = orc.lut("mitchell", M).astype(np.int64)
    p = np.arange(1 << M, dtype=np.int64)
    L = p[:, None] + p[None, :]                      # L scaled by 2^M
    fl = L >> M                                      # floor(L)
    frac = L - (fl << M)                             # frac(L) scaled by 2^M
    expect = (fl << 23) | (frac << (23 - M))
    assert np.array_equal(t, expect.reshape(-1))


def test_mitchell_error_bound_and_equality(orc):
    M = 7
    mit = orc.lut("mitchell", M).astype(np.int64)
    ex = orc.lut("exact", M).astype(np.int64)

    def value(e):
        carry = e >> 23
        return (1.0 + (e & 0x7FFFFF) / 2.0 ** 23) * 2.0 ** carry

    r = value(mit) / value(ex) - 1.0
    r = r.reshape(1 << M, 1 << M)
    assert r.max() <= 0.0
    assert r.min() == pytest.approx(-1.0 / 9.0, abs=1e-15)
    i, j = np.unravel_index(np.argmin(r), r.shape)
    assert (i, j) == (1 << (M - 1), 1 << (M - 1))    # x = y = 1/2
    zero = r == 0.0
    p = np.arange(1 << M)
    assert np.array_equal(zero, (p[:, None] == 0) | (p[None, :] == 0))


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
@pytest.mark.parametrize("M", [1, 4, 7, 10])
def test_lut_symmetric(orc, kind, M):
    t = orc.lut(kind, M).reshape(1 << M, 1 << M)
    assert np.array_equal(t, t.T)


def test_mitchell_scaling_in_normal_range(orc):
    """For e0 in [1, 253] the product is the mantissa product times 2^(e0-127),
    with the XOR sign: checked against float64 arithmetic on the LUT value."""
    M = 7
    rng = np.random.default_rng(7)
    n = 100_000
    ea = rng.integers(1, 255, size=n)
    eb = rng.integers(np.maximum(1, 128 - ea), np.minimum(255, 381 - ea))
    fa = rng.integers(0, 1 << 23, size=n)
    fb = rng.integers(0, 1 << 23, size=n)
    sa = rng.integers(0, 2, size=n)
    sb = rng.integers(0, 2, size=n)
    a = ((sa << 31) | (ea << 23) | fa).astype(np.uint32)
    b = ((sb << 31) | (eb << 23) | fb).astype(np.uint32)
    x = (fa >> (23 - M)) / 2.0 ** M
    y = (fb >> (23 - M)) / 2.0 ** M
    mant = np.where(x + y < 1.0, 1.0 + x + y, 2.0 * (x + y))
    ref = np.where(sa ^ sb, -1.0, 1.0) * np.ldexp(mant, (ea - 127 + eb - 127).astype(np.int32))
    got = orc.mul("mitchell", M, bits_f32(a), bits_f32(b)).astype(np.float64)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ specials
def test_special_values_hand_worked(orc):
    for kind, M, a, b, want in read_golden("special_values.txt"):
        got = orc.amsim_bits(kind, int(M), int(a, 16), int(b, 16))
        assert got == int(want, 16), (kind, M, a, b, hex(got), want)
        # operand order does not change the result for these symmetric kinds
        got2 = orc.amsim_bits(kind, int(M), int(b, 16), int(a, 16))
        assert got2 == int(want, 16)


def test_zero_sign_and_denormals(orc):
    rng = np.random.default_rng(3)
    x = rng.uniform(-4, 4, size=1000).astype(np.float32)
    den = bits_f32(rng.integers(1, 1 << 23, size=1000).astype(np.uint32)
                   | (rng.integers(0, 2, size=1000).astype(np.uint32) << 31))
    for kind in ("exact", "mitchell"):
        for z in (np.float32(0.0), np.float32(-0.0)):
            out = orc.mul(kind, 7, np.full(1000, z), x)
            assert np.all(out == 0)
            assert np.array_equal(np.signbit(out), np.signbit(x) ^ np.signbit(z))
        out = orc.mul(kind, 7, den, x)
        assert np.all(out == 0)
        assert np.array_equal(np.signbit(out), np.signbit(x) ^ np.signbit(den))


def test_nan_and_inf_propagation(orc):
    rng = np.random.default_rng(4)
    x = rng.uniform(-4, 4, size=1000).astype(np.float32)
    x[x == 0] = 1.0
    for kind in ("exact", "mitchell"):
        nan = orc.mul(kind, 7, np.full(1000, np.nan, np.float32), x)
        assert np.all(f32_bits(nan) == 0x7FC00000)
        inf = orc.mul(kind, 7, np.full(1000, np.inf, np.float32), x)
        assert np.all(np.isinf(inf))
        assert np.array_equal(np.signbit(inf), np.signbit(x))


@pytest.mark.parametrize("M", list(range(1, 12)))
def test_closed_forms_equal_oracle_tables(orc, M):
    """The register-only product values the raw-tile kernel computes for the
    two built-in kinds equal the oracle's expanded table entries (entry +
    1.0f's bits) for every index: Mitchell's is the float with bits
    1.0f + (qa + qb) << (23 - M), the exact one the fp32 product of 1.qa and
    1.qb."""
    q = np.arange(1 << M, dtype=np.uint32)
    qa, qb = np.meshgrid(q, q, indexing="ij")
    one = np.uint32(0x3F800000)
    mitchell = one + ((qa + qb) << np.uint32(23 - M))
    fa = (one + (qa << np.uint32(23 - M))).view(np.float32)
    fb = (one + (qb << np.uint32(23 - M))).view(np.float32)
    exact = (fa * fb).view(np.uint32)
    assert np.array_equal(mitchell.reshape(-1), orc.lut("mitchell", M) + one)
    assert np.array_equal(exact.reshape(-1), orc.lut("exact", M) + one)
