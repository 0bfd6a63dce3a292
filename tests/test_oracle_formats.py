"""Pins of the oracle's (1, e, m) formats with fewer exponent bits than fp32
(ApproxTrain Sec. V-B, last paragraph: e from 1 to 8 given an exponent casting
function).  Reading: IEEE-style bias 2^(e-1) - 1, biased 0 = zero, all ones =
Inf/NaN; operands are cast by re-biasing (zero below the smallest normal, Inf
from the all-ones exponent up), Algorithm 2 runs with that bias, the product
returns as fp32.  Facts that do not come from the oracle itself:

* hand-worked products at e = 4, 2 and 1 (tests/golden/format_values.txt);
* e = 5 against IEEE half precision (numpy float16's own smallest normal and
  overflow exponent): an operand is cast to zero exactly when its truncation
  is below float16's smallest normal, to Inf exactly when float16 overflows;
  products are the exact float64 product of the truncated operands, zero when
  the uncarried exponent sum is below float16's range and Inf when the
  product reaches 2^maxexp;
* e = 8 gives the fp32 results of the default format.
"""
import numpy as np
import pytest

from conftest import read_golden


def bits_f32(u):
    return np.asarray(u, dtype=np.uint32).view(np.float32)


def f32_bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def test_format_hand_worked(orc):
    for E, a, b, want in read_golden("format_values.txt"):
        got = orc.amsim_bits("exact", 3, int(a, 16), int(b, 16), ebits=int(E))
        assert got == int(want, 16), (E, a, b, hex(got), want)


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
def test_e8_is_the_default_format(orc, kind):
    rng = np.random.default_rng(5)
    a = rng.integers(0, 1 << 32, size=100_000, dtype=np.uint64).astype(np.uint32)
    b = rng.integers(0, 1 << 32, size=100_000, dtype=np.uint64).astype(np.uint32)
    got = f32_bits(orc.mul(kind, 7, bits_f32(a), bits_f32(b), ebits=8))
    want = f32_bits(orc.mul(kind, 7, bits_f32(a), bits_f32(b)))
    assert np.array_equal(got, want)


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
def test_half_format_matches_ieee_half_ranges(orc, kind):
    M = 10
    fi = np.finfo(np.float16)
    tiny = float(fi.tiny)                 # 2^-14, smallest normal half
    big = 2.0 ** fi.maxexp                # 2^16: every half binade is below it
    rng = np.random.default_rng(6)
    n = 200_000
    exps = rng.integers(-20, 20, size=n)
    sig = rng.uniform(1.0, 2.0, size=n)
    sgn = np.where(rng.random(n) < 0.5, -1.0, 1.0)
    a = (sgn * np.ldexp(sig, exps)).astype(np.float32)
    b = (np.where(rng.random(n) < 0.5, -1.0, 1.0)
         * np.ldexp(rng.uniform(1.0, 2.0, size=n), rng.integers(-20, 20, size=n))).astype(np.float32)
    keep = np.uint32((0xFFFFFFFF << (23 - M)) & 0xFFFFFFFF)
    ta = bits_f32(f32_bits(a) & keep).astype(np.float64)
    tb = bits_f32(f32_bits(b) & keep).astype(np.float64)
    # classification of each operand by float16's own ranges
    h_a = ta.astype(np.float16)
    h_b = tb.astype(np.float16)
    zero = (np.abs(ta) < tiny) | (np.abs(tb) < tiny)
    inf_op = np.isinf(h_a) | np.isinf(h_b)
    assert np.array_equal(np.isinf(h_a), np.abs(ta) >= big)
    _, ea = np.frexp(np.abs(ta))
    _, eb = np.frexp(np.abs(tb))
    esum = (ea - 1) + (eb - 1)                           # uncarried exponent of the product
    if kind == "exact":
        prod = ta * tb
    else:
        x = np.abs(ta) / np.ldexp(1.0, ea - 1) - 1.0
        y = np.abs(tb) / np.ldexp(1.0, eb - 1) - 1.0
        prod = np.sign(ta) * np.sign(tb) * np.where(x + y < 1.0, 1.0 + x + y, 2.0 * (x + y)) * np.ldexp(1.0, esum)
    sign = np.signbit(ta) ^ np.signbit(tb)
    want = np.where(esum < np.log2(tiny), 0.0, prod)
    want = np.where(np.abs(want) >= big, np.inf, want)
    want = np.where(inf_op, np.inf, want)
    want = np.where(zero & inf_op, np.nan, np.where(zero, 0.0, want))
    want = np.where(np.isnan(want), want, np.where(sign, -np.abs(want), np.abs(want)))
    got = orc.mul(kind, M, a, b, ebits=5).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(want[ok]))
    # every class is exercised
    assert zero.sum() > 1000 and inf_op.sum() > 1000 and (np.isinf(want) & ~inf_op).sum() > 100


def test_format_contraction_uses_format_products(orc):
    """A GEMM in a narrow format sums exactly the format's elementwise products."""
    rng = np.random.default_rng(8)
    A = (rng.standard_normal((4, 50)) * 30).astype(np.float32)
    B = (rng.standard_normal((50, 3)) * 30).astype(np.float32)
    got, sa = orc.gemm("mitchell", 4, A, B, ebits=4)
    prods = np.stack([orc.mul("mitchell", 4, np.repeat(A[i][:, None], 3, 1), B, ebits=4) for i in range(4)])
    ref = prods.astype(np.float64).sum(axis=1)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin].astype(np.float64), ref[fin].astype(np.float32).astype(np.float64))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
