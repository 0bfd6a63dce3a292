"""Elementwise AMSim on the GPU (Algorithm 2 of the ApproxTrain page,
Sec. V-B) against the CPU oracle: bit-exact on every input class."""
import numpy as np
import pytest

from gpu_helpers import bits, guarded, guards_intact, to_dev
from approximate_multiplier_dnn_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run_mul(amd, lut, a, b, offset=0):
    """Run amsim_mul on device copies (optionally at an element offset so the
    pointers are not 16-byte aligned); returns the host result."""
    import torch
    n = a.size
    da = torch.zeros(n + offset, dtype=torch.float32, device="cuda")
    db = torch.zeros(n + offset, dtype=torch.float32, device="cuda")
    da[offset:] = to_dev(a)
    db[offset:] = to_dev(b)
    buf, c = guarded((n + offset,))
    amd.amsim_mul(da[offset:], db[offset:], c[offset:], n, lut)
    torch.cuda.synchronize()
    assert guards_intact(buf)
    return c[offset:].cpu().numpy()


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
@pytest.mark.parametrize("M", list(range(1, 12)))
def test_lut_entries_on_device(amd, orc, luts, kind, M):
    lut = luts(kind, M)
    assert np.array_equal(lut.entries(), orc.lut(kind, M))
    info = lut.info()
    assert info["M"] == M and info["width_bits"] in (8, 16, 32)
    if kind == "mitchell" and M <= 7:
        assert info["width_bits"] == 8
    if kind == "exact" and M == 7:
        assert info["width_bits"] == 16


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
def test_special_value_mix_bitexact(amd, orc, luts, kind):
    """2^20 pairs ~ U[-1,1] with zeros, denormals, infinities, NaNs, and
    exponent-boundary values mixed in (the elementwise workload)."""
    d = wl.elementwise_pairs(1 << 20, seed=0)
    got = run_mul(amd, luts(kind, 7), d["a"], d["b"])
    ref = orc.mul(kind, 7, d["a"], d["b"])
    assert np.array_equal(bits(got), bits(ref))


@pytest.mark.parametrize("kind", ["exact", "mitchell"])
@pytest.mark.parametrize("M", list(range(1, 12)))
def test_all_mantissa_pairs_and_exponent_boundaries(amd, orc, luts, kind, M):
    """Every mantissa pair (M <= 7; a sample above) crossed with signs and the
    exponent pairs around e0 = ea+eb-127 in {-1,0,1,2,253,254,255}."""
    rng = np.random.default_rng(1000 + M)
    side = 1 << M
    if M <= 7:
        p, q = np.meshgrid(np.arange(side, dtype=np.uint32), np.arange(side, dtype=np.uint32), indexing="ij")
        p, q = p.reshape(-1), q.reshape(-1)
    else:
        p = rng.integers(0, side, size=1 << 16).astype(np.uint32)
        q = rng.integers(0, side, size=1 << 16).astype(np.uint32)
    e_pairs = np.array([(126, 0 + 1), (127, 1), (127, 0), (126, 1), (1, 126), (128, 1),
                        (254, 127), (253, 127), (254, 128), (190, 190), (191, 191), (100, 27), (200, 55)],
                       dtype=np.uint32)
    n = p.size
    ei = rng.integers(0, len(e_pairs), size=n)
    ea, eb = e_pairs[ei, 0], e_pairs[ei, 1]
    low = rng.integers(0, 1 << (23 - M), size=n, dtype=np.uint32) if M < 23 else 0
    low2 = rng.integers(0, 1 << (23 - M), size=n, dtype=np.uint32)
    sa = rng.integers(0, 2, size=n, dtype=np.uint32) << 31
    sb = rng.integers(0, 2, size=n, dtype=np.uint32) << 31
    a = (sa | (ea << 23) | (p << (23 - M)) | low).astype(np.uint32).view(np.float32)
    b = (sb | (eb << 23) | (q << (23 - M)) | low2).astype(np.uint32).view(np.float32)
    got = run_mul(amd, luts(kind, M), a, b)
    ref = orc.mul(kind, M, a, b)
    assert np.array_equal(bits(got), bits(ref))


@pytest.mark.parametrize("n,offset", [(1, 0), (3, 1), (1027, 1), (4096, 0), (4099, 3)])
def test_ragged_and_unaligned(amd, orc, luts, n, offset):
    d = wl.elementwise_pairs(n, seed=n)
    got = run_mul(amd, luts("mitchell", 7), d["a"], d["b"], offset=offset)
    assert np.array_equal(bits(got), bits(orc.mul("mitchell", 7, d["a"], d["b"])))


def test_zero_length_and_errors(amd, luts):
    import torch
    lut = luts("mitchell", 7)
    x = torch.zeros(4, device="cuda")
    amd.amsim_mul(x, x, x, 0, lut)
    with pytest.raises(amd.AmsimError) as e:
        amd.amsim_mul(x, x, x, -1, lut)
    assert e.value.status == amd.AMSIM_EINVAL
    with pytest.raises(amd.AmsimError):
        amd.amsim_mul(None, x, x, 4, lut)
