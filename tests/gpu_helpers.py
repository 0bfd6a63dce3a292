"""Helpers for the GPU parity tests: device buffers with guard canaries, the
contraction tolerance, and NaN/Inf-aware comparison."""
import numpy as np

GUARD = 64
SENTINEL = np.float32(-7.77e33)

# Contraction tolerance: per element |gpu - oracle| <= REL * sum_k |AMSim product|
# (fp32 accumulation in a different order than the oracle's double sum).
REL = 1e-5


def torch():
    import torch as t
    return t


def to_dev(a):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(shape, fill=None):
    """A device tensor view with GUARD sentinel floats before and after it."""
    t = torch()
    n = int(np.prod(shape)) if len(shape) else 1
    buf = t.full((n + 2 * GUARD,), float(SENTINEL), dtype=t.float32, device="cuda")
    view = buf[GUARD:GUARD + n].view(*shape)
    if fill is not None:
        view.copy_(t.from_numpy(np.ascontiguousarray(fill, dtype=np.float32)).cuda().view(*shape))
    return buf, view


def guards_intact(buf) -> bool:
    h = buf.cpu().numpy()
    return bool(np.all(h[:GUARD] == SENTINEL) and np.all(h[-GUARD:] == SENTINEL))


def assert_close(got, ref, scale, what=""):
    """got/ref: float32 arrays; scale: sum_k |product| (float64), same shape."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    nan_g, nan_r = np.isnan(got), np.isnan(ref)
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN pattern differs ({nan_g.sum()} vs {nan_r.sum()})"
    fin = ~nan_r
    inf_r = np.isinf(ref) & fin
    assert np.array_equal(got[inf_r], ref[inf_r]), f"{what}: infinities differ"
    m = fin & ~inf_r
    err = np.abs(got[m] - ref[m])
    tol = REL * scale[m]
    bad = err > tol
    if bad.any():
        i = np.argmax(err - tol)
        raise AssertionError(f"{what}: {bad.sum()} of {m.sum()} elements exceed tol; worst err {err[i]:.3e} "
                             f"tol {tol[i]:.3e} got {got[m][i]!r} ref {ref[m][i]!r}")


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
