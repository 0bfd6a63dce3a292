"""amsim_gemm_noalloc, the GEMM entry point for callers that cannot allocate
device memory at call time (no workspace argument; its stream-K partial sums
go to a fixed array inside the library).  Checked through the C ABI against
amsim_gemm with a caller workspace, on two calls in a row so the second call
runs over the array contents the first one left, within the contraction
tolerance the other tests use (1e-5 * sum_k |AMSim product| per element).

The first shape splits its reduction across CTAs (stream-K), so its partial
sums really go through the library's array; the test asserts that path.  The
array holds one stream-K slot pair per SM for up to 159 SMs, so on this GPU no
problem's plan exceeds it (a large multi-wave problem is run to show that); on
a larger device the call takes amsim_gemm's plan for a workspace of the array's
size, and the last test runs that fallback with a workspace too small for the
stream-K slots."""
import ctypes

import numpy as np
import pytest

from gpu_helpers import REL, assert_close, to_dev

pytestmark = pytest.mark.gpu


def _scale_bound(A, B):
    """sum_k |AMSim(a_k, b_k)| <= sum_k |a_k| |b_k| for the exact and Mitchell
    kinds (truncation and Mitchell only shrink magnitudes)."""
    return np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_noalloc_gemm_matches_workspace_gemm_twice(amd, orc, luts, kind):
    import torch
    L = amd.lib()
    lut = luts(kind, 7)
    rng = np.random.default_rng(77)
    for m, n, k in [(300, 500, 2000), (64, 70, 4000), (257, 129, 95)]:
        A = rng.standard_normal((m, k)).astype(np.float32)
        B = rng.standard_normal((k, n)).astype(np.float32)
        dA, dB = to_dev(A), to_dev(B)
        ref = torch.zeros((m, n), dtype=torch.float32, device="cuda")
        nb = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut)
        ws = amd.workspace(nb)
        amd.amsim_gemm("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, ref, n, lut, ws=ws)
        torch.cuda.synchronize()
        want = ref.cpu().numpy()
        bound = _scale_bound(A, B)
        for call in range(2):
            out = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
            rc = L.amsim_gemm_noalloc(b"N", b"N", m, n, k, ctypes.c_float(1.0), dA.data_ptr(), k, dB.data_ptr(), n,
                                      ctypes.c_float(0.0), out.data_ptr(), n, lut.handle,
                                      torch.cuda.current_stream().cuda_stream)
            assert rc == amd.AMSIM_OK, amd.status_string(rc)
            if (m, n, k) == (300, 500, 2000):
                assert amd.amsim_last_path() & amd.AMSIM_PATH_STREAMK, amd.amsim_last_path()
            torch.cuda.synchronize()
            got = out.cpu().numpy()
            assert_close(got, want, 2.0 * bound, f"noalloc vs workspace {m}x{n}x{k} call {call}")
        # and against the oracle on a few rows, with the exact sum of |products|
        rows = np.array([0, m // 2, m - 1])
        oref, sa = orc.gemm(kind, 7, A, B, rows=rows)
        assert_close(got[rows], oref, sa, f"noalloc vs oracle {m}x{n}x{k}")


def test_noalloc_rejects_bad_arguments(amd, luts):
    import torch
    L = amd.lib()
    lut = luts("mitchell", 7)
    x = torch.zeros(64, device="cuda")
    rc = L.amsim_gemm_noalloc(b"N", b"N", 4, 4, 4, ctypes.c_float(1.0), x.data_ptr(), 3, x.data_ptr(), 4,
                              ctypes.c_float(0.0), x.data_ptr(), 4, lut.handle, None)
    assert rc == amd.AMSIM_EINVAL
    rc = L.amsim_gemm_noalloc(b"N", b"N", 4, 4, 4, ctypes.c_float(1.0), x.data_ptr(), 4, x.data_ptr(), 4,
                              ctypes.c_float(0.0), x.data_ptr(), 4, None, None)
    assert rc == amd.AMSIM_EINVAL


def test_noalloc_large_multi_wave_problem_fits_the_array(amd, orc, luts):
    """A 2048 x 2048 x 256 GEMM has 256 tiles, more than one wave on any GPU of
    this family: stream-K over every SM, the largest plan the array must hold."""
    import torch
    L = amd.lib()
    lut = luts("mitchell", 7)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sms <= 159, "the array holds stream-K slots for up to 159 SMs"
    m = n = 2048
    k = 256
    rng = np.random.default_rng(5)
    A = rng.standard_normal((m, k)).astype(np.float32)
    B = rng.standard_normal((k, n)).astype(np.float32)
    dA, dB = to_dev(A), to_dev(B)     # kept alive until the kernel has read them
    out = torch.empty((m, n), dtype=torch.float32, device="cuda")
    rc = L.amsim_gemm_noalloc(b"N", b"N", m, n, k, ctypes.c_float(1.0), dA.data_ptr(), k, dB.data_ptr(), n,
                              ctypes.c_float(0.0), out.data_ptr(), n, lut.handle,
                              torch.cuda.current_stream().cuda_stream)
    assert rc == amd.AMSIM_OK, amd.status_string(rc)
    assert amd.amsim_last_path() & amd.AMSIM_PATH_STREAMK, amd.amsim_last_path()
    torch.cuda.synchronize()
    rows = np.array([0, 1000, m - 1])
    ref, sa = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert_close(out.cpu().numpy()[rows], ref, sa, "noalloc 2048x2048x256")


def test_workspace_too_small_for_streamk_drops_it(amd, orc, luts):
    """The fallback amsim_gemm_noalloc relies on when its array is smaller than
    a plan's stream-K slots: amsim_gemm, given less scratch than the stream-K
    plan asks for, runs the GEMM without stream-K and gets the same results
    within the contraction tolerance."""
    import torch
    lut = luts("mitchell", 7)
    m, n, k = 300, 500, 2000
    rng = np.random.default_rng(78)
    A = rng.standard_normal((m, k)).astype(np.float32)
    B = rng.standard_normal((k, n)).astype(np.float32)
    dA, dB = to_dev(A), to_dev(B)
    nb = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut)
    assert nb > 1024
    full = torch.empty((m, n), dtype=torch.float32, device="cuda")
    amd.amsim_gemm("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, full, n, lut, ws=amd.workspace(nb))
    assert amd.amsim_last_path() & amd.AMSIM_PATH_STREAMK
    small = torch.empty((m, n), dtype=torch.float32, device="cuda")
    amd.amsim_gemm("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, small, n, lut, ws=amd.workspace(1024))
    assert not amd.amsim_last_path() & amd.AMSIM_PATH_STREAMK, amd.amsim_last_path()
    torch.cuda.synchronize()
    got, want = small.cpu().numpy(), full.cpu().numpy()
    assert_close(got, want, 2.0 * _scale_bound(A, B), "no stream-K vs stream-K")
    rows = np.array([0, 150, m - 1])
    ref, sa = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert_close(got[rows], ref, sa, "no stream-K vs oracle")
