"""Device-side waits that give up are reported to the caller.

Every wait inside the library's kernels is bounded (copies: 2 s; flags that
other CTAs of the launch raise: amsim_set_flag_wait_limit, 2 s by default).  A
wait that gives up leaves that call's outputs wrong but lets the kernel run to
its end, and records its kind in a device status word that
amsim_device_errors reads.  The test provokes a timeout without any fault or
hang: with the flag-wait limit at 0, a phased launch whose second phase reads
the first phase's output gives up at the first completion flag not yet
raised (the CTAs of phase 0 never all finish within the same nanosecond).
Then the default limit is restored, the status cleared, and the same call
runs again with no timeout and results that match the oracle: the context
stays usable."""
import numpy as np
import pytest

from gpu_helpers import assert_close, to_dev
from approximate_multiplier_dnn_gb300 import GemmProblem

pytestmark = pytest.mark.gpu

DEFAULT_NS = 2_000_000_000


def _phased_pair(amd, lut, rng):
    import torch
    X = rng.standard_normal((512, 784)).astype(np.float32)
    W1 = (rng.standard_normal((784, 1000)) / 28).astype(np.float32)
    W2 = (rng.standard_normal((1000, 500)) / 32).astype(np.float32)
    dX, dW1, dW2 = to_dev(X), to_dev(W1), to_dev(W2)
    Y1 = torch.full((512, 1000), float("nan"), device="cuda")
    Y2 = torch.full((512, 500), float("nan"), device="cuda")
    probs = [GemmProblem.make("N", "N", 512, 1000, 784, 1.0, dX, 784, dW1, 1000, 0.0, Y1, 1000),
             GemmProblem.make("N", "N", 512, 500, 1000, 1.0, Y1, 1000, dW2, 500, 0.0, Y2, 500)]
    first, after = [0, 1], [0, 1]          # phase 1 reads phase 0's output
    ws = amd.workspace(amd.amsim_gemm_phased_workspace_size(probs, first, after, lut))
    keep = (dX, dW1, dW2)

    def run():
        amd.amsim_gemm_phased(probs, first, after, lut, ws=ws)
        return amd.amsim_last_path()
    return run, (X, W1, W2), (Y1, Y2), keep


def test_normal_calls_report_no_timeout(amd, luts):
    lut = luts("mitchell", 7)
    amd.amsim_device_errors(clear=True)
    run, _, _, _keep = _phased_pair(amd, lut, np.random.default_rng(1))
    assert run() & amd.AMSIM_PATH_PHASED
    rc, bits = amd.amsim_device_errors(clear=True)
    assert (rc, bits) == (amd.AMSIM_OK, 0)


def test_flag_wait_timeout_is_reported_and_context_survives(amd, orc, luts):
    import torch
    lut = luts("mitchell", 7)
    amd.amsim_device_errors(clear=True)
    run, (X, W1, W2), (Y1, Y2), _keep = _phased_pair(amd, lut, np.random.default_rng(2))
    try:
        amd.amsim_set_flag_wait_limit(0)
        assert run() & amd.AMSIM_PATH_PHASED
        rc, bits = amd.amsim_device_errors(clear=True)
    finally:
        amd.amsim_set_flag_wait_limit(DEFAULT_NS)
    assert rc == amd.AMSIM_ETIMEOUT, (rc, bits)
    assert bits & amd.AMSIM_WAIT_PHASE, bits
    # the status was cleared; the same call now completes without a timeout
    assert amd.amsim_device_errors(clear=False) == (amd.AMSIM_OK, 0)
    run()
    torch.cuda.synchronize()
    assert amd.amsim_device_errors(clear=True) == (amd.AMSIM_OK, 0)
    y1 = Y1.cpu().numpy()
    rows = np.array([0, 100, 511])
    ref, sa = orc.gemm("mitchell", 7, X, W1, rows=rows)
    assert_close(y1[rows], ref, sa, "phase 0 after the timeout test")
    ref, sa = orc.gemm("mitchell", 7, y1, W2, rows=rows)
    assert_close(Y2.cpu().numpy()[rows], ref, sa, "phase 1 after the timeout test")


def test_wait_limit_arguments(amd):
    L = amd.lib()
    assert L.amsim_set_flag_wait_limit(-1) == amd.AMSIM_EINVAL
    assert L.amsim_set_flag_wait_limit(10_000_000_001) == amd.AMSIM_EINVAL
    assert L.amsim_device_errors(None, 0) == amd.AMSIM_EINVAL
