"""amsim_set_cooperative_launches: with cooperative launches off, stream-K
GEMMs finish their cut tiles with the separate fixup kernel, which adds the
same partial sums in the same CTA order -- bit-identical to the fused
reduction -- on every kernel path (raw tiles with tail tiles and cost-cut
shares, predecoded planes, in-kernel decode); a phased call runs phase by
phase.  Every case is also checked against the oracle."""
import numpy as np
import pytest

from gpu_helpers import assert_close, to_dev
from approximate_multiplier_dnn_gb300 import GemmProblem

pytestmark = pytest.mark.gpu


def rnd(rng, shape):
    return rng.standard_normal(shape).astype(np.float32)


@pytest.fixture
def coop(amd):
    yield amd.amsim_set_cooperative_launches
    amd.amsim_set_cooperative_launches(True)


def run(amd, lut, A, lda, B, m, n, k, ws_bytes):
    import torch
    C = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    amd.amsim_gemm("N", "N", m, n, k, 1.0, A, lda, B, n, 0.0, C, n, lut,
                   ws=amd.workspace(ws_bytes) if ws_bytes else None)
    torch.cuda.synchronize()
    return C.cpu().numpy(), amd.amsim_last_path()


# (m, n, k, kernel path): raw tiles with a narrow tail (cost-cut shares), raw
# tiles with a wide tail, predecoded planes, in-kernel decode (A behind an odd
# leading dimension, scratch one byte short of the planes)
CASES = [(64, 320, 20000, "raw"), (64, 360, 12000, "raw"), (1000, 1000, 3000, "planes"),
         (1000, 1000, 3000, "in_kernel")]


@pytest.mark.parametrize("m,n,k,path", CASES)
def test_fixup_kernel_bit_identical_to_fused(amd, orc, luts, coop, m, n, k, path):
    import torch
    rng = np.random.default_rng(m + n + k)
    A, B = rnd(rng, (m, k)), rnd(rng, (k, n))
    lut = luts("mitchell", 7)
    lda = k + 1 if path == "in_kernel" else k
    dA = torch.zeros((m, lda), dtype=torch.float32, device="cuda")
    dA[:, :k] = to_dev(A)
    dB = to_dev(B)
    full = amd.amsim_gemm_workspace_size("N", "N", m, n, k, 1, lut)
    nb = full - 1 if path == "in_kernel" else full
    want = {"raw": amd.AMSIM_PATH_RAW_TILES, "planes": amd.AMSIM_PATH_PLANES,
            "in_kernel": amd.AMSIM_PATH_INKERNEL_DECODE}[path]
    outs = []
    for on in (True, False):
        coop(on)
        got, taken = run(amd, lut, dA, lda, dB, m, n, k, nb)
        assert taken & want and taken & amd.AMSIM_PATH_STREAMK, taken
        assert bool(taken & amd.AMSIM_PATH_FIXUP) == (not on), taken
        outs.append(got)
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    rows = np.array([0, m // 3, m - 1])
    ref, sa = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert_close(outs[1][rows], ref, sa, f"fixup {m}x{n}x{k} {path}")


def test_phased_call_without_cooperative_launches(amd, orc, luts, coop):
    """A two-phase call (the second phase reads the first's output) runs as
    consecutive grouped launches: no phased path, oracle parity."""
    import torch
    rng = np.random.default_rng(31)
    m, n, k = 256, 576, 3000
    A, B, W2 = rnd(rng, (m, k)), rnd(rng, (k, n)), rnd(rng, (n, 72))
    lut = luts("mitchell", 7)
    dA, dB, dW2 = to_dev(A), to_dev(B), to_dev(W2)
    C1 = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    C2 = torch.full((m, 72), float("nan"), dtype=torch.float32, device="cuda")
    probs = [GemmProblem.make("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, C1, n),
             GemmProblem.make("N", "N", m, 72, n, 1.0, C1, n, dW2, 72, 0.0, C2, 72)]
    first, after = [0, 1], [0, 1]
    nb = amd.amsim_gemm_phased_workspace_size(probs, first, after, lut)
    coop(False)
    amd.amsim_gemm_phased(probs, first, after, lut, ws=amd.workspace(nb))
    torch.cuda.synchronize()
    taken = amd.amsim_last_path()
    assert not taken & amd.AMSIM_PATH_PHASED, taken
    c1, c2 = C1.cpu().numpy(), C2.cpu().numpy()
    rows = np.array([0, 100, m - 1])
    ref, sa = orc.gemm("mitchell", 7, A, B, rows=rows)
    assert_close(c1[rows], ref, sa, "C1")
    ref2, sa2 = orc.gemm("mitchell", 7, c1, W2, rows=rows)
    assert_close(c2[rows], ref2, sa2, "C2")
