"""amsim_gemm_phased: ordered phases of GEMMs in one cooperative launch, each
phase waiting only for the phases it reads.  Every output is checked against
the oracle element by element; a GEMM that reads an earlier phase's output is
checked on the GPU's own copy of that output (the oracle truncates the same
mantissas only when it multiplies the same operands), and its inputs start as
NaN so that a read before the producing phase finished would show."""
import numpy as np
import pytest

from gpu_helpers import REL, assert_close, guarded, guards_intact, to_dev
from approximate_multiplier_dnn_gb300 import GemmProblem

pytestmark = pytest.mark.gpu


def rnd(rng, shape):
    return rng.standard_normal(shape).astype(np.float32)


def host(t):
    return t.detach().cpu().numpy()


def problem(A, B, C, ta=False, tb=False, alpha=1.0, beta=0.0):
    m = A.shape[1] if ta else A.shape[0]
    k = A.shape[0] if ta else A.shape[1]
    n = B.shape[0] if tb else B.shape[1]
    return GemmProblem.make("T" if ta else "N", "T" if tb else "N", m, n, k, alpha, A, A.shape[1], B, B.shape[1],
                            beta, C, n)


def run_phased(amd, lut, probs, first, after, ws="auto"):
    import torch
    if ws == "auto":
        nbytes = amd.amsim_gemm_phased_workspace_size(probs, first, after, lut)
        ws = amd.workspace(nbytes)
    amd.amsim_gemm_phased(probs, first, after, lut, ws=ws)
    torch.cuda.synchronize()
    return amd.amsim_last_path()


def chain(rng, m=256, d=(784, 1000, 500, 10)):
    """A three-layer forward chain with independent work between the layers."""
    X = rnd(rng, (m, d[0]))
    Ws = [(rnd(rng, (d[i], d[i + 1])) / np.sqrt(d[i])).astype(np.float32) for i in range(3)]
    E, F = rnd(rng, (300, 520)), rnd(rng, (520, 700))
    G, H = rnd(rng, (m, 500)), rnd(rng, (d[1], 500))
    return X, Ws, E, F, G, H


def build_chain(amd, rng):
    """Phases: {Y1 = X W1} {D = E F} {Y2 = Y1 W2, after Y1} {Q = G H^T}
    {Y3 = Y2 W3, after Y2} {R = Y1^T G, after Y1}."""
    X, Ws, E, F, G, H = chain(rng)
    dev = {k: to_dev(v) for k, v in dict(X=X, W1=Ws[0], W2=Ws[1], W3=Ws[2], E=E, F=F, G=G, H=H).items()}
    m = X.shape[0]
    outs = {}
    for name, shape in (("Y1", (m, 1000)), ("D", (300, 700)), ("Y2", (m, 500)), ("Q", (m, 1000)),
                        ("Y3", (m, 10)), ("R", (1000, 500))):
        outs[name] = guarded(shape, np.full(shape, np.nan, np.float32))
    o = {k: v[1] for k, v in outs.items()}
    probs = [problem(dev["X"], dev["W1"], o["Y1"]),
             problem(dev["E"], dev["F"], o["D"]),
             problem(o["Y1"], dev["W2"], o["Y2"]),
             problem(dev["G"], dev["H"], o["Q"], tb=True),
             problem(o["Y2"], dev["W3"], o["Y3"]),
             problem(o["Y1"], dev["G"], o["R"], ta=True)]
    first, after = [0, 1, 2, 3, 4, 5], [0, 0, 1, 0, 3, 1]
    # the device inputs travel with the host ones: the problems hold raw pointers
    host_in = dict(X=X, W1=Ws[0], W2=Ws[1], W3=Ws[2], E=E, F=F, G=G, H=H, _dev=dev)
    return probs, first, after, outs, host_in


def check_chain(orc, outs, h, kind="mitchell"):
    for name, (buf, _) in outs.items():
        assert guards_intact(buf), f"write outside {name}"
    o = {k: host(v[1]) for k, v in outs.items()}
    cases = [("Y1", h["X"], h["W1"], False, False), ("D", h["E"], h["F"], False, False),
             ("Y2", o["Y1"], h["W2"], False, False), ("Q", h["G"], h["H"], False, True),
             ("Y3", o["Y2"], h["W3"], False, False), ("R", o["Y1"], h["G"], True, False)]
    for name, A, B, ta, tb in cases:
        assert np.isfinite(A).all(), f"input of {name} not finite"
        ref, sa = orc.gemm(kind, 7, A, B, transA=ta, transB=tb)
        assert_close(o[name], ref, sa, name)


def test_phased_chain_one_launch(amd, orc, luts):
    rng = np.random.default_rng(40)
    lut = luts("mitchell", 7)
    probs, first, after, outs, h = build_chain(amd, rng)
    path = run_phased(amd, lut, probs, first, after)
    assert path & amd.AMSIM_PATH_PHASED and path & amd.AMSIM_PATH_RAW_TILES, path
    check_chain(orc, outs, h)


def test_phased_chain_repeated_calls(amd, orc, luts):
    """Completion flags carry the launch's epoch: a second call on new inputs
    waits for its own producers, not the first call's."""
    import torch
    rng = np.random.default_rng(41)
    lut = luts("mitchell", 7)
    probs, first, after, outs, h = build_chain(amd, rng)
    ws = amd.workspace(amd.amsim_gemm_phased_workspace_size(probs, first, after, lut))
    run_phased(amd, lut, probs, first, after, ws=ws)
    X2 = rnd(rng, h["X"].shape)
    Xd, W1d = to_dev(X2), to_dev(h["W1"])
    probs[0] = problem(Xd, W1d, outs["Y1"][1])
    for name in ("Y1", "Y2", "Y3", "R"):
        outs[name][1].fill_(float("nan"))
    h = dict(h, X=X2)
    path = run_phased(amd, lut, probs, first, after, ws=ws)
    assert path & amd.AMSIM_PATH_PHASED, path
    check_chain(orc, outs, h)


def test_phased_each_phase_after_the_previous(amd, orc, luts):
    """phase_after[ph] = ph everywhere: a strict sequence, each phase reading
    the one before it (reductions of a phase finish before the next loads)."""
    rng = np.random.default_rng(42)
    lut = luts("exact", 7)
    m = 200
    X = rnd(rng, (m, 300))
    Ws = [(rnd(rng, (300, 300)) / np.sqrt(300)).astype(np.float32) for _ in range(4)]
    bufs = [guarded((m, 300), np.full((m, 300), np.nan, np.float32)) for _ in range(4)]
    src = to_dev(X)
    wd = [to_dev(w) for w in Ws]          # alive until the call has run
    probs = []
    for i in range(4):
        probs.append(problem(src, wd[i], bufs[i][1]))
        src = bufs[i][1]
    path = run_phased(amd, lut, probs, [0, 1, 2, 3], [0, 1, 2, 3])
    assert path & amd.AMSIM_PATH_PHASED, path
    inp = X
    for i in range(4):
        assert guards_intact(bufs[i][0])
        got = host(bufs[i][1])
        ref, sa = orc.gemm("exact", 7, inp, Ws[i])
        assert_close(got, ref, sa, f"layer {i}")
        inp = got


def test_phased_empty_phase_and_small_phases(amd, orc, luts):
    """An empty phase, a zero-sized problem, phases with fewer iterations than
    SMs (plain share split) and a 10-wide operand read with plain loads."""
    rng = np.random.default_rng(43)
    lut = luts("mitchell", 7)
    A, B = rnd(rng, (64, 40)), rnd(rng, (40, 10))
    Cb, C = guarded((64, 10), np.full((64, 10), np.nan, np.float32))
    E = rnd(rng, (10, 64))
    Db, D = guarded((10, 10), np.full((10, 10), np.nan, np.float32))
    Za, Zb, Zc = (to_dev(np.zeros(s, np.float32)) for s in ((0, 8), (8, 4), (0, 4)))
    Ad, Bd, Ed = to_dev(A), to_dev(B), to_dev(E)
    probs = [problem(Ad, Bd, C), problem(Za, Zb, Zc), problem(Ed, C, D)]
    path = run_phased(amd, lut, probs, [0, 1, 1, 2], [0, 0, 1, 1])
    assert path & amd.AMSIM_PATH_PHASED, path
    assert guards_intact(Cb) and guards_intact(Db)
    ref, sa = orc.gemm("mitchell", 7, A, B)
    assert_close(host(C), ref, sa, "C")
    ref, sa = orc.gemm("mitchell", 7, E, host(C))
    assert_close(host(D), ref, sa, "D")


def test_phased_results_bit_identical_across_runs(amd, luts):
    """Tiles that the CTA shares cut are summed in a fixed order (the parts'
    CTA order), so repeated calls give the same bits; the MLP step (the bench's
    phased workload, nine GEMMs in five phases) likewise."""
    import torch
    from approximate_multiplier_dnn_gb300 import steps
    from approximate_multiplier_dnn_gb300 import workloads as wl
    rng = np.random.default_rng(47)
    lut = luts("mitchell", 7)
    probs, first, after, outs, h = build_chain(amd, rng)
    ws = amd.workspace(amd.amsim_gemm_phased_workspace_size(probs, first, after, lut))
    runs = []
    for _ in range(3):
        for _, (buf, view) in outs.items():
            view.fill_(float("nan"))
        path = run_phased(amd, lut, probs, first, after, ws=ws)
        assert path & amd.AMSIM_PATH_PHASED, path
        runs.append({k: host(v[1]).view(np.uint32).copy() for k, v in outs.items()})
    for r in runs[1:]:
        for k in r:
            assert np.array_equal(r[k], runs[0][k]), f"{k} differs between runs"
    st = steps.MLPStep(wl.mlp(), lut)
    res = []
    for _ in range(3):
        st.run()
        torch.cuda.synchronize()
        assert amd.amsim_last_path() & amd.AMSIM_PATH_PHASED
        res.append([host(t).view(np.uint32).copy() for t in st.outputs()])
    for r in res[1:]:
        for a, b in zip(r, res[0]):
            assert np.array_equal(a, b), "MLP step outputs differ between runs"


def test_phased_without_scratch_runs_phase_by_phase(amd, orc, luts):
    rng = np.random.default_rng(44)
    lut = luts("mitchell", 7)
    probs, first, after, outs, h = build_chain(amd, rng)
    path = run_phased(amd, lut, probs, first, after, ws=None)
    assert not path & amd.AMSIM_PATH_PHASED, path
    check_chain(orc, outs, h)


def test_phased_rejects_bad_layouts(amd, luts):
    import torch
    lut = luts("mitchell", 7)
    A = torch.zeros((4, 4), device="cuda")
    C = torch.zeros((4, 4), device="cuda")
    probs = [problem(A, A, C) for _ in range(2)]
    for first, after in (([1, 1], [0, 0]), ([0, 3], [0, 0]), ([0, 1], [0, 2]), ([0, 1], [-1, 0]),
                         ([0, 1], [1, 0]), ([1, 0], [0, 0])):
        with pytest.raises(amd.AmsimError):
            amd.amsim_gemm_phased(probs, first, after, lut)
        assert amd.amsim_gemm_phased_workspace_size(probs, first, after, lut) == 0


@pytest.mark.parametrize("kind", ["mitchell", "exact"])
def test_phased_alpha_beta_and_transposes(amd, orc, luts, kind):
    """alpha and beta != 0 on cut tiles (the last part to arrive adds all
    parts in order and stores alpha * sum + beta * C), all four transpose
    pairs, and a phase that reads a transposed output of an earlier one."""
    rng = np.random.default_rng(45)
    lut = luts(kind, 7)
    m, n, k = 300, 520, 700
    A, B = rnd(rng, (k, m)), rnd(rng, (n, k))                  # op(A) = A^T, op(B) = B^T
    C0 = rnd(rng, (m, n))
    Cb, C = guarded((m, n), C0)
    E, F = rnd(rng, (m, 260)), rnd(rng, (260, 400))            # N, N
    G0 = rnd(rng, (m, 400))
    Gb, Gt = guarded((m, 400), G0)
    H = rnd(rng, (n, 96))                                      # phase 2 reads C^T
    Ob, O = guarded((n, 96), np.full((n, 96), np.nan, np.float32))
    Wt = rnd(rng, (96, m))                                     # O = C^T (n x m) . Wt^T (m x 96)
    dev = [to_dev(x) for x in (A, B, E, F, Wt)]
    probs = [problem(dev[0], dev[1], C, ta=True, tb=True, alpha=0.75, beta=-1.25),
             problem(dev[2], dev[3], Gt, alpha=2.0, beta=0.5),
             problem(C, dev[4], O, ta=True, tb=True)]
    path = run_phased(amd, lut, probs, [0, 1, 2], [0, 0, 1])
    assert path & amd.AMSIM_PATH_PHASED, path
    for buf in (Cb, Gb, Ob):
        assert guards_intact(buf)
    ref, sa = orc.gemm(kind, 7, A, B, transA=True, transB=True, alpha=0.75, beta=-1.25, C0=C0)
    # beta * C is rounded once and then each added part rounds at its magnitude:
    # allow 16 ulps of it beside the products' own bound
    assert_close(host(C), ref, 0.75 * sa + 1.25 * np.abs(C0.astype(np.float64)) / REL * 2.0 ** -20, "C")
    ref, sa = orc.gemm(kind, 7, E, F, alpha=2.0, beta=0.5, C0=G0)
    assert_close(host(Gt), ref, 2.0 * sa + 0.5 * np.abs(G0.astype(np.float64)) / REL * 2.0 ** -20, "G")
    ref, sa = orc.gemm(kind, 7, host(C), Wt, transA=True, transB=True)
    assert_close(host(O), ref, sa, "O")


def test_phased_batched_problems(amd, orc, luts):
    """Strided-batched problems (one with a broadcast operand) across phases."""
    rng = np.random.default_rng(46)
    lut = luts("mitchell", 7)
    batch, m, n, k = 6, 128, 200, 96
    A = rnd(rng, (batch, m, k))
    B = rnd(rng, (k, n))                                       # broadcast: strideB = 0
    Yb, Y = guarded((batch, m, n), np.full((batch, m, n), np.nan, np.float32))
    V = rnd(rng, (batch, n, 64))
    Zb, Z = guarded((batch, m, 64), np.full((batch, m, 64), np.nan, np.float32))
    dA, dB, dV = to_dev(A), to_dev(B), to_dev(V)
    probs = [GemmProblem.make("N", "N", m, n, k, 1.0, dA, k, dB, n, 0.0, Y, n, strideA=m * k, strideB=0,
                              strideC=m * n, batch=batch),
             GemmProblem.make("N", "N", m, 64, n, 1.0, Y, n, dV, 64, 0.0, Z, 64, strideA=m * n, strideB=n * 64,
                              strideC=m * 64, batch=batch)]
    path = run_phased(amd, lut, probs, [0, 1], [0, 1])
    assert path & amd.AMSIM_PATH_PHASED, path
    assert guards_intact(Yb) and guards_intact(Zb)
    y = host(Y)
    for b in range(batch):
        ref, sa = orc.gemm("mitchell", 7, A[b], B)
        assert_close(y[b], ref, sa, f"Y[{b}]")
        ref, sa = orc.gemm("mitchell", 7, y[b], V[b])
        assert_close(host(Z)[b], ref, sa, f"Z[{b}]")
