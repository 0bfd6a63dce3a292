"""Host-side models bench.py uses for its roofline lines (no GPU)."""
import importlib.util
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_bank_degree_special_cases():
    b = load_bench()
    # a 128-byte row (M = 7, 8-bit entries) holds one word per bank: every
    # gather is a single wavefront however the columns fall
    assert b.bank_degree(7, 8) == 1.0
    # 16-bit entries of M = 7: two words per bank; 32 lanes all but surely hit
    # both words of some bank
    assert abs(b.bank_degree(7, 16) - 2.0) < 1e-3
    # a wider row can only spread the words over more conflicts
    seq = [b.bank_degree(M, 16) for M in range(7, 12)]
    assert all(x <= y + 1e-9 for x, y in zip(seq, seq[1:]))
    assert all(1.0 <= x <= 32.0 for x in seq)


def test_bank_degree_matches_brute_force():
    """A direct count over random gathers agrees with the vectorised one."""
    b = load_bench()
    rng = np.random.default_rng(7)
    M, wb = 9, 16
    tot = 0
    n = 3000
    for _ in range(n):
        cols = rng.integers(0, 1 << M, size=32)
        words = {int(c) * (wb // 8) // 4 for c in cols}
        per_bank = {}
        for w in words:
            per_bank[w % 32] = per_bank.get(w % 32, 0) + 1
        tot += max(per_bank.values())
    assert abs(tot / n - b.bank_degree(M, wb)) < 0.05


def test_distinct_sectors_formula():
    b = load_bench()
    rng = np.random.default_rng(8)
    for M, wb in [(9, 16), (11, 16)]:
        sectors = (1 << M) * wb // 8 // 32
        got = np.mean([len(set(rng.integers(0, sectors, size=32).tolist())) for _ in range(4000)])
        assert abs(got - b.distinct_sectors_per_warp_lookup(M, wb)) < 0.1


def test_path_names_decodes_bits():
    b = load_bench()

    class Fake:
        AMSIM_PATH_PLANES = 1
        AMSIM_PATH_STREAMK = 16
        AMSIM_PATH_WIDE_TILES = 4096

    assert b.path_names(Fake, 1 | 4096) == ["planes", "wide_tiles"]
    assert b.path_names(Fake, 0) == []
