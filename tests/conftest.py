import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(scope="session")
def amd():
    """The built library on a CUDA device (fails loudly when either is missing)."""
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import approximate_multiplier_dnn_gb300 as am
    am.build()
    am.lib()
    torch.cuda.set_device(0)
    return am


@pytest.fixture(scope="session")
def luts(amd):
    """Device LUT handles, built once per (kind, M)."""
    cache = {}

    def get(kind, M):
        key = (kind, M)
        if key not in cache:
            cache[key] = amd.Lut.build(kind, M)
        return cache[key]

    yield get
    for v in cache.values():
        v.close()
