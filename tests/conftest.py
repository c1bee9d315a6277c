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
    """Parse a tests/golden fixture: '# comment' lines skipped, 'key v1 v2 ...'."""
    out = {}
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            out[parts[0]] = parts[1:]
            rows.append(parts)
    return out, rows


@pytest.fixture(scope="session")
def golden():
    return read_golden


@pytest.fixture(scope="session")
def epq_lib():
    """Build (if stale) and load libepq.so; the C ABI under test."""
    from moe_experts_gb300 import build as _build
    _build.build()
    import moe_experts_gb300 as epq
    epq.load()
    return epq


@pytest.fixture(scope="session")
def cuda_dev(epq_lib):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but CUDA is not available")
    torch.cuda.init()
    return torch.device("cuda:0")
