import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parse a golden fixture: '#' comments, then 'key v1 v2 ...' lines.
    Repeated keys collect into a list of rows."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out.setdefault(key, []).append(vals)
    return out


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library; a GPU test fails loudly when it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_draft_bf16_gb300 import dtree
    return dtree.lib()
