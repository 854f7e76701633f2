import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def force_pair():
    """Run the test's calls on the CTA-pair kernel where it applies (GQA groups
    of a multiple of 4 query heads, heads 72..128, contiguous K/V); the
    library's own choice is restored afterwards."""
    import causal_prefill_flash_gb300 as fa
    fa.debug_force_path("pair")
    try:
        yield
    finally:
        fa.debug_force_path("auto")


@pytest.fixture
def force_persistent():
    """Run the test's split-KV calls on the persistent kernel, whatever their
    schedule (the library otherwise runs one-piece-per-CTA schedules on the
    split-KV kernel); the library's own choice is restored afterwards."""
    import causal_prefill_flash_gb300 as fa
    fa.debug_force_path("persistent")
    try:
        yield
    finally:
        fa.debug_force_path("auto")
