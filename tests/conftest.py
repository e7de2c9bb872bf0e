import functools
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


@functools.lru_cache(maxsize=None)
def cached_case(cfg_id: int, order: str = "raster"):
    """One generated workload per process (workload 5 takes ~15 s to voxelise)."""
    from synth import make_case
    return make_case(cfg_id, order)


@pytest.fixture(scope="session")
def case():
    return cached_case
