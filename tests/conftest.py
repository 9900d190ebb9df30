import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library, loaded; building it first if needed."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w4a16_group_quantised_gb300 import build as libbuild
    libbuild.build()
    import w4a16_group_quantised_gb300 as w
    w.load_library()
    return w
