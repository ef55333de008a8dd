import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu)")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def cuda_lib():
    """Build (if stale) and load libpagedattn; skip when no CUDA device is present."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_gqa_08_gb300 import build, load_library
    build.build()
    lib = load_library()
    from paged_kv_gqa_08_gb300 import pa_read_device_errors
    pa_read_device_errors(reset=True)  # start the session with clear device flags
    return lib
