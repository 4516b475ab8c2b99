import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    # The CUDA library (cross-compiled for sm_103a; loads without a GPU) and the
    # C oracle are built in-tree on first use; both builds are no-ops when current.
    from lossless_kv_cache_bf16_gb300 import build
    from oracle import oracle

    build.build()
    oracle.build()


@pytest.fixture(scope="session")
def orc():
    from oracle import oracle

    return oracle.default()
