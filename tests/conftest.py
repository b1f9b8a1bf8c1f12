import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running (full-size model)")


@pytest.fixture(scope="session")
def weights_dir(tmp_path_factory):
    d = os.environ.get("S2_WEIGHTS_DIR")
    if d:
        os.makedirs(d, exist_ok=True)
        return d
    return str(tmp_path_factory.mktemp("s2w"))


@pytest.fixture(scope="session")
def micro_path(weights_dir):
    from s2_inputs import MICRO, ensure_weights
    return ensure_weights(MICRO, weights_dir)


@pytest.fixture(scope="session")
def tiny_path(weights_dir):
    from s2_inputs import TINY, ensure_weights
    return ensure_weights(TINY, weights_dir)
