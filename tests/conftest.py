import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: larger CPU case")


@pytest.fixture(scope="session")
def tiny_artifact():
    import synth
    return synth.ensure_artifact("tiny", 0)


@pytest.fixture(scope="session")
def qwen_artifact():
    import synth
    return synth.ensure_artifact("qwen3-0.6b", 0)


@pytest.fixture(scope="session")
def llama_artifact():
    import synth
    return synth.ensure_artifact("llama-1b", 0)
