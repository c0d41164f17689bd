import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built h3attn library")


@pytest.fixture(scope="session")
def h3():
    """The CUDA library binding; GPU tests fail loudly if it cannot load."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    import joint_audio_video_gb300 as h3lib
    h3lib.load()
    return h3lib
