import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


_SCENES = {}


@pytest.fixture(scope="session")
def scene_cache():
    """get(cfg) -> a benchmark scene generated on the GPU, keeping only the latest one alive."""
    import synth

    def get(cfg):
        if cfg not in _SCENES:
            _SCENES.clear()
            _SCENES[cfg] = synth.make_scene(cfg, device="cuda")
        return _SCENES[cfg]
    return get
