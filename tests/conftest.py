import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_constants():
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", "page_constants.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = int(v)
    return out


_FULL_WEIGHTS = {}


@pytest.fixture(scope="session")
def full_weights():
    """Seeded weights of the full PersonaPlex shape, (host numpy, device torch), made once
    per session for the GPU tests that need them."""
    if "w" not in _FULL_WEIGHTS:
        import synth
        seed = 1
        _FULL_WEIGHTS["w"] = (synth.make_weights_host(synth.FULL, seed),
                              synth.make_weights_device(synth.FULL, seed))
    return _FULL_WEIGHTS["w"]
