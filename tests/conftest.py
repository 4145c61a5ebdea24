import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


def load_golden(name):
    import json

    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        return json.load(f)


def build_product_library():
    """Run pagedattention_decode_pkv_gb300/build.py by path: importing it as a
    submodule would load the package (and a stale libpkv.so) first."""
    import importlib.util

    path = os.path.join(ROOT, "pagedattention_decode_pkv_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_pkv_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build_library()


@pytest.fixture(scope="session")
def pkv():
    """The product binding; builds libpkv.so in-tree first if needed (nvcc, sm_103a)."""
    build_product_library()
    import pagedattention_decode_pkv_gb300 as mod

    return mod


@pytest.fixture(scope="session")
def cuda_dev(pkv):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
