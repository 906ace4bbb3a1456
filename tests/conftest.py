import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a); run with -m gpu")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes of CPU oracle time)")


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_sessionstart(session):
    # the host-side generator is plain C; build it if it is missing
    import synth
    synth.build_host()
    # the CUDA libraries are cross-compiled here when nvcc is present and they are missing
    if shutil.which("nvcc") and not _cuda_available():
        try:
            from sparse_expert_mlp_router_b300 import build as moe_build
        except ImportError:
            moe_build = None
        if moe_build is not None and not os.path.exists(moe_build.LIB_PATH):
            moe_build.build()
        if not os.path.exists(synth.DEVICE_LIB):
            synth.build_device()


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device in this process")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
