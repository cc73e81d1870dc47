import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The package loads libmoe.so at import and refuses to run without it; build
# it in-tree (nvcc cross-compiles for sm_103a without a GPU) when a fresh
# checkout has none yet.
if not os.path.exists(os.path.join(ROOT, "moe_expert_layer_ep_gb300", "libmoe.so")):
    import subprocess
    subprocess.run([sys.executable, os.path.join(ROOT, "moe_expert_layer_ep_gb300", "build.py")], check=True)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmoe")
    config.addinivalue_line("markers", "slow: CPU test that takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    # Tests marked gpu need a device; everything else must pass on CPU.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
