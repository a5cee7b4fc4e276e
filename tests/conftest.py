import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: longer CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def golden(name):
    import json
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def stp_lib():
    """libstp.so, built in-tree if it is missing or older than its sources."""
    from sft_trie_build_gb300 import build, stp
    srcs = [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC)]
    srcs.append(os.path.join(ROOT, "include", "stp.h"))
    if (not os.path.exists(build.LIB)
            or os.path.getmtime(build.LIB) < max(os.path.getmtime(s) for s in srcs)):
        build.build()
    return stp.lib()
