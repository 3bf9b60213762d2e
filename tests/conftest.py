import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(autouse=True)
def _library_built(request):
    """GPU tests call the CUDA library: build it (in-tree, sm_103a) once per session first."""
    if "gpu" in request.keywords:
        _build_once()


_built = []


def _build_once():
    if not _built:
        from paged_gqa_decode_global_gb300 import binding, build
        build.build()
        binding.load_library()
        _built.append(True)
