import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests are collected everywhere but skipped when no device is present,
    # so that `-m "not gpu"` and a bare run both work on a CPU-only machine.
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


_KERNELS = {"auto": 0, "cuda_core": 1, "tensor_core": 2}


@pytest.fixture
def use_kernel():
    """Force a decode kernel ("auto", "cuda_core" or "tensor_core") through the
    library's PA_OPT_DECODE_KERNEL switch; the previous value comes back after
    the test."""
    from paged_kv_decode_cache_gb300 import build, pa
    build.build()
    prev = pa.pa_get_option(pa.PA_OPT_DECODE_KERNEL)

    def _set(kernel):
        pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, _KERNELS[kernel])
    yield _set
    pa.pa_set_option(pa.PA_OPT_DECODE_KERNEL, prev)


@pytest.fixture
def merge_path():
    """'cluster' (the default where P <= 16) or 'grid' (PA_OPT_SPLIT_MERGE =
    PA_MERGE_GRID); the previous value comes back after the test."""
    from paged_kv_decode_cache_gb300 import build, pa
    build.build()
    prev = pa.pa_get_option(pa.PA_OPT_SPLIT_MERGE)

    def _set(path):
        pa.pa_set_option(pa.PA_OPT_SPLIT_MERGE,
                         pa.PA_MERGE_GRID if path == "grid" else pa.PA_MERGE_AUTO)
    yield _set
    pa.pa_set_option(pa.PA_OPT_SPLIT_MERGE, prev)


@pytest.fixture
def cascade_mode():
    """Set PA_OPT_CASCADE ("auto", "always" or "never"); the previous value comes back after the test."""
    from paged_kv_decode_cache_gb300 import build, pa
    build.build()
    prev = pa.pa_get_option(pa.PA_OPT_CASCADE)

    def _set(mode):
        pa.pa_set_option(pa.PA_OPT_CASCADE, {"auto": pa.PA_CASCADE_AUTO, "always": pa.PA_CASCADE_ALWAYS,
                                             "never": pa.PA_CASCADE_NEVER}[mode])
    yield _set
    pa.pa_set_option(pa.PA_OPT_CASCADE, prev)

