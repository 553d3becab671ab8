import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libsgq.so")


def pytest_collection_modifyitems(config, items):
    """Skip GPU tests with a clear reason when no GPU is present, unless they
    were selected explicitly with -m gpu (then they fail loudly instead)."""
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    markexpr = config.getoption("-m") or ""
    if "gpu" in markexpr and "not gpu" not in markexpr:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def sgq_lib():
    """The CUDA library, built in-tree if it is missing or older than its sources."""
    import glob

    import __graft_entry__ as g
    from swiglu_fp8_activation_gb300 import binding

    lib = os.path.join(g.PKG, "libsgq.so")
    srcs = glob.glob(os.path.join(g.CSRC, "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(s) for s in srcs):
        g.build_cuda()
        binding._lib = None
    return binding.library()
