import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(autouse=True)
def _device_checks(request):
    """With the checks build (MOE_LIBRARY=checks): after every GPU test, no
    kernel's index check failed and every workspace guard gap made during the
    test still holds its pattern."""
    yield
    if os.environ.get("MOE_LIBRARY") != "checks" or request.node.get_closest_marker("gpu") is None:
        return
    import torch

    from sparse_mixture_experts_68_b300 import binding as B
    if not torch.cuda.is_available() or not B.is_checks_build():
        return
    torch.cuda.synchronize()
    fails, site, line = B.checks_read(clear=True)
    assert fails == 0, f"{fails} device check(s) failed; first: site {site}, line {line}"
    for layer in B.take_checked_layers():
        assert layer.guards_intact(), f"a kernel wrote into a workspace guard ({layer.wl.name})"
