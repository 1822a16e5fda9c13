"""The GPU parity tests of the small layers, the staged steps, the edge cases,
the decode tiles and expert-choice routing, run again against the checks
build of the library (libmoe_checks.so: every kernel checks the indices it
gathers or scatters through, and moe_forward's workspace has a guard gap after
each region).  After each of those tests, tests/conftest.py asserts that no
check failed and that every guard gap still holds its fill pattern.  The
compute-sanitizer tools are not available here, so these checks stand in for
them on the layer's own index arithmetic."""

import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB_CHECKS = os.path.join(ROOT, "sparse_mixture_experts_68_b300", "libmoe_checks.so")


def test_small_layers_under_the_checks_build():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    assert os.path.exists(LIB_CHECKS), "libmoe_checks.so is not built"
    env = dict(os.environ, MOE_LIBRARY="checks")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_layer.py"),
           os.path.join(ROOT, "tests", "test_gpu_expert_choice.py"),
           "-k", "small or stages or edge or capacity_one or decode or select or profiled"
                 " or host or graph"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-25:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout, tail
