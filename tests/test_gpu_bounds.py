"""The bounds-checked build (libmoe_debug.so, compiled with -DMOE_DEBUG_BOUNDS).

Every global and shared-memory index the route kernel and both expert kernels
compute is checked before its access; a miss is recorded as
MOE_ERR_DEVICE_BOUNDS with a diagnostics record and the access is skipped. No
check traps, so the GPU stays usable. compute-sanitizer is closed on this machine;
this build is the substitute evidence that no kernel indexes out of range.

* The small parity cases, the exact-arithmetic cases and the Guard's limit
  cases run once against the bounds-checked library, in a child process
  (MOE_DEBUG_BOUNDS=1 selects it); every step must finish with MOE_OK.
* A positive control shows the checks are live without any out-of-bounds
  access: MOE_FLAG_TEST_BOUNDS halves the combine-counter capacity the checks
  see, so a check trips at an index that is still inside the buffer.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from moe_expert_layer_top_gb300 import abi

from gpu_cases import CudaStep, check_y, oracle_experts

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    import moe_expert_layer_top_gb300 as pkg
    pkg.build.build()
    assert os.path.exists(pkg.build.DEBUG_LIB_PATH)
    assert torch.cuda.is_available()


@pytest.fixture
def debug_library():
    """Load libmoe_debug.so for one test, then go back to libmoe.so."""
    prev = os.environ.get("MOE_DEBUG_BOUNDS")
    os.environ["MOE_DEBUG_BOUNDS"] = "1"
    abi._lib = None
    abi.load()
    try:
        yield
    finally:
        torch.cuda.synchronize()
        if prev is None:
            os.environ.pop("MOE_DEBUG_BOUNDS", None)
        else:
            os.environ["MOE_DEBUG_BOUNDS"] = prev
        abi._lib = None
        abi.load()


@pytest.mark.parametrize("path", ["gemv", "mma"])
def test_bounds_checks_are_live(path, debug_library):
    assert abi.library_path().endswith("libmoe_debug.so")
    flags = {"gemv": abi.MOE_FLAG_PATH_GEMV, "mma": abi.MOE_FLAG_PATH_MMA}[path]
    T, H, E, k, I = 40, 512, 8, 2, 256
    g = CudaStep(T, H, E, k, I, "zipf", seed=11, flags=flags | abi.MOE_FLAG_TEST_BOUNDS).run()
    assert g.status_code == abi.MOE_ERR_DEVICE_BOUNDS
    assert g.diag[0] == 6 and g.diag[1] == {"gemv": 34, "mma": 22}[path], g.diag
    assert g.diag[3] >= g.diag[4]          # the index and the (halved) limit the check saw
    g.close()
    # the same step without the hook, on the bounds-checked library: clean and correct
    ok = CudaStep(T, H, E, k, I, "zipf", seed=11, flags=flags).run()
    assert ok.status_code == abi.MOE_OK, (abi.moe_status_string(ok.status_code), ok.diag)
    r = oracle.moe_step(ok.x_bits, ok.lg, k, oracle_experts(11, E, H, I))
    check_y(ok.y_bits, r["y"])
    ok.close()


def test_parity_and_limit_cases_under_the_bounds_checked_build():
    env = dict(os.environ, MOE_DEBUG_BOUNDS="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_parity.py", "tests/test_gpu_exact.py", "tests/test_gpu_limits.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and "failed" not in r.stdout, tail
