"""The coverage and bounds build (include/pk_debug.h) on the GPU.

Builds libpk_coverage.so (the same sources with PK_DEBUG_COVERAGE) and runs
tests/coverage_cases.py against it in a child process: every kernel family
and path, on small ragged grids, must store each interior cell exactly once
per storing pass, never a ring or pad cell, and read only inside its rows,
with the oracle's bits.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_every_pass_stores_each_interior_cell_once():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from iterative_stencil_solver_gb300 import build_ext
    lib = build_ext.build(coverage=True)
    env = dict(os.environ, PK_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "coverage_cases.py")], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "coverage checks passed" in r.stdout
