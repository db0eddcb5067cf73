"""The checked build (libdg_debug.so: every kernel compiled with DG_DEBUG=1,
bounds checks before each TMA load and plain global store, ring-fill checks
after each wait, failures recorded in the status word without a trap) runs
small cases of every form in a child process with DG_DEBUG=1: results match
the oracle, no check fires, and the checked library is the one loaded."""
import os
import subprocess
import sys

import pytest

from moe_grouped_gemm_bf16_gb300 import _build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_runs_every_form_clean():
    _build.build(debug=True)
    env = dict(os.environ, DG_DEBUG="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_build_cases.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout[-3000:] + out.stderr[-3000:]
    assert "checked ok" in out.stdout and "libdg_debug.so" in out.stdout, out.stdout[-2000:]
