"""The debug build (WS_DEBUG=1 selects libws_b300_debug.so, whose kernels
bounds-check every index they compute for a global-memory access and record
a failure in the device error word instead of touching memory): one small
pass of every kernel, in a child process so that this process keeps the
normal library, matches the oracle with the error word clean."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_build_runs_clean_and_matches_the_oracle():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    env = dict(os.environ, WS_DEBUG="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_build_case.py")],
                         capture_output=True, text=True, timeout=900, cwd=ROOT, env=env)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-3000:]
    assert "debug build ok" in res.stdout
