"""The index-checking build (libdpg_debug.so, compiled with DPG_DEBUG): parity
with the oracle and no failed check on ragged, accumulation, 10,000-tensor and
pack/unpack cases; a check made to fail by lowering its bound records its
kernel and skips the access, with no fault.  Runs tests/debug_checks_worker.py
in a process of its own, with DPG_LIBRARY=debug and DPG_TEST_HOOKS=1."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checking_build_parity_and_recorded_failures():
    from zero_optimizer_step_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, DPG_LIBRARY="debug", DPG_TEST_HOOKS="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "debug_checks_worker.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout + r.stderr)[-4000:]
    assert "debug checks ok" in r.stdout
