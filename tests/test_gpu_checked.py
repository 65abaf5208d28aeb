"""The checked debug build (libnf4_checked.so, NF4_CHECKED=1) on the GPU: every
product path on small ragged shapes, with in-kernel index checks, matches the
oracle and leaves the device status clean; an injected failure of an index check
is recorded as NF4_ERR_BOUNDS without an out-of-range access.  The cases run in a
child process (tests/checked_cases.py), since the binding loads one library per
process."""
import os
import subprocess
import sys

import pytest

from bit_nf4_quantized_linear_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_checked_build_every_path_clean():
    build.build(checked=True)
    env = dict(os.environ, NF4_CHECKED="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    out = r.stdout + r.stderr
    assert r.returncode == 0, out[-4000:]
    assert "CHECKED OK" in r.stdout, out[-4000:]
    assert "ok injected failure recorded" in r.stdout
