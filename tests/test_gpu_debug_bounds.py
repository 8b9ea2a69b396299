"""GPU: the whole GPU suite again on the bounds-checking build.

libtp_b300_debug.so is the library compiled with -DTP_DEBUG_BOUNDS: every
index into a source spectrum, a staged brick, a warp's accumulator tile, an
output image, a gradient row or a workspace list is checked before the
access, a failed check skips the access and sets a bit of a device word
(tp_debug_bounds_word in tp.h).  The child run below repeats every GPU test
on that build (TP_B300_LIB=debug), where the autouse fixture of conftest.py
also requires the word to be zero after each test: the parity cases, edge
cases and full-size launches then show that no index leaves its buffer.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


CHILD_SELFTEST = """
import backprojection_tp_project_gather_b300 as tp
assert tp.LIB_PATH.endswith("libtp_b300_debug.so"), tp.LIB_PATH
tp.tp_debug_bounds_word(reset=True)
for bit in (0, 5, 31):
    tp.tp_debug_bounds_selftest(bit)
    assert tp.tp_debug_bounds_word(reset=True) == 1 << bit, bit
assert tp.tp_debug_bounds_word() == 0
print("selftest ok")
"""


def test_check_word_reports_a_failed_check():
    """The reporting path: a check that fails by construction (it guards no
    access) sets its bit, and reset clears the word."""
    from backprojection_tp_project_gather_b300 import build as b
    b.build(debug=True)
    env = dict(os.environ, TP_B300_LIB="debug")
    r = subprocess.run([sys.executable, "-c", CHILD_SELFTEST], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "selftest ok" in r.stdout, r.stdout + r.stderr


def test_gpu_suite_on_bounds_checking_build():
    from backprojection_tp_project_gather_b300 import build as b
    lib = b.build(debug=True)
    assert os.path.exists(lib)
    env = dict(os.environ, TP_B300_LIB="debug")
    cmd = [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests"), "-m", "gpu", "-x", "-q",
           "-p", "no:cacheprovider",
           "--ignore", os.path.join(ROOT, "tests", "test_gpu_debug_bounds.py")]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    summary = r.stdout.strip().splitlines()[-1]
    print("bounds-checking build:", summary)
    assert " passed" in summary and "error" not in summary and "failed" not in summary, tail
