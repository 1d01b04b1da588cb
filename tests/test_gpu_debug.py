"""The debug build on a B300 (needs a GPU): ``libbitlinear_debug.so``, built
with -DBITLINEAR_DEBUG, checks every plain global load and store of the
kernels against its buffer's extent, skips a failing access and reports it
as BITLINEAR_ERR_BOUNDS.

Both tests run in child processes with BITLINEAR_DEBUG=1, which makes the
binding load the debug library:
- the reporting path, through bitlinear_debug_selftest (a kernel that
  records one failed check without touching memory: no access is ever made
  out of bounds on purpose);
- the guard-byte, fused, variant and engine-route parity suites again, on the
  debug library: every call there asserts bitlinear_check_status() == OK, so
  a single failed bounds check anywhere fails them.
"""
import os
import subprocess
import sys

import pytest

from bitlinear_02_b300 import build as blbuild

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _env():
    env = dict(os.environ)
    env["BITLINEAR_DEBUG"] = "1"
    return env


@pytest.fixture(scope="module", autouse=True)
def _debug_lib():
    blbuild.build()
    blbuild.build(debug=True)


def test_selftest_reports_err_bounds():
    code = (
        "import torch, bitlinear_02_b300 as bl\n"
        "assert bl.library_path().endswith('libbitlinear_debug.so')\n"
        "bl.load_library(); torch.cuda.init()\n"
        "assert bl.bitlinear_check_status() == bl.OK\n"
        "assert bl.bitlinear_debug_selftest() == bl.OK\n"
        "assert bl.bitlinear_check_status() == bl.ERR_BOUNDS\n"
        "assert bl.bitlinear_check_status() == bl.OK  # read and cleared\n"
        "print('selftest ok')\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_env(), capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "selftest ok" in r.stdout
    assert "device bounds check failed in" in r.stderr and "api.cu" in r.stderr


def test_parity_suites_pass_with_bounds_checks():
    args = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
            "tests/test_gpu_guards.py", "tests/test_gpu_fused.py", "tests/test_gpu_variants.py",
            "tests/test_gpu_engines.py::test_every_route_bit_exact"]
    r = subprocess.run(args, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=1200)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert "passed" in r.stdout and "failed" not in r.stdout, tail
