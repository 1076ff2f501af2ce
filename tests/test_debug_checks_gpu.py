"""The bounds-checking build on the GPU.

libfa_gb300_debug.so is the library compiled with FA_DEBUG_CHECKS: every kernel
checks each global index it computes (row statistics, fp8 scales and codes, the
output rows it stores, the boxes of its TMA stores) against the tensor's size,
skips an access that fails and records device status 7.  It stands in for a
memory checker on a GPU where none can run.

Both tests run in a child process with FA_GB300_LIBRARY pointing at that build,
so this process keeps the normal library:
  * the self-test enqueues one failing check (no memory is touched) and the
    status must come back as the bounds-check error, then clear;
  * the parity suites (forward, backward both paths, fp16, dropout, fp8) run
    against the checking build and, after every test, the status word must be
    clear: no kernel computed an index outside its tensor.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["test_fwd_gpu.py", "test_bwd_gpu.py", "test_f16_gpu.py", "test_dropout_gpu.py",
          "test_fp8_gpu.py"]


@pytest.fixture(scope="module")
def debug_env(fa):
    from exact_io_aware_tcgen05_gb300 import build as b
    env = dict(os.environ)
    env["FA_GB300_LIBRARY"] = b.build(debug=True)
    return env


def _run(cmd, env, timeout):
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, (r.stdout[-4000:], r.stderr[-4000:])
    return r.stdout


def test_selftest_reports_a_failed_check(debug_env):
    script = (
        "import torch, exact_io_aware_tcgen05_gb300 as fa\n"
        "assert fa.fa_debug_checks_enabled()\n"
        "s = torch.cuda.current_stream()\n"
        "fa.fa_debug_check_selftest(s)\n"
        "st = fa.fa_device_status(s, check=False)\n"
        "assert st == fa.FA_ERR_CUDA, st\n"
        "assert 'bounds-checking' in fa.fa_last_error(), fa.fa_last_error()\n"
        "assert fa.fa_device_status(s, check=False) == fa.FA_OK\n"
        "print('selftest ok')\n")
    assert "selftest ok" in _run([sys.executable, "-c", script], debug_env, 600)


def test_parity_suites_pass_with_bounds_checks(debug_env):
    env = dict(debug_env, FA_GB300_CHECK_STATUS="1")
    out = _run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                *[os.path.join("tests", s) for s in SUITES]], env, 3000)
    assert " passed" in out and "failed" not in out, out[-2000:]
