"""The GPU parity cases of small and ragged shapes under the bounds-checked build (GPU).

compute-sanitizer is closed on this machine.  Besides the guard bands, the
library has a bounds-checked variant (libdfl_check.so, compiled with
-DDFL_CHECK): every index a kernel computes for a plain global store (GEMM
epilogues incl. the cache scatter, attention outputs and partials, the mix's
output rows) is checked against the extent the kernel's shape gives; one
outside it records DFL_ERR_BOUNDS in the device error word and the store is
skipped, nothing traps.  This test runs the operation, acceptance, cached and
small whole-step parity tests in a child process on that variant: they must
pass, and each test module ends by reading the error word, which must be 0.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_cases_pass_under_the_bounds_checked_build():
    from block_diffusion_speculative_dfl_gb300._build import LIB_CHECK, build
    assert build(checked=True) == LIB_CHECK
    env = dict(os.environ, DFL_CHECKED_BUILD="1")
    probe = subprocess.run([sys.executable, "-c", "import block_diffusion_speculative_dfl_gb300 as d; "
                            "print(d.load()._name)"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libdfl_check.so"), probe.stdout + probe.stderr
    files = ["tests/test_gpu_ops.py", "tests/test_gpu_accept_ext.py", "tests/test_gpu_cached.py",
             "tests/test_gpu_step.py"]
    r = subprocess.run([sys.executable, "-m", "pytest", *files, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
                        "-k", "not full_size"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
