"""The parity suite's small cases, run against the debug-check build.

compute-sanitizer is not available on this machine, so the kernel checks itself
instead.  ``libtgemm_debug.so`` is the same source compiled with
TGEMM_DEBUG_CHECKS=1.  Every shared-memory, tensor-memory and TMA address it
forms is tested against the plan's layout before use, and a failed check is
reported as TGEMM_ERR_CHECK instead of being carried out.  The tests below run
in a child process that loads that build (``TGEMM_LIB``).  There, each run's
status must be 0 and each result must match the oracle.
"""

import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_suite_passes_under_debug_checks(cuda_lib):
    from software_pipelined_tiled_02_gb300 import build

    lib = build.build(debug=True)
    env = dict(os.environ, TGEMM_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_random_sweep.py"),
                        os.path.join(ROOT, "tests", "test_gemm.py"),
                        os.path.join(ROOT, "tests", "test_watchdog.py"),
                        "-k", "random_sweep or small_shapes or pair_small or split_k_parity or integer or stall or cluster_split or multicast or "
                        "stream_k"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    passed = re.search(r"(\d+) passed", r.stdout)
    assert passed and int(passed.group(1)) >= 400, r.stdout[-2000:]


def test_debug_build_is_the_one_loaded():
    # The child processes above pick the library through TGEMM_LIB; check the
    # selection logic itself without a GPU.
    code = ("import os, software_pipelined_tiled_02_gb300 as tg; "
            "L = tg.load(); print(os.path.basename(L._name))")
    from software_pipelined_tiled_02_gb300 import build

    lib = build.build(debug=True)
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=dict(os.environ, TGEMM_LIB=lib),
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "libtgemm_debug.so"
