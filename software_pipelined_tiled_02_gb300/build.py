"""Build the CUDA library ``libtgemm.so`` in-tree for sm_103a (GB300).

One translation unit, one ``-gencode`` target, static CUDA runtime; the
result sits next to this file and is what the Python binding loads.
``build(debug=True)`` makes ``libtgemm_debug.so`` instead: the same kernel
with TGEMM_DEBUG_CHECKS=1, which checks every address it forms and reports
TGEMM_ERR_CHECK instead of touching memory outside its layout.  The tests
run a part of the parity suite against it (``TGEMM_LIB`` selects it).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libtgemm.so")
LIB_DEBUG = os.path.join(HERE, "libtgemm_debug.so")
SOURCES = [os.path.join(CSRC, "tgemm.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "layout.h")] + [os.path.join(INCLUDE, "tgemm.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtgemm.so")


def command(out: str = LIB, verbose_ptxas: bool = False, debug: bool = False) -> list[str]:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-o", out, *SOURCES]
    if debug:
        cmd.insert(1, "-DTGEMM_DEBUG_CHECKS=1")
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile ``libtgemm.so`` (or, with ``debug``, ``libtgemm_debug.so``)
    unless it is newer than every source."""
    lib = LIB_DEBUG if debug else LIB
    if not force and up_to_date(lib):
        return lib
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run(command(tmp, verbose_ptxas=verbose, debug=debug), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> list[str]:
    """Compile the release and the debug-check library side by side (two nvcc
    processes), skipping whichever is up to date."""
    jobs = []
    for debug, lib in ((False, LIB), (True, LIB_DEBUG)):
        if force or not up_to_date(lib):
            tmp = lib + f".{os.getpid()}.tmp"
            jobs.append((lib, tmp, subprocess.Popen(command(tmp, debug=debug), stdout=subprocess.PIPE,
                                                    stderr=subprocess.STDOUT, text=True)))
    errors = []
    for lib, tmp, proc in jobs:
        out, _ = proc.communicate()
        if proc.returncode != 0:
            errors.append(f"nvcc failed for {os.path.basename(lib)}:\n{out}")
        else:
            os.replace(tmp, lib)
    if errors:
        raise RuntimeError("\n".join(errors))
    return [LIB, LIB_DEBUG]


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
