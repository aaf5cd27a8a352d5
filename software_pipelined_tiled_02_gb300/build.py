"""Build the CUDA library ``libtgemm.so`` in-tree for sm_103a (GB300).

One translation unit, one ``-gencode`` target, static CUDA runtime; the
result sits next to this file and is what the Python binding loads.
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
SOURCES = [os.path.join(CSRC, "tgemm.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("ptx.cuh", "layout.h")] + [os.path.join(INCLUDE, "tgemm.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtgemm.so")


def command(out: str = LIB, verbose_ptxas: bool = False) -> list[str]:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-o", out, *SOURCES]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libtgemm.so`` unless it is newer than every source."""
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    r = subprocess.run(command(tmp, verbose_ptxas=verbose), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + r.stdout + r.stderr)
    if verbose:
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
