import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
# The mutation test runs the oracle pins against a deliberately broken copy of
# the oracle package placed in another directory; that directory comes first.
if os.environ.get("ORACLE_PKG_ROOT"):
    sys.path.insert(0, os.environ["ORACLE_PKG_ROOT"])

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


def golden_lines(name):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def hand_cases():
    cases, cur = [], None
    for t in golden_lines("gemm_hand_cases.txt"):
        if t[0] == "case":
            cur = dict(name=t[1], M=int(t[2]), N=int(t[3]), K=int(t[4]), A=[], B=[], C=[], S=[])
            cases.append(cur)
        else:
            cur[t[0]].append([float(v) for v in t[1:]])
    return cases


@pytest.fixture(scope="session")
def cuda_lib():
    """The built product library, on a machine with a GPU."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import software_pipelined_tiled_02_gb300 as tg

    tg.load()
    return tg
