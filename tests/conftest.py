import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes on the CPU side)")


def read_golden_kv(name):
    """Parse a `key = v1 v2 ...` fixture file into {key: [int, ...]}."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[key] = [int(v, 0) for v in val.split()]
    return out


def read_golden_unpack(name):
    """Parse `<kind> <hex word> -> <codes>` lines into [(kind, word, [codes])]."""
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            kind, word = lhs.split()
            out.append((kind, int(word, 16), [int(v) for v in rhs.split()]))
    return out
