import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def expand(spec, n, default=0.0):
    """Expand {"i": v, "a..b": v} index maps into a dense list of length n."""
    out = [default] * n
    for key, v in spec.items():
        if ".." in key:
            a, b = key.split("..")
            for i in range(int(a), int(b) + 1):
                out[i] = v
        else:
            out[int(key)] = v
    return out
