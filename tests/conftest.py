import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: 'key: v1 v2 ...' lines, '#' comments."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.split()
    return out


@pytest.fixture
def golden():
    return load_golden


def _lib_stale() -> bool:
    from bit_weight_only_lbq_gb300 import build as B
    if not os.path.exists(B.LIB):
        return True
    t = os.path.getmtime(B.LIB)
    srcs = [os.path.join(B.CSRC, f) for f in os.listdir(B.CSRC)] + [os.path.join(B.INCLUDE, "lbq.h")]
    return any(os.path.getmtime(s) > t for s in srcs)


@pytest.fixture(scope="session")
def lbq():
    """The binding, with liblbq.so built in-tree if missing or older than its sources."""
    if _lib_stale():
        from bit_weight_only_lbq_gb300 import build as B
        B.build()
    from bit_weight_only_lbq_gb300 import lbq as L
    L.lib()
    return L
