import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkq.so")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


def load_golden(name):
    """Parse a tests/golden fixture: '# ...' comments, 'hex ..' byte lines, 'key v ...' lines."""
    path = os.path.join(ROOT, "tests", "golden", name)
    data, fields = bytearray(), {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "hex":
                data.extend(int(v, 16) for v in vals)
            else:
                fields[key] = [float(v) for v in vals]
    return bytes(data), fields
