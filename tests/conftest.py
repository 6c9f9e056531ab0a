import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


def load_golden(name):
    """Parse a tests/golden fixture: '#' comments, 'key: value' lines; repeated keys concatenate."""
    fields = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            fields.setdefault(key.strip(), []).append(val.strip())
    return fields


def _golden_stream(name):
    import numpy as np

    g = load_golden(name)
    values = np.array([int(v, 16) for v in " ".join(g["values"]).split()], dtype=np.uint16)
    stream = np.frombuffer(bytes.fromhex("".join(g["stream"])), dtype=np.uint8)
    return int(g["e0"][0]), values, stream


@pytest.fixture(scope="session")
def golden_tiny():
    """Five values whose two escapes are kept as an exponent plane (3k > m)."""
    return _golden_stream("tiny_stream.txt")


@pytest.fixture(scope="session")
def golden_tiny_list():
    """Seven values whose two escapes are kept as a (position, exponent) list (3k <= m)."""
    return _golden_stream("tiny_list_stream.txt")
