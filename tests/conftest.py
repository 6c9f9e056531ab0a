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


def golden_stream(name):
    """(e0, values, stream) of a fixture.  'values' lists hex BF16 patterns, 'hex*count' for a run;
    the stream is 'length' bytes, zero except for the 'bytes OFFSET' lines (hex, spaces allowed)."""
    import numpy as np

    g = load_golden(name)
    vals = []
    for tok in " ".join(g["values"]).split():
        v, _, count = tok.partition("*")
        vals += [int(v, 16)] * (int(count) if count else 1)
    stream = np.zeros(int(g["length"][0]), dtype=np.uint8)
    for key, lines in g.items():
        if key.startswith("bytes "):
            off = int(key.split()[1])
            data = bytes.fromhex("".join(lines).replace(" ", ""))
            assert off + len(data) <= stream.size, (name, key)
            stream[off:off + len(data)] = np.frombuffer(data, np.uint8)
    return int(g["e0"][0]), np.array(vals, dtype=np.uint16), stream


@pytest.fixture(scope="session")
def golden_raw():
    """Five values stored in the raw form (their coded form would be longer)."""
    return golden_stream("tiny_raw_stream.txt")


@pytest.fixture(scope="session")
def golden_plane():
    """Two chunks (4096 + 5 values); chunk 1 keeps its two escapes as an exponent plane."""
    return golden_stream("two_chunk_plane_stream.txt")


@pytest.fixture(scope="session")
def golden_list():
    """Two chunks (4096 + 7 values); both keep their escapes as (position, exponent) lists."""
    return golden_stream("two_chunk_list_stream.txt")
