import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running test")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_fixture(name):
    """Data rows and '# key value' header entries of a golden fixture."""
    rows, meta = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line:
                continue
            if line.startswith("#"):
                parts = line[1:].strip().split()
                if len(parts) >= 2 and parts[0].endswith(":"):
                    meta[parts[0][:-1]] = parts[1:]
                elif len(parts) == 2 and parts[0].isidentifier():
                    meta[parts[0]] = parts[1:]
                continue
            rows.append(line.split())
    return rows, meta


@pytest.fixture
def fixture_reader():
    return read_fixture
