import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workloads")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def golden():
    """Reads a fixture from tests/golden (lines of `key: ints`, `#` comments)."""
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

    def load(name):
        out = {}
        with open(os.path.join(here, name)) as fh:
            for line in fh:
                line = line.strip()
                if not line or line.startswith("#"):
                    continue
                key, _, value = line.partition(":")
                out[key.strip()] = [int(x) for x in value.split()]
        return out

    return load
