import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running (full-size workload sample)")


def golden_path(name: str) -> str:
    return os.path.join(GOLDEN, name)


def read_table(name: str):
    rows = []
    with open(golden_path(name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle._load()
    return oracle


@pytest.fixture(scope="session")
def synth_mod():
    import synth

    synth._load_host()
    return synth
