import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_sessionstart(session):
    """Bring the in-tree library up to date with its sources before any test loads it
    (a no-op when the build stamp matches; tests that need the library report a clear
    error if it cannot be built here)."""
    try:
        from block_quantized_token_format_gb300 import build as _build
        _build.build()
    except Exception as e:  # noqa: BLE001 - reported by the tests that need the library
        sys.stderr.write(f"conftest: library build skipped: {e}\n")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
