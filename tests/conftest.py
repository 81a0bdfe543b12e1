import sys
from pathlib import Path

HERE = Path(__file__).resolve().parent
for p in (HERE, HERE.parent):
    if str(p) not in sys.path:
        sys.path.insert(0, str(p))


def pytest_sessionstart(session):
    """Build the library (and the C oracle) when a source is newer than the
    built file, so no test runs against a stale build."""
    from paged_kv_cache_kvcs_gb300 import build as lib_build
    from oracle import build as oracle_build
    lib_build.build()
    oracle_build.build()


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
