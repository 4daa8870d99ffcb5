import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


@pytest.fixture(autouse=True)
def _no_guard_refusals(request):
    """Against the guarded debug build (NVFP4_DEBUG_GUARDS=1), a GPU test
    fails if an index guard refused an access during it."""
    yield
    if os.environ.get("NVFP4_DEBUG_GUARDS", "0") in ("", "0") or request.node.get_closest_marker("gpu") is None:
        return
    import nvfp4_block_scaled_29_b300 as nv
    rec = nv.nvfp4_debug_guard_record()
    assert rec is None, f"an index guard refused an access: site {rec[0]}, byte offset {rec[1]}"


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def read_golden(path):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows
