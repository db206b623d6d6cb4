import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(autouse=True)
def _debug_build_record_stays_clean(request):
    """Under MATTN_DEBUG=1 (the debug build, with device-side bounds checks)
    every GPU test must leave the checks' record empty."""
    yield
    if os.environ.get("MATTN_DEBUG", "0") in ("", "0") or "gpu" not in request.keywords:
        return
    import masked_attention_gb300 as M
    if M._lib is None:  # the test never loaded the library
        return
    rec = M.debug_record(clear=True)
    assert rec["count"] == 0, f"device bounds check failed: {rec}"
