import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """After every GPU test that loaded the library, the device status
    record must be clear: no bounded wait ran out and (in the debug build)
    no bounds check failed.  Tests that provoke a record read it themselves."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    cpa = sys.modules.get("context_long_sequence_gb300")
    if cpa is None or getattr(cpa, "_lib", None) is None:
        return
    code, block, line, file_id = cpa.cp_get_status_detail()
    assert code == 0, (f"device status {code} ({cpa.cp_strerror(code)}): block {block}, "
                       f"line {line}, file id {file_id}")
