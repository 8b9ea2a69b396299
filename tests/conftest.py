import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: longer CPU checks")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(autouse=True)
def _index_checks_clean(request):
    """Under the bounds-checking build (TP_B300_LIB=debug) every GPU test
    must also leave the library's index-check word at zero."""
    yield
    if os.environ.get("TP_B300_LIB") != "debug" or request.node.get_closest_marker("gpu") is None:
        return
    import backprojection_tp_project_gather_b300 as tp
    word = tp.tp_debug_bounds_word(reset=True)
    assert word == 0, f"index checks failed in {request.node.nodeid}: bits {word:#x}"
