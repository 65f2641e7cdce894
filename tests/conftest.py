import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def q():
    """The binding, with the library built (in-tree) first."""
    from quantized_weight_prefill_q4_gb300.build import build_library

    build_library()
    import quantized_weight_prefill_q4_gb300 as pkg

    pkg.library()
    return pkg
