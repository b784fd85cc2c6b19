import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: large CPU work (full-size oracle runs)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library through its Python binding; GPU tests only."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a GPU")
    import linear_attention_serving_kda_gb300 as kda

    kda.load()  # raises if the library is missing: no silent fallback
    return kda


@pytest.fixture(autouse=True)
def _name_parity_records(request):
    from tests import parity

    parity.CURRENT[0] = request.node.name
    yield


@pytest.fixture(autouse=True)
def _guard_regions(request):
    """After every GPU test: no guard region around a buffer the library
    wrote (outputs, states, verify logs, workspaces of every DeviceCase the
    test made) has changed -- the out-of-bounds check that stands in for a
    memory sanitizer."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch

    from linear_attention_serving_kda_gb300 import runtime

    torch.cuda.synchronize()
    bad = [dc.wl.name for dc in list(runtime.LIVE) if not dc.guards_intact()]
    runtime.LIVE.clear()
    assert not bad, f"guard bytes changed around a library buffer of: {bad}"


def pytest_terminal_summary(terminalreporter):
    try:
        from tests.parity import RECORD
    except Exception:
        return
    if RECORD:
        terminalreporter.write_line("parity record (what, rel L2, max-abs/RMS):")
        for what, e, m in RECORD:
            terminalreporter.write_line(f"  {what:70s} {e:.3e} {m:.3e}")
