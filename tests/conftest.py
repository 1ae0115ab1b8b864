import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    import paged_kv_cache_arena_gb300 as K
    K.kshipra_device_status()  # clear anything left over
    return K


@pytest.fixture
def clean_status(gpu):
    """Fails a test that leaves a device status bit set; resets options."""
    yield gpu
    code = gpu.kshipra_device_status()
    gpu.kshipra_set_option(gpu.KSHIPRA_OPT_SPLIT_TOKENS, 0)
    gpu.kshipra_set_option(gpu.KSHIPRA_OPT_DECODE_MAX_ROWS, 16)
    assert code == 0, "device status word 0x%x" % code


def pytest_terminal_summary(terminalreporter):
    """Achieved errors of the full-size workloads against the oracle."""
    try:
        from helpers import RECORDED, TOL
    except ImportError:
        return
    rows = [r for r in RECORDED if r[0].startswith("full ")]
    if not rows:
        return
    terminalreporter.write_sep("-", "attention vs float64 oracle, full-size workloads (every output row)")
    for what, dtype, max_abs, max_rel, n in rows:
        atol, rtol = TOL[dtype]
        terminalreporter.write_line("%-40s %-4s rows %5d  max abs %.3e (tol %.1e)  max rel %.3e (tol %.1e)" % (
            what, dtype, n, max_abs, atol, max_rel, rtol))
