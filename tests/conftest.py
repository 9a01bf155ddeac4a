import math
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload")


def eval_expr(s: str) -> float:
    """Evaluate a fixture expression such as '3*sqrt(2)/5' or '1 + 2^-8' in double
    precision (the powers of two used by the fixtures are exact)."""
    return float(eval(s.replace("^", "**"), {"__builtins__": {}}, {"sqrt": math.sqrt}))


@pytest.fixture(scope="session")
def golden_dir():
    return GOLDEN


@pytest.fixture
def debug_env(monkeypatch):
    """Set or clear the library's debug knobs (RMSNORM_FORCE_VARIANT,
    RMSNORM_WAIT_LIMIT_CYCLES, RMSNORM_NO_PDL) for one test.  The library reads
    them once, so every change is followed by a reload, and the test's own
    environment is restored and reloaded when it ends."""
    import row_wise_normalization_02_gb300 as rn

    class _Env:
        def set(self, name, value):
            monkeypatch.setenv(name, value)
            rn.rmsnorm_reload_debug_env()

        def delete(self, name, raising=True):
            monkeypatch.delenv(name, raising=raising)
            rn.rmsnorm_reload_debug_env()

    yield _Env()
    monkeypatch.undo()
    rn.rmsnorm_reload_debug_env()
