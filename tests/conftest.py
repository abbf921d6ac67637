import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (parity and timing on the device)")


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


@pytest.fixture(scope="session", autouse=True)
def _built_libraries():
    """Build the oracle and the host input generator when missing or stale (gcc, seconds)."""
    import subprocess

    import oracle
    import pkv_inputs

    if not os.environ.get("PKV_ORACLE_LIB") and _stale(oracle.LIB, [os.path.join(ROOT, "oracle", "pkv_oracle.c")]):
        oracle.build()
    if _stale(pkv_inputs.HOST_LIB, [os.path.join(ROOT, "pkv_inputs", "hostgen.c")]):
        subprocess.run(pkv_inputs.build_commands()[0], check=True)
    yield


def cuda_available():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:
        return False
