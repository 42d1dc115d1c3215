import os
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parent.parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpagedkv.so")
    config.addinivalue_line("markers", "slow: large sizes (still part of the default run)")


@pytest.fixture(scope="session", autouse=True)
def _native_parts():
    """Build the oracle and the input generator (plain C; cheap, CPU only)."""
    import oracle
    from paged_kv_cache_11_gb300 import _build
    oracle.build()
    _build.build_generator()
    yield


def has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def gpu():
    """Skip-free guard: a test marked gpu fails loudly when no GPU or library is present."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("test marked gpu ran without a CUDA device")
    from paged_kv_cache_11_gb300 import _build
    _build.build_library()
    import paged_kv_cache_11_gb300 as pkv
    pkv.binding._lib()
    return torch.device("cuda:0")
