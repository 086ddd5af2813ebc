import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


def load_golden(name: str) -> dict:
    """Parse a ``key value value ...`` fixture; '#' starts a comment line."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


@pytest.fixture
def golden():
    return load_golden


def f32(vals) -> np.ndarray:
    return np.asarray([float(x) for x in vals], dtype=np.float32)


def ulp32(x) -> np.ndarray:
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(np.maximum(x, np.float32(np.finfo(np.float32).tiny)))


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree and loaded; GPU tests need a CUDA device."""
    import torch

    from gradient_compression_sgd_gb300 import build

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    import gradient_compression_sgd_gb300 as gc

    gc.lib()
    return gc


def rel_err(a, b) -> float:
    """max |a - b| / max(|b|, tiny) elementwise."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b) / np.maximum(np.abs(b), np.finfo(np.float32).tiny)))
