import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def max_rel_err(got, ref) -> float:
    """Floored relative error: max_i |g_i - r_i| / max(|r_i|, 0.01 * rms(r)).

    The floor keeps elements that are tiny relative to the tensor's scale from dominating
    (in the spirit of the magnitude guard of the f64 gradchecks in gdn_backward.rs)."""
    g = np.asarray(got, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    assert g.shape == r.shape, (g.shape, r.shape)
    if r.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    floor = max(0.01 * rms, 1e-30)
    return float(np.max(np.abs(g - r) / np.maximum(np.abs(r), floor)))


@pytest.fixture
def rel_err():
    return max_rel_err
