import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the compiled library")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def device_gumbel_error():
    """max |G_device - G_exact| over 2^20 columns of three random streams:
    the device's uniforms are bit-exact, G_exact = -log(-log u) in binary64
    of those uniforms.  (GPU tests only.)"""
    import numpy as np
    import torch

    import verify_markov_head_gb300 as vm

    n = 1 << 20
    g = torch.empty(n, device="cuda")
    u = torch.empty(n, device="cuda")
    worst = 0.0
    for seed, step, dom, row in ((0, 0, 0, 0), (2, 0, 0, 7), (99, 3, 2, 1234)):
        vm.dspark_gumbel_stream(seed, step, dom, row, n, g, u)
        torch.cuda.synchronize()
        gu = u.cpu().double().numpy()
        worst = max(worst, float(np.abs(g.cpu().double().numpy() + np.log(-np.log(gu))).max()))
    return worst
