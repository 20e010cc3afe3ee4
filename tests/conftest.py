import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs on a GB300)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def lmhead_full():
    """The fused LM-head workload (B=16, K=7, d=8192, V=128256, T=1) with its
    fp64 logits and their accumulation bound (oracle.gemm_bound), built once."""
    from oracle import gemm_bound
    from speculative_decoding_verification_11_gb300 import workloads
    b = workloads.lmhead()
    return b, gemm_bound.bands(b.hidden, b.w_vocab_t, b.temperature)
