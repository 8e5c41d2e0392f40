import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built fp4idx library")
    config.addinivalue_line("markers", "slow: full-size workload parity (minutes)")


@pytest.fixture(scope="session")
def cos_sin():
    from sparse_attention_fp4_gb300 import workloads
    return workloads.rope_cos_sin_table()
