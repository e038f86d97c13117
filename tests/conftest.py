import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU oracle case")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.lib()


@pytest.fixture
def pin_gemm_path():
    """Pin the library's GEMM path for one test (a test hook of the C ABI); the
    choice by rows is restored afterwards."""
    import moe_gemm_exl3_gb300 as m
    yield m.exl3_set_gemm_path
    m.exl3_set_gemm_path("rows")
