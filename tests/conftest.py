import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    from oracle import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def oracle_act(oracle_mod):
    """Memoised (gate_up, oracle act) of a named workload, as bfloat16 bit
    patterns: the oracle's SwiGLU of the full batch is computed once per
    session and shared by every test that compares against it."""
    cache = {}

    def get(name):
        if name not in cache:
            from memory_bound_moe_gb300.workloads import WORKLOADS, as_u16, generate
            gu = as_u16(generate(WORKLOADS[name], seed=0, parts=("gate_up",))["gate_up"])
            cache[name] = (gu, oracle_mod.swiglu(gu))
        return cache[name]

    return get
