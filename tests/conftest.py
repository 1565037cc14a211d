import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(autouse=True)
def _workspace_guards_intact(request):
    """After every GPU test: no kernel wrote past the end of a buffer of the
    library's workspace (its guard regions are unchanged).  The bounds check
    that stands in for a memory sanitizer on every GPU test."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    coli = sys.modules.get("int4_routed_expert_f32_gb300")
    if coli is None:
        return
    try:
        changed, total = coli.dbg_check_guards()
    except coli.ColiError:
        return          # not configured (released, or a failed configure under test)
    assert changed == 0, f"{changed} of {total} workspace guard regions changed: a write past a buffer's end"


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def golden_path(name: str) -> str:
    return os.path.join(ROOT, "tests", "golden", name)


@pytest.fixture(scope="session")
def glm_expert_cache():
    """Oracle-packed experts of the GLM-5.2-shaped layer (weight seed 1),
    shared by every test module that checks the decode, verify or prefill
    workloads (about 4.9 GB of host memory once all are packed)."""
    return {}
