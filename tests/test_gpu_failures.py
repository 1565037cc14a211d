"""Failure detection without a GPU fault: each failure is injected on the host
(a workspace allocation that fails, a launch reported as failed) or is a
device-side wait with a short bound that the test makes run out.  Each test
checks that the failure comes back as its status, and that the next normal
forward is bit-exact against the oracle (the library recovered: counters
reset, workspace intact)."""
import numpy as np
import pytest
import torch

import synth
from helpers import OracleLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coli():
    import int4_routed_expert_f32_gb300 as c
    torch.cuda.set_device(0)
    yield c
    c.dbg_inject(c.INJECT_NONE)
    c.set_path(c.PATH_AUTO, 0)


@pytest.fixture(scope="module")
def tiny(coli):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["tiny"]
    return wl, build_device_layer(wl), OracleLayer(wl)


def _fwd(coli, L, x):
    return coli.layer_forward(torch.from_numpy(x).cuda(), L["router_w"], L["router_b"], L["expert_w4"],
                              L["expert_rs"], L["shared_w4"], L["shared_rs"]).cpu().numpy()


def _configure(coli, wl, T=64):
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, T)


def test_bounded_wait_runs_out_and_reports_timeout(coli, tiny):
    """Every down unit of one streaming forward waits for a gate/up count its
    tile never reaches, with a 20 us bound: the launch returns, the device
    status says COLI_E_TIMEOUT, and the next forward is bit-exact."""
    wl, L, ref = tiny
    _configure(coli, wl)
    coli.set_path(coli.PATH_GEMV)
    try:
        x = synth.activations(wl, 61, n_tok=4)
        coli.dbg_inject(coli.INJECT_WAIT_TIMEOUT, 20)
        _fwd(coli, L, x)                                  # returns: every wait is bounded
        assert coli.get_device_status() == coli.E_TIMEOUT
        assert coli.get_device_status() == coli.OK        # read and cleared
        for step in range(2):
            x = synth.activations(wl, 62 + step, n_tok=4)
            np.testing.assert_array_equal(_fwd(coli, L, x), ref.forward(x))
            assert coli.get_device_status() == coli.OK
    finally:
        coli.set_path(coli.PATH_AUTO)


def test_workspace_allocation_failure_reports_nomem(coli, tiny):
    """A workspace allocation that fails gives COLI_E_NOMEM and leaves the
    library unconfigured (COLI_E_NOSHAPE); a later configure succeeds and the
    forward is bit-exact."""
    wl, L, ref = tiny
    coli.dbg_inject(coli.INJECT_ALLOC_FAIL, 1)
    with pytest.raises(coli.ColiError) as ei:
        _configure(coli, wl)
    assert ei.value.code == coli.E_NOMEM
    x = synth.activations(wl, 71, n_tok=4)
    with pytest.raises(coli.ColiError) as ei:
        _fwd(coli, L, x)
    assert ei.value.code == coli.E_NOSHAPE
    _configure(coli, wl)
    np.testing.assert_array_equal(_fwd(coli, L, x), ref.forward(x))
    assert coli.get_device_status() == coli.OK


@pytest.mark.parametrize("path,T,nth", [("gemv", 4, 1), ("gemv", 4, 2), ("gemv", 20, 3),
                                         ("gemm", 20, 1), ("gemm", 20, 6), ("gemm", 20, 9)])
def test_launch_failure_reports_cuda_error(coli, tiny, path, T, nth):
    """The nth launch of a forward (routing, gather, GEMMs, combine) reported
    as failed: the call returns COLI_E_CUDA, and the next forward on the same
    workspace is bit-exact."""
    wl, L, ref = tiny
    _configure(coli, wl)
    coli.set_path(coli.PATH_GEMV if path == "gemv" else coli.PATH_GEMM)
    try:
        x = synth.activations(wl, 80 + nth, n_tok=T)
        coli.dbg_inject(coli.INJECT_LAUNCH_FAIL, nth)
        with pytest.raises(coli.ColiError) as ei:
            _fwd(coli, L, x)
        assert ei.value.code == coli.E_CUDA
        coli.dbg_inject(coli.INJECT_NONE)
        assert coli.get_device_status() == coli.OK
        np.testing.assert_array_equal(_fwd(coli, L, x), ref.forward(x))
        assert coli.get_device_status() == coli.OK
    finally:
        coli.dbg_inject(coli.INJECT_NONE)
        coli.set_path(coli.PATH_AUTO)


def test_workspace_guard_change_is_reported(coli, tiny):
    """The guard regions between the workspace's buffers (the bounds check
    every GPU test ends with) report a changed byte: guard regions changed from
    the host, as a stray device write past a buffer would change them, are
    counted and restored, and the next forward is bit-exact."""
    wl, L, ref = tiny
    _configure(coli, wl, 8)
    x = synth.activations(wl, 71, n_tok=8)
    np.testing.assert_array_equal(_fwd(coli, L, x), ref.forward(x))
    changed, total = coli.dbg_check_guards()
    assert changed == 0 and total >= 30
    for k in (0, total // 2, total - 1):
        coli.dbg_inject(coli.INJECT_GUARD, k)
        assert coli.dbg_check_guards() == (1, total)
        assert coli.dbg_check_guards() == (0, total)       # restored
    coli.dbg_inject(coli.INJECT_GUARD, 1)
    coli.dbg_inject(coli.INJECT_GUARD, 2)
    assert coli.dbg_check_guards() == (2, total)
    with pytest.raises(coli.ColiError):
        coli.dbg_inject(coli.INJECT_GUARD, total)
    np.testing.assert_array_equal(_fwd(coli, L, x), ref.forward(x))
