"""The host-memory expert tier: routed experts in (page-locked) host memory,
an LRU cache of them in HBM slots, the same kernels reading the slots.  Every
forward must equal the oracle bit for bit whether its experts were resident
or copied in, and the cache's bookkeeping must follow the LRU rule."""
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
    c.tier_release()
    c.set_path(c.PATH_AUTO, 0)


def _host(L):
    return L["expert_w4"].cpu().pin_memory(), L["expert_rs"].cpu().pin_memory()


def _fwd(coli, L, hw, hrs, x):
    return coli.tier_forward(torch.from_numpy(np.ascontiguousarray(x)).cuda(), L["router_w"], L["router_b"], hw,
                             hrs, L["shared_w4"], L["shared_rs"]).cpu().numpy()


@pytest.fixture(scope="module")
def tiny(coli):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["tiny"]
    L = build_device_layer(wl)
    return wl, L, _host(L), OracleLayer(wl)


def test_tier_decode_evicts_and_stays_bit_exact(coli, tiny, orc):
    """Three slots for eight experts, one token (two experts) per forward:
    forwards copy in the experts they miss, evicting least recently used
    ones; every output equals the oracle; hits + misses count every chosen
    expert; an expert chosen by the previous forward is still resident (with
    three slots and two experts a forward, nothing the previous forward used
    can be the least recently used)."""
    wl, L, (hw, hrs), ref = tiny
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 8)
    coli.tier_configure(3)
    total = 0
    prev = set()
    last = (0, 0)
    for step in range(12):
        x = synth.activations(wl, 1000 + step, n_tok=1)
        np.testing.assert_array_equal(_fwd(coli, L, hw, hrs, x), ref.forward(x))
        idx, _ = orc.route(x, ref.W, ref.b, wl.top_k, wl.routed_scale)
        chosen = set(int(e) for e in idx.ravel())
        total += len(chosen)
        h, m, b, r = coli.tier_stats()
        assert h + m == total
        assert r <= 3
        assert b == m * (wl.expert_bytes + 4 * wl.expert_scales)
        # an expert of the previous forward that is chosen again is a hit
        assert h - last[0] >= len(chosen & prev)
        last, prev = (h, m), chosen
    assert m > 3 and h > 0                             # the cache both hit and evicted
    assert coli.get_device_status() == coli.OK


def test_tier_refuses_a_union_larger_than_its_slots(coli, tiny):
    wl, L, (hw, hrs), ref = tiny
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 16)
    coli.tier_configure(2)
    x = synth.activations(wl, 5, n_tok=16)            # 16 tokens choose more than two experts
    with pytest.raises(coli.ColiError) as ei:
        _fwd(coli, L, hw, hrs, x)
    assert ei.value.code == coli.E_INVAL
    coli.tier_configure(wl.n_experts)
    np.testing.assert_array_equal(_fwd(coli, L, hw, hrs, x), ref.forward(x))


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_tier_batches_on_both_paths(coli, tiny, path):
    wl, L, (hw, hrs), ref = tiny
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 300)
    coli.tier_configure(wl.n_experts)
    coli.set_path(coli.PATH_GEMV if path == "gemv" else coli.PATH_GEMM)
    try:
        for T in (5, 300):
            x = synth.activations(wl, 2000 + T, n_tok=T)
            np.testing.assert_array_equal(_fwd(coli, L, hw, hrs, x), ref.forward(x))
    finally:
        coli.set_path(coli.PATH_AUTO)


def test_tier_glm_decode(coli, glm_expert_cache):
    """The GLM-5.2-shaped layer with its 256 routed experts (4.9 GB) in host
    memory and 32 HBM slots (a 4-token forward chooses up to 32 experts):
    decode and 4-token forwards, bit-exact."""
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["decode"]
    L = build_device_layer(wl)
    hw, hrs = _host(L)
    L["expert_w4"] = None                               # the tier reads the host copy only
    torch.cuda.empty_cache()
    ref = OracleLayer(wl, cache=glm_expert_cache)
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 4)
    coli.tier_configure(32)
    for step, T in enumerate((1, 1, 4, 1)):
        x = synth.activations(wl, 3000 + step, n_tok=T)
        got = coli.tier_forward(torch.from_numpy(x).cuda(), L["router_w"], L["router_b"], hw, hrs, L["shared_w4"],
                                L["shared_rs"]).cpu().numpy()
        np.testing.assert_array_equal(got, ref.forward(x))
    h, m, b, r = coli.tier_stats()
    assert m > 0 and r <= 32
    assert coli.get_device_status() == coli.OK
    coli.tier_release()
