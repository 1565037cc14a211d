"""End-to-end parity of the layer forward (C ABI) against the oracle.

Every float output is held to max|err| <= 1e-3 * rms(oracle); because the CUDA
path follows the oracle's F32 order wherever a float decides an integer, the
outputs are in fact expected bit-identical, which is asserted too.  Integer
intermediates (Q8_0 codes, router indices, hidden codes) are bit-exact."""
import numpy as np
import pytest
import torch

import synth
from helpers import OracleLayer, assert_float_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coli():
    import int4_routed_expert_f32_gb300 as c
    torch.cuda.set_device(0)
    return c


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _forward(coli, L, x, router_b=None):
    return coli.layer_forward(_cuda(x), L["router_w"], L["router_b"] if router_b is None else router_b,
                              L["expert_w4"], L["expert_rs"], L["shared_w4"], L["shared_rs"])


def _configure(coli, wl, max_tok):
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, max_tok)


# --------------------------------------------------------------------------- #
# tiny layer: full intermediates                                               #
# --------------------------------------------------------------------------- #
@pytest.fixture(scope="module")
def tiny(coli):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["tiny"]
    return wl, build_device_layer(wl), OracleLayer(wl)


@pytest.mark.parametrize("T", [4, 1, 3, 37])
def test_tiny_forward_and_intermediates(coli, tiny, T):
    wl, L, ref = tiny
    _configure(coli, wl, 64)
    x = synth.activations(wl, T, n_tok=T)
    r = coli.dbg_forward_intermediates(_cuda(x), L["router_w"], L["router_b"], L["expert_w4"],
                                       L["expert_rs"], L["shared_w4"], L["shared_rs"],
                                       wl.hidden, wl.ffn, wl.top_k)
    out, it = ref.forward(x, intermediates=True)
    assert coli.get_device_status() == coli.OK
    np.testing.assert_array_equal(r["qx"].cpu().numpy(), it["qx"])
    np.testing.assert_array_equal(r["dx"].cpu().numpy(), it["dx"])
    np.testing.assert_array_equal(r["idx"].cpu().numpy(), it["idx"])
    np.testing.assert_array_equal(r["w"].cpu().numpy(), it["w"])
    y = r["y"].cpu().numpy()
    P = T * wl.top_k
    np.testing.assert_array_equal(y[:P].reshape(T, wl.top_k, wl.hidden), it["y_routed"])
    np.testing.assert_array_equal(y[P:], it["y_shared"])
    got = r["out"].cpu().numpy()
    assert_float_close(got, out)
    np.testing.assert_array_equal(got, out)


def test_tiny_edge_cases(coli, tiny):
    wl, L, ref = tiny
    _configure(coli, wl, 8)
    empty = torch.empty((0, wl.hidden), dtype=torch.float32, device="cuda")
    coli.layer_forward(empty, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                       L["shared_w4"], L["shared_rs"])
    # n_tok above max_tok is an argument error, reported before any launch
    x = _cuda(synth.activations(wl, 0, n_tok=9))
    with pytest.raises(coli.ColiError) as ei:
        coli.layer_forward(x, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                           L["shared_w4"], L["shared_rs"])
    assert ei.value.code == coli.E_INVAL
    # exactly max_tok tokens
    x = synth.activations(wl, 5, n_tok=8)
    np.testing.assert_array_equal(_forward(coli, L, x).cpu().numpy(), ref.forward(x))
    # misaligned weights are rejected
    with pytest.raises(coli.ColiError):
        coli.layer_forward(_cuda(x), L["router_w"], L["router_b"], L["expert_w4"].view(-1)[1:],
                           L["expert_rs"], L["shared_w4"], L["shared_rs"])


def test_tiny_hostio_matches_device_call(coli, tiny):
    wl, L, ref = tiny
    _configure(coli, wl, 8)
    x = synth.activations(wl, 3, n_tok=4)
    xh = torch.from_numpy(x).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    coli.layer_forward_hostio(xh, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                              L["shared_w4"], L["shared_rs"], oh)
    np.testing.assert_array_equal(oh.numpy(), ref.forward(x))


def test_prepared_layer_matches_the_plain_calls(coli, tiny):
    """PreparedLayer marshals the weights once; its device and host-I/O
    forwards give the oracle's output bit for bit, over several inputs."""
    wl, L, ref = tiny
    _configure(coli, wl, 8)
    layer = coli.PreparedLayer(L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"], L["shared_w4"],
                               L["shared_rs"])
    oh = torch.empty((4, wl.hidden)).pin_memory()
    for step in range(3):
        x = synth.activations(wl, 70 + step, n_tok=4)
        want = ref.forward(x)
        np.testing.assert_array_equal(layer.forward(_cuda(x)).cpu().numpy(), want)
        layer.forward_hostio(torch.from_numpy(x).pin_memory(), oh)
        np.testing.assert_array_equal(oh.numpy(), want)
    assert coli.get_device_status() == coli.OK


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_hostio_pinned_and_pageable_outputs(coli, tiny, path):
    """Pinned (device-mapped) output buffers receive the combine's stores
    directly; pageable ones a copy of the device result.  Both must match the
    oracle bit for bit, over repeated calls with fresh inputs."""
    wl, L, ref = tiny
    _configure(coli, wl, 8)
    coli.set_path({"gemv": coli.PATH_GEMV, "gemm": coli.PATH_GEMM}[path])
    try:
        for step in range(3):
            x = synth.activations(wl, 40 + step, n_tok=5)
            want = ref.forward(x)
            xh = torch.from_numpy(x).pin_memory()
            for oh in (torch.full_like(xh, float("nan")).pin_memory(), torch.full((5, wl.hidden), float("nan"))):
                coli.layer_forward_hostio(xh, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                                          L["shared_w4"], L["shared_rs"], oh)
                np.testing.assert_array_equal(oh.numpy(), want)
            # a pageable input as well
            oh = torch.empty((5, wl.hidden)).pin_memory()
            coli.layer_forward_hostio(torch.from_numpy(x.copy()), L["router_w"], L["router_b"], L["expert_w4"],
                                      L["expert_rs"], L["shared_w4"], L["shared_rs"], oh)
            np.testing.assert_array_equal(oh.numpy(), want)
    finally:
        coli.set_path(coli.PATH_AUTO)
    assert coli.get_device_status() == coli.OK


# --------------------------------------------------------------------------- #
# GLM-5.2-shaped layer (256 experts + shared, all resident)                    #
# --------------------------------------------------------------------------- #
@pytest.fixture(scope="module")
def glm(coli, glm_expert_cache):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["decode"]
    return build_device_layer(wl), OracleLayer(wl, cache=glm_expert_cache)


def test_decode_batch1(coli, glm):
    L, ref = glm
    wl = synth.WORKLOADS["decode"]
    _configure(coli, wl, 2048)
    for step in range(3):
        x = synth.activations(wl, step)
        got = _forward(coli, L, x).cpu().numpy()
        want = ref.forward(x)
        assert_float_close(got, want)
        np.testing.assert_array_equal(got, want)
    assert coli.get_device_status() == coli.OK


def test_verify_batch4(coli, glm):
    L, ref = glm
    wl = synth.WORKLOADS["verify"]
    _configure(coli, wl, 2048)
    for step in range(2):
        x = synth.activations(wl, step)
        got = _forward(coli, L, x).cpu().numpy()
        want = ref.forward(x)
        assert_float_close(got, want)
        np.testing.assert_array_equal(got, want)


@pytest.fixture(scope="module")
def prefill_ref(glm, glm_expert_cache):
    """The oracle's whole 2048-token prefill forward (Zipf-skewed routing),
    with every pair's expert output: computed once for the module."""
    wl = synth.WORKLOADS["prefill"]
    ref = OracleLayer(wl, cache=glm_expert_cache)
    x = synth.activations(wl, 0)
    out, it = ref.forward(x, intermediates=True)
    return wl, ref, x, out, it


@pytest.mark.parametrize("path", ["auto", "gemv"])
def test_prefill_2048_every_token(coli, glm, prefill_ref, path):
    """Every one of the 2048 prefill tokens, bit for bit against the oracle:
    routing, each (token, expert) pair's output y (all routed pairs and every
    token of the shared expert, i.e. each of its 16 tiles of 128 tokens) and
    the combined output.  AUTO runs the grouped tensor-core GEMM at this size;
    the streaming GEMV path is checked on the same batch."""
    L, _ = glm
    wl, ref, x, want, it = prefill_ref
    _configure(coli, wl, 2048)
    assert coli.auto_uses_gemm(wl.n_tok, wl.top_k, wl.n_experts)
    coli.set_path(coli.PATH_AUTO if path == "auto" else coli.PATH_GEMV)
    try:
        r = coli.dbg_forward_intermediates(_cuda(x), L["router_w"], _cuda(ref.b), L["expert_w4"],
                                           L["expert_rs"], L["shared_w4"], L["shared_rs"],
                                           wl.hidden, wl.ffn, wl.top_k)
        assert coli.get_device_status() == coli.OK
    finally:
        coli.set_path(coli.PATH_AUTO)
    idx = r["idx"].cpu().numpy()
    np.testing.assert_array_equal(idx, it["idx"])
    np.testing.assert_array_equal(r["w"].cpu().numpy(), it["w"])
    counts = np.bincount(idx.ravel(), minlength=wl.n_experts)
    assert counts.max() >= 100, counts.max()          # the Zipf skew is in effect
    T, k, H = wl.n_tok, wl.top_k, wl.hidden
    y = r["y"].cpu().numpy()
    np.testing.assert_array_equal(y[:T * k].reshape(T, k, H), it["y_routed"])
    np.testing.assert_array_equal(y[T * k:], it["y_shared"])
    got = r["out"].cpu().numpy()
    assert_float_close(got, want)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_tiny_residual_forward(coli, tiny, path):
    """layer_forward_residual = x + the layer's output on RMSNorm(x), the add
    fused into the combine (one F32 add, as the stacked-layer sweep chains its
    layers)."""
    wl, L, ref = tiny
    _configure(coli, wl, 64)
    T = 37
    x = synth.activations(wl, 21, n_tok=T)
    coli.set_path(coli.PATH_GEMM if path == "gemm" else coli.PATH_GEMV)
    try:
        got = coli.layer_forward_residual(_cuda(x), L["router_w"], L["router_b"], L["expert_w4"],
                                          L["expert_rs"], L["shared_w4"], L["shared_rs"]).cpu().numpy()
    finally:
        coli.set_path(coli.PATH_AUTO)
    import oracle
    want = (x + ref.forward(oracle.rmsnorm(x))).astype(np.float32)
    np.testing.assert_array_equal(got, want)
