"""Parity of the grouped tensor-core path (tcgen05 GEMM over the batch union of
all experts) against the oracle, and against the streaming GEMV path.

The GEMM computes each Q8_0 block's integer dot product exactly (int4 and int8
codes are exact in bf16, a block sum is exact in F32) and folds the blocks in
the oracle's order, so every output is expected bit-identical to the oracle
and to the GEMV path; the 1e-3 * rms bound is asserted as well."""
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
    yield c
    c.set_path(c.PATH_AUTO, 0)


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _intermediates(coli, wl, L, x):
    return coli.dbg_forward_intermediates(_cuda(x), L["router_w"], L["router_b"], L["expert_w4"],
                                          L["expert_rs"], L["shared_w4"], L["shared_rs"],
                                          wl.hidden, wl.ffn, wl.top_k)


@pytest.fixture(scope="module")
def tiny(coli):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["tiny"]
    return wl, build_device_layer(wl), OracleLayer(wl)


# T = 1 and 5 take the one-launch routing; 37 leaves most tiles ragged; 130 and
# 300 give experts (and the shared expert) more than one 128-row tile.
@pytest.mark.parametrize("T", [1, 5, 37, 130, 300])
def test_tiny_gemm_matches_oracle_and_gemv(coli, tiny, T):
    wl, L, ref = tiny
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 512)
    x = synth.activations(wl, 100 + T, n_tok=T)
    coli.set_path(coli.PATH_GEMM)
    r = _intermediates(coli, wl, L, x)
    assert coli.get_device_status() == coli.OK
    out, it = ref.forward(x, intermediates=True)
    P = T * wl.top_k
    y = r["y"].cpu().numpy()
    np.testing.assert_array_equal(r["idx"].cpu().numpy(), it["idx"])
    np.testing.assert_array_equal(y[:P].reshape(T, wl.top_k, wl.hidden), it["y_routed"])
    np.testing.assert_array_equal(y[P:], it["y_shared"])
    got = r["out"].cpu().numpy()
    assert_float_close(got, out)
    np.testing.assert_array_equal(got, out)
    # the streaming path gives the same hidden codes, expert outputs and result
    coli.set_path(coli.PATH_GEMV)
    v = _intermediates(coli, wl, L, x)
    coli.set_path(coli.PATH_AUTO)
    for key in ("qh", "dh", "y", "out"):
        np.testing.assert_array_equal(r[key].cpu().numpy(), v[key].cpu().numpy(), err_msg=key)


def test_tiny_gemm_zero_router_ties(coli, tiny):
    """An all-zero router makes every expert tie: the lowest indices win, so
    experts 0..k-1 get all T tokens (several tiles each) and the rest none."""
    wl, L, ref = tiny
    T = 260
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 512)
    x = synth.activations(wl, 7, n_tok=T)
    zw = torch.zeros_like(L["router_w"])
    zb = torch.zeros_like(L["router_b"])
    coli.set_path(coli.PATH_GEMM)
    got = coli.layer_forward(_cuda(x), zw, zb, L["expert_w4"], L["expert_rs"], L["shared_w4"],
                             L["shared_rs"]).cpu().numpy()
    coli.set_path(coli.PATH_AUTO)
    assert coli.get_device_status() == coli.OK
    import oracle
    w4 = [None] * wl.n_experts
    rs = [None] * wl.n_experts
    for e in range(wl.top_k):
        w4[e], rs[e] = ref.expert(e)
    want = oracle.moe_forward(x, np.zeros_like(ref.W), np.zeros_like(ref.b), w4, rs, ref.shared[0],
                              ref.shared[1], wl.hidden, wl.ffn, wl.top_k, wl.routed_scale)
    np.testing.assert_array_equal(got, want)


def test_tiny_gemm_hostio(coli, tiny):
    wl, L, ref = tiny
    T = 70
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 128)
    x = synth.activations(wl, 3, n_tok=T)
    coli.set_path(coli.PATH_GEMM)
    xh = torch.from_numpy(x).pin_memory()
    outh = torch.empty_like(xh).pin_memory()
    coli.layer_forward_hostio(xh, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                              L["shared_w4"], L["shared_rs"], outh)
    coli.set_path(coli.PATH_AUTO)
    np.testing.assert_array_equal(outh.numpy(), ref.forward(x))


# --------------------------------------------------------------------------- #
# GLM-5.2-shaped layer                                                         #
# --------------------------------------------------------------------------- #
@pytest.fixture(scope="module")
def glm(coli, glm_expert_cache):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["decode"]
    return build_device_layer(wl), OracleLayer(wl, cache=glm_expert_cache)


@pytest.mark.parametrize("T", [64, 200])
def test_glm_gemm_matches_gemv_and_oracle(coli, glm, T):
    L, ref = glm
    wl = synth.WORKLOADS["verify"]
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 2048)
    x = synth.activations(wl, 50 + T, n_tok=T)
    outs = {}
    for path in (coli.PATH_GEMM, coli.PATH_GEMV):
        coli.set_path(path)
        outs[path] = coli.layer_forward(_cuda(x), L["router_w"], L["router_b"], L["expert_w4"],
                                        L["expert_rs"], L["shared_w4"], L["shared_rs"]).cpu().numpy()
    coli.set_path(coli.PATH_AUTO)
    assert coli.get_device_status() == coli.OK
    np.testing.assert_array_equal(outs[coli.PATH_GEMM], outs[coli.PATH_GEMV])
    # every token against the oracle
    want = ref.forward(x)
    assert_float_close(outs[coli.PATH_GEMM], want)
    np.testing.assert_array_equal(outs[coli.PATH_GEMM], want)


def test_prefill_2048_gemm_matches_gemv(coli, glm):
    """The full prefill batch (2048 tokens, Zipf-skewed routing): every output
    of the tensor-core path equals the streaming path's."""
    L, _ = glm
    wl = synth.WORKLOADS["prefill"]
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 2048)
    _, b = synth.router(wl)
    bd = _cuda(b)
    x = _cuda(synth.activations(wl, 1))
    outs = {}
    for path in (coli.PATH_GEMM, coli.PATH_GEMV):
        coli.set_path(path)
        outs[path] = coli.layer_forward(x, L["router_w"], bd, L["expert_w4"], L["expert_rs"],
                                        L["shared_w4"], L["shared_rs"]).cpu().numpy()
    coli.set_path(coli.PATH_AUTO)
    assert coli.get_device_status() == coli.OK
    np.testing.assert_array_equal(outs[coli.PATH_GEMM], outs[coli.PATH_GEMV])
