"""The int8-weight experts (the int8 container: one two's-complement code per
weight, s = max|row| / 127) through the same layer: the device packer, the
int8 block dots, and whole forwards against the oracle's int8 path, bit for
bit, on both expert paths.  The pages name an int8 container to which the int4 packing decodes
bit-identically, and an int8 MTP head ("colibri: a pure-C inference engine
..." (discuss.pytorch.kr), section "Key features"; "Open-source engine that
ran 744B GLM-5.2 ..." (jeff.news), section "MTP is sensitive"): the last test
checks that claim on the device path, int4 codes widened into the int8
container giving the int4 path's outputs bit for bit."""
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
    c.set_weight_bits(4)
    c.set_path(c.PATH_AUTO, 0)


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("rows,K", [(7, 256), (64, 6144), (300, 2048)])
def test_pack_int8_bitexact(coli, orc, rows, K):
    g = np.random.default_rng(rows + 5)
    w = (g.standard_normal((rows, K)) * 0.02).astype(np.float32)
    w[0] = 0.0
    w[-1, 3] = 0.5
    w[1, ::5] = np.float32(0.02) * 126.5 / 127.0     # near-half-way codes after /s
    q, s = coli.pack_int8(_cuda(w))
    rq, rs = orc.pack_int8_rows(w)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_block_dots_w8_bitexact(coli, orc):
    g = np.random.default_rng(2)
    K = 6144
    w8 = g.integers(-127, 128, (97, K)).astype(np.int8)
    w8[0] = -127
    w8[1] = 127
    q = g.integers(-127, 128, K).astype(np.int8)
    q[:64] = -127
    I = coli.dbg_block_dots_w8(_cuda(w8), _cuda(q))
    np.testing.assert_array_equal(I.cpu().numpy(), orc.block_dots_w8(w8, q))


def _forward(coli, wl, L, x, router_b=None):
    coli.set_weight_bits(8)
    try:
        return coli.layer_forward(_cuda(x), L["router_w"], L["router_b"] if router_b is None else router_b,
                                  L["expert_w4"], L["expert_rs"], L["shared_w4"], L["shared_rs"]).cpu().numpy()
    finally:
        coli.set_weight_bits(4)


@pytest.fixture(scope="module")
def tiny8(coli):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["tiny"]
    return wl, build_device_layer(wl, wbits=8), OracleLayer(wl, wbits=8)


@pytest.mark.parametrize("T", [1, 4, 37, 300])
def test_tiny_int8_forward(coli, tiny8, T):
    wl, L, ref = tiny8
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 512)
    x = synth.activations(wl, 500 + T, n_tok=T)
    coli.set_weight_bits(8)
    try:
        r = coli.dbg_forward_intermediates(_cuda(x), L["router_w"], L["router_b"], L["expert_w4"],
                                           L["expert_rs"], L["shared_w4"], L["shared_rs"],
                                           wl.hidden, wl.ffn, wl.top_k)
    finally:
        coli.set_weight_bits(4)
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


@pytest.mark.parametrize("T", [1, 37, 300])
def test_tiny_int8_gemm(coli, tiny8, T):
    """The grouped tensor-core GEMM on int8-container weights (int8 codes
    converted to bf16 operands): bit-exact against the oracle and equal to the
    streaming path, at item sizes from one token to several 128-token items."""
    wl, L, ref = tiny8
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 512)
    x = synth.activations(wl, 700 + T, n_tok=T)
    outs = {}
    for path in (coli.PATH_GEMM, coli.PATH_GEMV):
        coli.set_path(path)
        try:
            outs[path] = _forward(coli, wl, L, x)
        finally:
            coli.set_path(coli.PATH_AUTO)
    assert coli.get_device_status() == coli.OK
    want = ref.forward(x)
    np.testing.assert_array_equal(outs[coli.PATH_GEMM], want)
    np.testing.assert_array_equal(outs[coli.PATH_GEMV], want)


@pytest.fixture(scope="module")
def glm8(coli):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["decode"]
    L = build_device_layer(wl, wbits=8)
    yield L, OracleLayer(wl, wbits=8)
    del L
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,T,path", [("decode", 1, "auto"), ("verify", 4, "auto"), ("verify", 64, "auto"),
                                         ("verify", 200, "gemm")])
def test_glm_int8_forward(coli, glm8, name, T, path):
    """The GLM-5.2-shaped layer with int8 experts (about 9.7 GB resident):
    every token bit-exact against the oracle, on the streaming path and on
    the grouped GEMM."""
    L, ref = glm8
    wl = synth.WORKLOADS[name]
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 256)
    coli.set_path(coli.PATH_GEMM if path == "gemm" else coli.PATH_AUTO)
    try:
        for step in range(2 if T < 64 else 1):
            x = synth.activations(wl, 600 + step, n_tok=T)
            got = _forward(coli, wl, L, x)
            want = ref.forward(x)
            assert_float_close(got, want)
            np.testing.assert_array_equal(got, want)
    finally:
        coli.set_path(coli.PATH_AUTO)
    assert coli.get_device_status() == coli.OK


@pytest.mark.parametrize("T", [1, 4, 37])
def test_int4_codes_in_the_int8_container_give_identical_bits(coli, T):
    """The pages' claim, on the device: an int4 layer's codes widened into
    the int8 container (code = nibble - 8, same row scales) give the int4
    path's hidden codes, expert outputs and layer output bit for bit."""
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["tiny"]
    L4 = build_device_layer(wl)

    def widen(w4):
        b = w4.to(torch.int16)
        lo, hi = (b & 15) - 8, (b >> 4) - 8
        return torch.stack([lo, hi], dim=-1).reshape(*w4.shape[:-1], 2 * w4.shape[-1]).to(torch.int8) \
            .view(torch.uint8).contiguous()

    L8 = dict(L4, expert_w4=widen(L4["expert_w4"]), shared_w4=widen(L4["shared_w4"]))
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 64)
    x = synth.activations(wl, 900 + T, n_tok=T)
    r = {}
    for bits, L in ((4, L4), (8, L8)):
        coli.set_weight_bits(bits)
        try:
            r[bits] = coli.dbg_forward_intermediates(_cuda(x), L["router_w"], L["router_b"], L["expert_w4"],
                                                     L["expert_rs"], L["shared_w4"], L["shared_rs"],
                                                     wl.hidden, wl.ffn, wl.top_k)
        finally:
            coli.set_weight_bits(4)
    for key in ("qh", "dh", "y", "out"):
        np.testing.assert_array_equal(r[4][key].cpu().numpy(), r[8][key].cpu().numpy(), err_msg=key)
