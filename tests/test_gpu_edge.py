"""Edge cases of the layer, through both expert paths, against the oracle.

Extreme and odd shapes (the smallest hidden size, a single expert, top-1,
top-k equal to the expert count, the largest hidden and FFN sizes the ABI
accepts, an expert count that is not a power of two, a batch of 1000 tokens),
and degenerate inputs: an all-zero batch, logits large enough to saturate the
sigmoid in both directions, and experts with all-zero weight rows (row scale
0) or a single non-zero weight per row.  Every output is compared bit for bit
(the 1e-3 * rms bound is implied)."""
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
    c.set_path(c.PATH_AUTO, 0)


def _path(coli, name):
    return {"gemv": coli.PATH_GEMV, "gemm": coli.PATH_GEMM}[name]


def _run(coli, path, wl, L, x, max_tok=None):
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, max_tok or x.shape[0])
    coli.set_path(_path(coli, path))
    try:
        out = coli.layer_forward(torch.from_numpy(np.ascontiguousarray(x)).cuda(), L["router_w"],
                                 L["router_b"], L["expert_w4"], L["expert_rs"], L["shared_w4"],
                                 L["shared_rs"]).cpu().numpy()
        status = coli.get_device_status()
    finally:
        coli.set_path(coli.PATH_AUTO)
    assert status == coli.OK
    return out


# name, hidden, ffn, experts, top_k, tokens
SHAPES = [
    ("min_hidden_single_expert", 128, 128, 1, 1, 5),
    ("top1", 256, 128, 8, 1, 9),
    ("topk_equals_E", 384, 128, 16, 16, 7),
    ("odd_E", 256, 256, 5, 3, 33),
    ("max_hidden", 16384, 128, 4, 2, 3),
    ("max_ffn", 128, 16384, 4, 2, 3),
    ("many_tokens", 256, 128, 8, 2, 1000),
    # one token: the single-token routing tail (warp sorts of 64-bit key
    # images, a rank among the warps' candidates, one dispatch phase)
    ("t1_odd_E", 256, 128, 5, 3, 1),
    ("t1_k16", 256, 128, 40, 16, 1),
    ("t1_E256", 256, 128, 256, 8, 1),
    # one token with more gate/up units (17 tiles x 32) than expert-kernel
    # blocks, so that units are claimed in a second wave (even and odd stage
    # counts per row)
    ("t1_split_even", 1024, 1024, 32, 16, 1),
    ("t1_split_odd", 768, 1024, 32, 16, 1),
]


@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("shape", SHAPES, ids=[s[0] for s in SHAPES])
def test_shapes(coli, shape, path):
    from synth.device import build_device_layer
    name, H, F, E, k, T = shape
    wl = synth.Workload(name, H, F, E, k, T, 700 + len(name))
    L = build_device_layer(wl)
    x = synth.activations(wl, 1)
    got = _run(coli, path, wl, L, x)
    want = OracleLayer(wl).forward(x)
    np.testing.assert_array_equal(got, want)


# --------------------------------------------------------------------------- #
# degenerate inputs on the tiny layer                                          #
# --------------------------------------------------------------------------- #
@pytest.fixture(scope="module")
def tiny(coli):
    from synth.device import build_device_layer
    wl = synth.WORKLOADS["tiny"]
    return wl, build_device_layer(wl), OracleLayer(wl)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_zero_batch(coli, tiny, path):
    """x = 0: every Q8_0 scale is 0, every logit 0 (sigma 0.5, selection by
    the bias alone, weights 2.5/k), every expert output 0."""
    wl, L, ref = tiny
    x = np.zeros((6, wl.hidden), np.float32)
    got = _run(coli, path, wl, L, x)
    want = ref.forward(x)
    np.testing.assert_array_equal(got, want)
    assert not np.any(got)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_saturated_router(coli, tiny, path):
    """Inputs scaled so that router logits pass +-88: sigma saturates to 0 and
    1 exactly on both sides, and the selection falls back on the bias and the
    lowest-index rule among the saturated experts."""
    wl, L, ref = tiny
    x = (synth.activations(wl, 3, n_tok=8) * np.float32(2000.0)).astype(np.float32)
    import oracle
    _, _, logits, sigma = oracle.route(x, ref.W, ref.b, wl.top_k, wl.routed_scale, want_logits=True)
    assert np.any(sigma == 1.0) and np.any(sigma == 0.0)      # the case is exercised
    got = _run(coli, path, wl, L, x)
    want = ref.forward(x)
    np.testing.assert_array_equal(got, want)


def _custom_layer(coli, wl, flats):
    """Device and oracle layers packed from the given F32 expert weights
    (flats[e] = gate | up | down, E routed + 1 shared), each side with its own
    converter."""
    import oracle
    H, F, E = wl.hidden, wl.ffn, wl.n_experts
    W, b = synth.router(wl)
    L = dict(router_w=torch.from_numpy(W).cuda(), router_b=torch.from_numpy(b).cuda(),
             expert_w4=torch.zeros((E, wl.expert_bytes), dtype=torch.uint8, device="cuda"),
             expert_rs=torch.zeros((E, 2 * F + H), dtype=torch.float32, device="cuda"),
             shared_w4=torch.zeros((wl.expert_bytes,), dtype=torch.uint8, device="cuda"),
             shared_rs=torch.zeros((2 * F + H,), dtype=torch.float32, device="cuda"))
    mats = ((0, F, H), (F * H, F, H), (2 * F * H, H, F))
    w4s, rss = [], []
    for e, flat in enumerate(flats):
        dev_w4 = L["shared_w4"] if e == E else L["expert_w4"][e]
        dev_rs = L["shared_rs"] if e == E else L["expert_rs"][e]
        o4, ors, w4off, rsoff = [], [], 0, 0
        for off, rows, K in mats:
            m = np.ascontiguousarray(flat[off:off + rows * K].reshape(rows, K))
            coli.pack_int4(torch.from_numpy(m).cuda(), dev_w4[w4off:w4off + rows * K // 2].view(rows, K // 2),
                           dev_rs[rsoff:rsoff + rows])
            p, s = oracle.pack_int4_rows(m)
            o4.append(p.ravel())
            ors.append(s)
            w4off += rows * K // 2
            rsoff += rows
        w4s.append(np.concatenate(o4))
        rss.append(np.concatenate(ors))
    torch.cuda.synchronize()
    return L, (W, b, w4s, rss)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_zero_and_one_hot_weight_rows(coli, path):
    """Rows of all-zero weights (row scale 0, codes 0) and rows with a single
    non-zero weight (which maps to +-7), in the gate, up and down matrices of
    every routed expert and of the shared expert; a zero router makes the
    bias alone pick the experts."""
    import oracle
    wl = synth.WORKLOADS["tiny"]
    H, F, E = wl.hidden, wl.ffn, wl.n_experts
    rng = np.random.default_rng(31)
    flats = [synth.expert_f32_rows(wl, e).copy() for e in range(E + 1)]
    for e in range(E + 1):
        f = flats[e]
        gate = f[:F * H].reshape(F, H)
        up = f[F * H:2 * F * H].reshape(F, H)
        down = f[2 * F * H:].reshape(H, F)
        for r in rng.choice(F, 9, replace=False):
            gate[r] = 0.0
        for r in rng.choice(F, 7, replace=False):
            up[r] = 0.0
            up[r, rng.integers(H)] = rng.choice([-0.3, 0.3])
        for r in rng.choice(H, 11, replace=False):
            down[r] = 0.0
        gate[rng.integers(F)] = 0.0
        gate[rng.integers(F), :] = 0.0
    L, (W, b, w4s, rss) = _custom_layer(coli, wl, flats)
    zero_W = torch.zeros_like(L["router_w"])
    L["router_w"] = zero_W
    x = synth.activations(wl, 5, n_tok=13)
    got = _run(coli, path, wl, L, x)
    want = oracle.moe_forward(x, np.zeros_like(W), b, w4s[:E], rss[:E], w4s[E], rss[E], H, F, wl.top_k,
                              wl.routed_scale)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("E,k", [(8, 2), (256, 8), (37, 16)])
def test_one_token_tied_keys(coli, path, E, k):
    """One token, a zero router (every sigma = 0.5) and biases drawn from
    four values: most selection keys tie, and the lowest expert index must
    win among equal keys, exactly as in the oracle."""
    import oracle
    from synth.device import build_device_layer
    wl = synth.Workload("t1_ties", 256, 128, E, k, 1, 900 + E + k)
    L = build_device_layer(wl)
    rng = np.random.default_rng(E * 31 + k)
    b = rng.choice(np.array([-0.25, 0.0, 0.125, 0.5], np.float32), size=E).astype(np.float32)
    L["router_w"] = torch.zeros_like(L["router_w"])
    L["router_b"] = torch.from_numpy(b).cuda()
    x = synth.activations(wl, 11)
    got = _run(coli, path, wl, L, x)
    ref = OracleLayer(wl)
    ridx, _ = oracle.route(x, np.zeros_like(ref.W), b, k, wl.routed_scale)
    order = sorted(range(E), key=lambda e: (-b[e], e))[:k]
    assert list(ridx[0]) == order                       # the oracle follows the rule
    w4, rs = [None] * E, [None] * E
    for e in order:
        w4[e], rs[e] = ref.expert(e)
    want = oracle.moe_forward(x, np.zeros_like(ref.W), b, w4, rs, ref.shared[0], ref.shared[1],
                              wl.hidden, wl.ffn, k, wl.routed_scale)
    np.testing.assert_array_equal(got, want)


# --------------------------------------------------------------------------- #
# expert FFN widths that are a multiple of 32 but not of 128                   #
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("F,T", [(160, 5), (96, 1), (224, 300)])
def test_ffn_multiple_of_32(coli, F, T):
    """An FFN width of 32 * odd (or 32 * 3, 32 * 7) runs on the streaming
    path with 16-byte weight stages, bit-exact; AUTO picks that path even for a
    batch large enough for the grouped GEMM, and a forward forced onto the
    GEMM (whose tiles need F % 128 == 0) is refused with COLI_E_UNIMPL before
    any launch."""
    from synth.device import build_device_layer
    wl = synth.Workload(f"ffn{F}", 256, F, 8, 2, T, 950 + F)
    L = build_device_layer(wl)
    x = synth.activations(wl, 1)
    want = OracleLayer(wl).forward(x)
    got = _run(coli, "gemv", wl, L, x)
    np.testing.assert_array_equal(got, want)
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, T)
    coli.set_path(coli.PATH_AUTO, 1)          # AUTO would take the GEMM from one token on
    try:
        got = coli.layer_forward(torch.from_numpy(x).cuda(), L["router_w"], L["router_b"], L["expert_w4"],
                                 L["expert_rs"], L["shared_w4"], L["shared_rs"]).cpu().numpy()
        np.testing.assert_array_equal(got, want)
        coli.set_path(coli.PATH_GEMM)
        with pytest.raises(coli.ColiError) as ei:
            coli.layer_forward(torch.from_numpy(x).cuda(), L["router_w"], L["router_b"], L["expert_w4"],
                               L["expert_rs"], L["shared_w4"], L["shared_rs"])
        assert ei.value.code == coli.E_UNIMPL
    finally:
        coli.set_path(coli.PATH_AUTO, 0)
    assert coli.get_device_status() == coli.OK
