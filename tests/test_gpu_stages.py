"""Stage-isolated parity of each CUDA kernel against the oracle, through the
C ABI, on identical inputs.  Integer and index results must be bit-exact;
so must the F32 results whose order is fixed by the method's definition
(quantiser scales, router logits and weights)."""
import numpy as np
import pytest
import torch

import synth
from helpers import oracle_expert

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coli():
    import int4_routed_expert_f32_gb300 as c
    torch.cuda.set_device(0)
    return c


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def test_quantize_bitexact(coli, orc):
    g = np.random.default_rng(0)
    parts = [g.standard_normal(32 * 512) * s for s in (1.0, 1e-3, 50.0)]
    ties = np.array([0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 126.5, -126.5] * 4) ; ties[0] = 127.0
    zero = np.zeros(32)
    x = np.concatenate(parts + [ties, zero]).astype(np.float32)
    q, d = coli.dbg_quantize(_cuda(x))
    rq, rd = orc.q8_0(x)
    np.testing.assert_array_equal(q.cpu().numpy(), rq)
    np.testing.assert_array_equal(d.cpu().numpy().view(np.uint32), rd.view(np.uint32))


@pytest.mark.parametrize("rows,K", [(7, 256), (64, 6144), (300, 2048)])
def test_pack_int4_bitexact(coli, orc, rows, K):
    g = np.random.default_rng(rows)
    w = (g.standard_normal((rows, K)) * 0.02).astype(np.float32)
    w[0] = 0.0
    w[-1, 3] = 0.5
    w[1, ::7] = np.float32(0.02) * 3.5        # exact half-way codes after /s
    p, s = coli.pack_int4(_cuda(w))
    rp, rs = orc.pack_int4_rows(w)
    np.testing.assert_array_equal(p.cpu().numpy(), rp)
    np.testing.assert_array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def test_block_dots_bitexact(coli, orc):
    g = np.random.default_rng(1)
    K = 6144
    w4 = g.integers(0, 256, (97, K // 2), dtype=np.uint8)
    w4[0] = 0x00
    w4[1] = 0xFF
    q = g.integers(-127, 128, K).astype(np.int8)
    q[:64] = -127
    I = coli.dbg_block_dots(_cuda(w4), _cuda(q))
    np.testing.assert_array_equal(I.cpu().numpy(), orc.block_dots(w4, q))


@pytest.mark.parametrize("wl_name,T", [("tiny", 4), ("tiny", 37), ("decode", 1), ("decode", 4),
                                       ("decode", 64), ("prefill", 45)])
def test_route_bitexact(coli, orc, wl_name, T):
    wl = synth.WORKLOADS[wl_name]
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, max(T, 64))
    W, b = synth.router(wl)
    x = synth.activations(wl, 7, n_tok=T)
    idx, w, logits = coli.dbg_route(_cuda(x), _cuda(W), _cuda(b), wl.top_k, want_logits=True)
    ridx, rw, rlogits, _ = orc.route(x, W, b, wl.top_k, wl.routed_scale, want_logits=True)
    np.testing.assert_array_equal(logits.cpu().numpy().view(np.uint32), rlogits.view(np.uint32))
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    np.testing.assert_array_equal(w.cpu().numpy().view(np.uint32), rw.view(np.uint32))


def test_route_ties_and_zero_router(coli, orc):
    wl = synth.WORKLOADS["tiny"]
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 8)
    g = np.random.default_rng(4)
    base = (g.standard_normal(wl.hidden) * 0.02).astype(np.float32)
    W = np.tile(base, (wl.n_experts, 1))
    b = np.zeros(wl.n_experts, np.float32)
    x = g.standard_normal((3, wl.hidden)).astype(np.float32)
    idx, w = coli.dbg_route(_cuda(x), _cuda(W), _cuda(b), wl.top_k)
    np.testing.assert_array_equal(idx.cpu().numpy(), [[0, 1]] * 3)
    W0 = np.zeros_like(W)
    b = (g.standard_normal(wl.n_experts) * 0.01).astype(np.float32)
    idx, w = coli.dbg_route(_cuda(x), _cuda(W0), _cuda(b), wl.top_k)
    ridx, rw = orc.route(x, W0, b, wl.top_k, wl.routed_scale)
    np.testing.assert_array_equal(idx.cpu().numpy(), ridx)
    assert np.all(w.cpu().numpy() == np.float32(2.5 / wl.top_k))


@pytest.mark.parametrize("T,k,E", [(1, 8, 256), (4, 2, 8), (2048, 8, 256), (1500, 3, 37)])
def test_dispatch_bitexact(coli, orc, T, k, E):
    coli.configure(256, 128, E, k, 2.5, T)
    g = np.random.default_rng(T)
    zipf = 1.0 / (np.arange(E) + 1.0) ** 1.1
    idx = np.stack([g.choice(E, size=k, replace=False, p=zipf / zipf.sum()) for _ in range(T)])
    idx = idx.astype(np.int32)
    counts, offsets, perm, inv = coli.dbg_dispatch(_cuda(idx), E)
    rc, ro, rp, ri = orc.dispatch(idx, E)
    np.testing.assert_array_equal(counts.cpu().numpy(), rc)
    np.testing.assert_array_equal(offsets.cpu().numpy(), ro)
    np.testing.assert_array_equal(perm.cpu().numpy(), rp)
    np.testing.assert_array_equal(inv.cpu().numpy(), ri)
    assert coli.get_device_status() == coli.OK


def test_dispatch_reports_bad_index(coli):
    # an index outside [0, E) is rejected by the kernel's own bounds check and
    # reported through the status word; nothing is written out of range
    coli.configure(256, 128, 8, 2, 2.5, 4)
    idx = np.array([[0, 1], [2, 9], [3, 4], [5, -1]], np.int32)
    coli.dbg_dispatch(_cuda(idx), 8)
    assert coli.get_device_status() == coli.E_DEVICE
    assert coli.get_device_status() == coli.OK          # read-and-clear


@pytest.mark.parametrize("wl_name,n", [("tiny", 1), ("tiny", 7), ("decode", 1), ("decode", 4),
                                       ("decode", 9)])
def test_expert_hidden_requant_bitexact(coli, orc, wl_name, n):
    wl = synth.WORKLOADS[wl_name]
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 16)
    ew4, ers = oracle_expert(wl, 3)
    x = synth.activations(wl, 11, n_tok=n)
    qx, dx = orc.q8_0(x)
    h, qh, dh = coli.dbg_expert_hidden(_cuda(ew4), _cuda(ers), _cuda(qx), _cuda(dx), wl.ffn)
    h, qh, dh = h.cpu().numpy(), qh.cpu().numpy(), dh.cpu().numpy()
    for t in range(n):
        r = orc.expert_ffn(ew4, ers, wl.hidden, wl.ffn, qx[t], dx[t])
        # the hidden before requantisation follows the oracle's F32 order exactly
        np.testing.assert_array_equal(h[t].view(np.uint32), r["h"].view(np.uint32))
        np.testing.assert_array_equal(qh[t], r["qh"])
        np.testing.assert_array_equal(dh[t].view(np.uint32), r["dh"].view(np.uint32))
    # the requantiser alone, given the GPU's own h
    q2, d2 = orc.q8_0(h)
    np.testing.assert_array_equal(qh, q2)
    np.testing.assert_array_equal(dh.view(np.uint32), d2.view(np.uint32))


def test_rmsnorm_bit_exact():
    """The stacked layer's pre-norm: same F32 operation sequence as the oracle."""
    import oracle
    import int4_routed_expert_f32_gb300 as coli
    rng = np.random.default_rng(11)
    for T, H in ((5, 6144), (3, 256), (1, 128)):
        x = (rng.standard_normal((T, H)) * rng.uniform(0.01, 100.0, size=(T, 1))).astype(np.float32)
        got = coli.dbg_rmsnorm(torch.from_numpy(x).cuda()).cpu().numpy()
        np.testing.assert_array_equal(got, oracle.rmsnorm(x))
