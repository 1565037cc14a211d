"""Pins of the CPU oracle to facts outside itself.

Each test checks the oracle against something it does not compute: worked
values from the rounding rule, closed forms, invariants, brute force with an
independent method (float64 numpy, integer unpacking by bit operations, numpy's
stable sort), or a special case that reduces to a library routine.  The tests
are chosen so that a plausible slip anywhere in the oracle (a dropped term, a
wrong sign or offset, a transposed operand, the bias in the wrong place) fails
at least one of them.
"""
import math

import numpy as np
import pytest

from conftest import golden_path

import synth

TINY = synth.WORKLOADS["tiny"]


def _f32_ulp(v):
    v = np.float32(abs(v))
    return float(np.spacing(v))


# --------------------------------------------------------------------------- #
# rounding rule and Q8_0                                                      #
# --------------------------------------------------------------------------- #
def _read_golden(name):
    rows = []
    for line in open(golden_path(name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line)
    return rows


def test_lrintf_half_even_worked_values(orc):
    for row in _read_golden("lrintf_half_even.txt"):
        v, want = row.split()
        assert orc.lrintf(float(v)) == int(want), row
        # special case that reduces to a library routine: numpy's rint
        assert int(np.rint(np.float32(v))) == int(want), row


def test_q8_0_worked_blocks(orc):
    for row in _read_golden("q8_0_worked_blocks.txt"):
        name, xs, d, qs = [s.strip() for s in row.split(";")]
        x = np.array([float(t) for t in xs.split()], np.float32)
        q_want = np.array([int(t) for t in qs.split()], np.int8)
        assert x.size == 32 and q_want.size == 32, name
        q, dd = orc.q8_0(x)
        assert float(dd[0]) == float(d), name
        np.testing.assert_array_equal(q, q_want, err_msg=name)


def test_q8_0_invariants(orc):
    g = np.random.default_rng(11)
    blocks = [g.standard_normal(32) * s for s in (1e-30, 1e-3, 1.0, 7.0, 1e6)]
    one = np.zeros(32)
    one[17] = -3.25
    blocks.append(one)
    x = np.concatenate(blocks).astype(np.float32)
    q, d = orc.q8_0(x)
    for b in range(x.size // 32):
        xb = x[32 * b: 32 * b + 32].astype(np.float64)
        qb = q[32 * b: 32 * b + 32].astype(np.int64)
        db = float(d[b])
        amax = np.abs(xb).max()
        assert abs(db * 127 - amax) <= 2 * _f32_ulp(amax)
        assert np.all(np.abs(qb) <= 127)
        k = int(np.argmax(np.abs(xb)))
        assert qb[k] == (127 if xb[k] > 0 else -127)
        # reconstruction error at most half a step (plus float rounding of x/d)
        err = np.abs(xb - qb * db)
        assert np.all(err <= db * (0.5 + 1e-6)), (b, err.max() / db)


# --------------------------------------------------------------------------- #
# int4 container                                                              #
# --------------------------------------------------------------------------- #
def test_pack_roundtrip_all_nibble_pairs(orc):
    a, b = np.meshgrid(np.arange(-7, 8), np.arange(-7, 8), indexing="ij")
    q = np.stack([a.ravel(), b.ravel()], 1).ravel()           # 225 pairs, 450 codes
    q = np.concatenate([q, [7, -7]]).astype(np.int64)          # pin max|w| -> s
    K = 480
    q = np.concatenate([q, np.zeros(K - q.size, np.int64)])
    s = 0.25                                                   # power of two: w/s exact
    w = (q * s).astype(np.float32)[None, :]
    packed, scale = orc.pack_int4_rows(w)
    assert float(scale[0]) == s
    np.testing.assert_array_equal(orc.unpack_int4_rows(packed)[0], q)
    # byte layout: element 2j in the low nibble, 2j+1 in the high, code + 8
    lo = (q[0::2] + 8).astype(np.uint8)
    hi = (q[1::2] + 8).astype(np.uint8)
    np.testing.assert_array_equal(packed[0], lo | (hi << 4))


def test_pack_invariants(orc):
    g = np.random.default_rng(5)
    w = (g.standard_normal((16, 256)) * 0.02).astype(np.float32)
    w[3] = 0.0
    w[7, 100] = 0.9                                            # an outlier row
    packed, scale = orc.pack_int4_rows(w)
    qs = orc.unpack_int4_rows(packed).astype(np.int64)
    assert float(scale[3]) == 0.0 and np.all(packed[3] == 0x88)
    for r in range(16):
        if r == 3:
            continue
        s = float(scale[r])
        amax = float(np.abs(w[r]).max())
        assert abs(s * 7 - amax) <= 2 * _f32_ulp(amax)
        assert np.all(np.abs(qs[r]) <= 7)
        k = int(np.argmax(np.abs(w[r])))
        assert qs[r, k] == (7 if w[r, k] > 0 else -7)
        assert np.all(np.abs(w[r].astype(np.float64) - qs[r] * s) <= s * (0.5 + 1e-6))


# --------------------------------------------------------------------------- #
# own exponential and sigmoid                                                 #
# --------------------------------------------------------------------------- #
def test_exp_within_two_ulp():
    import oracle
    zs = np.concatenate([np.linspace(-87, 88, 20001), [-1e-8, 0.0, 1e-8, 0.5, -0.5, 1.0, 88.0, -87.0]])
    worst = 0.0
    for z in zs.astype(np.float32):
        got = oracle.exp(float(z))
        ref = math.exp(float(z))
        worst = max(worst, abs(got - ref) / _f32_ulp(np.float32(ref)))
    assert worst <= 2.0, worst
    assert oracle.exp(0.0) == 1.0
    assert math.isinf(oracle.exp(89.0)) and oracle.exp(-88.0) == 0.0


def test_sigmoid_values():
    import oracle
    assert oracle.sigmoid(0.0) == 0.5
    assert oracle.sigmoid(100.0) == 1.0 and oracle.sigmoid(-100.0) == 0.0
    for z in np.linspace(-30, 30, 6001).astype(np.float32):
        ref = 1.0 / (1.0 + math.exp(-float(z)))
        got = oracle.sigmoid(float(z))
        assert abs(got - ref) <= 3 * _f32_ulp(np.float32(ref)) + 1e-45, z


# --------------------------------------------------------------------------- #
# router                                                                      #
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("H", [256, 2048, 6144])
def test_router_logit_vs_double(orc, H):
    g = np.random.default_rng(H)
    for _ in range(20):
        x = g.standard_normal(H).astype(np.float32)
        w = (g.standard_normal(H) * 0.02).astype(np.float32)
        ref = float(np.dot(x.astype(np.float64), w.astype(np.float64)))
        mag = float(np.abs(x.astype(np.float64) * w).sum())
        assert abs(orc.router_logit(x, w) - ref) <= 1e-5 * mag + 1e-30


def test_router_logit_exact_on_integers(orc):
    # every product and partial sum is a small integer, so any order is exact:
    # a dropped or doubled element shows up as a wrong integer
    g = np.random.default_rng(3)
    for H in (256, 2048, 6144):
        x = g.integers(-50, 51, H).astype(np.float32)
        w = g.integers(-50, 51, H).astype(np.float32)
        assert orc.router_logit(x, w) == float(np.dot(x.astype(np.int64), w.astype(np.int64)))


def _route_ref64(x, W, b, k, scale):
    logits = x.astype(np.float64) @ W.astype(np.float64).T
    sig = 1.0 / (1.0 + np.exp(-logits))
    sel = sig + b.astype(np.float64)
    T, E = sel.shape
    idx = np.empty((T, k), np.int64)
    w = np.empty((T, k))
    gap = np.empty(T)
    for t in range(T):
        order = np.lexsort((np.arange(E), -sel[t]))
        idx[t] = order[:k]
        gap[t] = sel[t, order[k - 1]] - sel[t, order[k]] if k < E else 1.0
        w[t] = sig[t, idx[t]] / sig[t, idx[t]].sum() * scale
    return idx, w, gap


@pytest.mark.parametrize("shape", [(256, 8, 2, 16), (6144, 256, 8, 8)])
def test_route_vs_float64_bruteforce(orc, shape):
    H, E, k, T = shape
    g = np.random.default_rng(H + E)
    x = g.standard_normal((T, H)).astype(np.float32)
    W = (g.standard_normal((E, H)) * 0.02).astype(np.float32)
    b = (g.standard_normal(E) * 0.01).astype(np.float32)
    idx, w = orc.route(x, W, b, k, 2.5)
    ridx, rw, gap = _route_ref64(x, W, b, k, 2.5)
    for t in range(T):
        if gap[t] > 1e-5:                       # not a near tie at the k-th place
            assert set(idx[t]) == set(ridx[t]), t
        # weights follow the returned experts, renormalised to routed_scale
        logit64 = x[t].astype(np.float64) @ W[idx[t]].astype(np.float64).T
        sig64 = 1.0 / (1.0 + np.exp(-logit64))
        np.testing.assert_allclose(w[t], sig64 / sig64.sum() * 2.5, rtol=2e-6)
        # rank order: selection keys non-increasing
        sel64 = sig64 + b[idx[t]]
        assert np.all(np.diff(sel64) <= 1e-6)


@pytest.mark.parametrize("k,E", [(2, 8), (8, 256), (8, 8)])
def test_route_zero_router_closed_form(orc, k, E):
    # W = 0: every logit is 0, sigma = 1/2, the selection is the top-k of the
    # bias, and every weight is exactly routed_scale / k
    H = 256
    g = np.random.default_rng(k * E)
    x = g.standard_normal((3, H)).astype(np.float32)
    W = np.zeros((E, H), np.float32)
    b = (g.standard_normal(E) * 0.01).astype(np.float32)
    idx, w = orc.route(x, W, b, k, 2.5)
    want = np.lexsort((np.arange(E), -b.astype(np.float64)))[:k]
    for t in range(3):
        np.testing.assert_array_equal(idx[t], want)
        assert np.all(w[t] == np.float32(2.5 / k))


def test_route_ties_go_to_lower_index(orc):
    H, E, k = 256, 8, 3
    g = np.random.default_rng(9)
    base = (g.standard_normal(H) * 0.02).astype(np.float32)
    W = np.tile(base, (E, 1))                   # identical rows: identical logits
    b = np.zeros(E, np.float32)
    x = g.standard_normal((2, H)).astype(np.float32)
    idx, w = orc.route(x, W, b, k, 2.5)
    np.testing.assert_array_equal(idx, [[0, 1, 2], [0, 1, 2]])
    b[5] = 1e-3                                 # a strictly larger key wins first
    idx, _ = orc.route(x, W, b, k, 2.5)
    np.testing.assert_array_equal(idx, [[5, 0, 1], [5, 0, 1]])


# --------------------------------------------------------------------------- #
# dispatch                                                                    #
# --------------------------------------------------------------------------- #
@pytest.mark.parametrize("T,k,E", [(4, 2, 8), (1, 8, 256), (2048, 8, 256), (37, 3, 5)])
def test_dispatch_vs_stable_sort(orc, T, k, E):
    g = np.random.default_rng(T * k)
    zipf = 1.0 / (np.arange(E) + 1.0) ** 1.1
    idx = np.stack([g.choice(E, size=k, replace=False, p=zipf / zipf.sum()) for _ in range(T)])
    idx = idx.astype(np.int32)
    counts, offsets, perm, inv = orc.dispatch(idx, E)
    flat = idx.ravel()
    np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=E))]))
    np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
    np.testing.assert_array_equal(inv[perm], np.arange(T * k))
    assert sorted(perm.tolist()) == list(range(T * k))
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg // k) > 0)


# --------------------------------------------------------------------------- #
# integer dot products and the expert FFN                                      #
# --------------------------------------------------------------------------- #
def _unpack_bits(packed):
    lo = (packed & 0x0F).astype(np.int64) - 8
    hi = (packed >> 4).astype(np.int64) - 8
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.int64)
    out[:, 0::2] = lo
    out[:, 1::2] = hi
    return out


def test_block_dots_bruteforce(orc):
    g = np.random.default_rng(2)
    K = 512
    packed = g.integers(0, 256, (24, K // 2), dtype=np.uint8)
    packed[0] = 0x00                                           # all codes -8
    packed[1] = 0xFF                                           # all codes +7
    q = g.integers(-127, 128, K).astype(np.int8)
    q[:32] = 127
    I = orc.block_dots(packed, q)
    ref = (_unpack_bits(packed) * q.astype(np.int64)).reshape(24, K // 32, 32).sum(-1)
    np.testing.assert_array_equal(I, ref)
    assert I[0, 0] == -8 * 127 * 32 and I[1, 0] == 7 * 127 * 32


def test_rows_dot_matches_dequantised_double_dot(orc):
    g = np.random.default_rng(4)
    K = 6144
    w = (g.standard_normal((8, K)) * 0.02).astype(np.float32)
    x = g.standard_normal(K).astype(np.float32)
    packed, s = orc.pack_int4_rows(w)
    q, d = orc.q8_0(x)
    got = orc.rows_dot(packed, s, q, d)
    wq = _unpack_bits(packed) * s[:, None].astype(np.float64)
    xq = q.astype(np.float64) * np.repeat(d.astype(np.float64), 32)
    terms = wq * xq[None, :]
    ref = terms.sum(1)
    assert np.all(np.abs(got - ref) <= 1e-6 * np.abs(terms).sum(1))


def _swiglu64(Wg, Wu, Wd, x):
    g = Wg @ x
    u = Wu @ x
    h = g / (1.0 + np.exp(-g)) * u
    return Wd @ h, h


def _rel_rms(a, b):
    return float(np.sqrt(np.mean((a - b) ** 2)) / np.sqrt(np.mean(b ** 2)))


def test_expert_ffn_against_float_swiglu(orc):
    H, F = TINY.hidden, TINY.ffn
    g = np.random.default_rng(8)
    Wg = (g.standard_normal((F, H)) * 0.02).astype(np.float32)
    Wu = (g.standard_normal((F, H)) * 0.02).astype(np.float32)
    Wd = (g.standard_normal((H, F)) * 0.02).astype(np.float32)
    pg, sg = orc.pack_int4_rows(Wg)
    pu, su = orc.pack_int4_rows(Wu)
    pd, sd = orc.pack_int4_rows(Wd)
    ew4 = np.concatenate([pg.ravel(), pu.ravel(), pd.ravel()])
    ers = np.concatenate([sg, su, sd])
    deq = lambda p, s: _unpack_bits(p) * s[:, None].astype(np.float64)
    Dg, Du, Dd = deq(pg, sg), deq(pu, su), deq(pd, sd)
    for trial in range(6):
        x = g.standard_normal(H).astype(np.float32)
        qx, dx = orc.q8_0(x)
        r = orc.expert_ffn(ew4, ers, H, F, qx, dx)
        # (1) dequantised weights, exact activations: only the two activation
        # quantisers differ; predicted error from their measured noise
        y_ref, h_ref = _swiglu64(Dg, Du, Dd, x.astype(np.float64))
        ex = _rel_rms(qx * np.repeat(dx, 32).astype(np.float64), x.astype(np.float64))
        eh = _rel_rms(r["qh"] * np.repeat(r["dh"], 32).astype(np.float64), r["h"].astype(np.float64))
        pred = math.sqrt((2 * ex) ** 2 + eh ** 2)
        err = _rel_rms(r["y"].astype(np.float64), y_ref)
        assert err <= 2 * pred, (trial, err, pred)
        # (2) gate is gate and up is up: swapping them is far off
        y_swap, _ = _swiglu64(Du, Dg, Dd, x.astype(np.float64))
        assert _rel_rms(y_swap, y_ref) > 10 * err
        # (3) unquantised weights: int4 noise dominates, ~ s/sqrt(12) per weight
        y32, _ = _swiglu64(Wg.astype(np.float64), Wu.astype(np.float64), Wd.astype(np.float64),
                           x.astype(np.float64))
        ew = np.mean([_rel_rms(deq(p, s), W.astype(np.float64))
                      for p, s, W in ((pg, sg, Wg), (pu, su, Wu), (pd, sd, Wd))])
        pred_w = math.sqrt(3 * ew ** 2 + pred ** 2)
        assert _rel_rms(r["y"].astype(np.float64), y32) <= 2 * pred_w


# --------------------------------------------------------------------------- #
# the whole layer                                                             #
# --------------------------------------------------------------------------- #
def _tiny_layer(orc, wl=TINY, same_experts=False):
    W, b = synth.router(wl)
    ew4, ers = [], []
    for e in range(wl.n_experts + 1):
        src = wl.n_experts if same_experts else e
        flat = synth.expert_f32_rows(wl, src)
        F, H = wl.ffn, wl.hidden
        pg, sg = orc.pack_int4_rows(flat[:F * H].reshape(F, H))
        pu, su = orc.pack_int4_rows(flat[F * H:2 * F * H].reshape(F, H))
        pd, sd = orc.pack_int4_rows(flat[2 * F * H:].reshape(H, F))
        ew4.append(np.concatenate([pg.ravel(), pu.ravel(), pd.ravel()]))
        ers.append(np.concatenate([sg, su, sd]))
    return W, b, ew4[:-1], ers[:-1], ew4[-1], ers[-1]


def test_forward_composes_its_steps(orc):
    wl = TINY
    W, b, ew4, ers, sw4, srs = _tiny_layer(orc)
    x = synth.activations(wl, 0)
    out, it = orc.moe_forward(x, W, b, ew4, ers, sw4, srs, wl.hidden, wl.ffn, wl.top_k,
                              wl.routed_scale, intermediates=True)
    idx, w = orc.route(x, W, b, wl.top_k, wl.routed_scale)
    np.testing.assert_array_equal(it["idx"], idx)
    for t in range(wl.n_tok):
        qx, dx = orc.q8_0(x[t])
        ys = orc.expert_ffn(sw4, srs, wl.hidden, wl.ffn, qx, dx)["y"].astype(np.float64)
        acc = ys.copy()
        for r in range(wl.top_k):
            y = orc.expert_ffn(ew4[idx[t, r]], ers[idx[t, r]], wl.hidden, wl.ffn, qx, dx)["y"]
            acc += float(w[t, r]) * y.astype(np.float64)
        assert np.all(np.abs(out[t] - acc) <= 1e-6 * (np.abs(acc) + np.abs(ys).max()))


def test_forward_all_experts_equal_shared(orc):
    # every routed expert is the shared one: out = y * (1 + sum of weights),
    # and the weights sum to routed_scale
    wl = TINY
    W, b, ew4, ers, sw4, srs = _tiny_layer(orc, same_experts=True)
    x = synth.activations(wl, 1)
    out, it = orc.moe_forward(x, W, b, ew4, ers, sw4, srs, wl.hidden, wl.ffn, wl.top_k,
                              wl.routed_scale, intermediates=True)
    ys = it["y_shared"].astype(np.float64)
    np.testing.assert_allclose(it["w"].sum(1), 2.5, rtol=1e-6)
    np.testing.assert_allclose(out, ys * 3.5, rtol=1e-5, atol=1e-6 * np.abs(ys).max())


def test_forward_independent_of_batch_composition(orc):
    # the placement of a token in a batch never changes its result
    wl = TINY
    W, b, ew4, ers, sw4, srs = _tiny_layer(orc)
    x = synth.activations(wl, 2)
    out = orc.moe_forward(x, W, b, ew4, ers, sw4, srs, wl.hidden, wl.ffn, wl.top_k, wl.routed_scale)
    for t in range(wl.n_tok):
        one = orc.moe_forward(x[t:t + 1], W, b, ew4, ers, sw4, srs, wl.hidden, wl.ffn, wl.top_k,
                              wl.routed_scale)
        np.testing.assert_array_equal(one[0], out[t])
    rev = orc.moe_forward(x[::-1].copy(), W, b, ew4, ers, sw4, srs, wl.hidden, wl.ffn, wl.top_k,
                          wl.routed_scale)
    np.testing.assert_array_equal(rev[::-1], out)


def test_forward_rejects_missing_expert(orc):
    wl = TINY
    W, b, ew4, ers, sw4, srs = _tiny_layer(orc)
    x = synth.activations(wl, 0)
    idx, _ = orc.route(x, W, b, wl.top_k, wl.routed_scale)
    ew4 = list(ew4)
    ew4[int(idx[0, 0])] = None
    with pytest.raises(ValueError):
        orc.moe_forward(x, W, b, ew4, ers, sw4, srs, wl.hidden, wl.ffn, wl.top_k, wl.routed_scale)


# --------------------------------------------------------------------------- #
# Pre-norm of the stacked-layer sweep: x / sqrt(mean(x^2) + eps)               #
# --------------------------------------------------------------------------- #
def test_rmsnorm_constant_vector_gives_unit_sign(orc):
    """A constant row c (|c| = 2^10, so eps is below half an ulp of mean(x^2)):
    mean(x^2) = c^2 exactly and every output is sign(c) exactly.  A sum in
    place of the mean, or a missing square root, fails this."""
    x = np.full((3, 256), 1024.0, np.float32)
    x[1] = -1024.0
    x[2, :128] = 1024.0
    x[2, 128:] = -1024.0
    xn = orc.rmsnorm(x)
    np.testing.assert_array_equal(xn, np.sign(x))


def test_rmsnorm_power_of_two_scaling_is_exact(orc):
    """Scaling a row by 2 scales every partial sum by 4 exactly and the root
    by 2 exactly, so the output does not change in any bit (eps absorbed)."""
    x = (np.random.default_rng(5).standard_normal((4, 6144)) * 1024.0).astype(np.float32)
    np.testing.assert_array_equal(orc.rmsnorm(x), orc.rmsnorm((2.0 * x).astype(np.float32)))


def test_rmsnorm_matches_double_precision(orc):
    rng = np.random.default_rng(6)
    for H in (256, 6144):
        x = rng.standard_normal((7, H)).astype(np.float32) * np.float32(3.0)
        xd = x.astype(np.float64)
        want = xd / np.sqrt(np.mean(xd * xd, axis=1, keepdims=True) + 1e-6)
        got = orc.rmsnorm(x)
        assert np.max(np.abs(got - want) / np.abs(want).max()) < 2e-6


def test_rmsnorm_zero_row_is_zero(orc):
    x = np.zeros((2, 256), np.float32)
    np.testing.assert_array_equal(orc.rmsnorm(x), x)


# --------------------------------------------------------------------------- #
# Thread count: OpenMP runs over independent outputs only                     #
# --------------------------------------------------------------------------- #
def test_results_do_not_depend_on_thread_count(orc):
    """Every parallel loop of the oracle writes disjoint outputs, each with its
    own sequential arithmetic, so one thread and several give identical bits:
    routing, the intermediates and the layer output of a multi-token batch
    (including tokens that share experts), and the router logits."""
    from helpers import OracleLayer
    wl = synth.Workload("threads", 512, 256, 16, 4, 9, 41)
    ref = OracleLayer(wl)
    x = synth.activations(wl, 3)
    idx, _ = orc.route(x, ref.W, ref.b, wl.top_k, wl.routed_scale)
    w4, rs = [None] * wl.n_experts, [None] * wl.n_experts
    for e in set(int(v) for v in idx.ravel()):
        w4[e], rs[e] = ref.expert(e)
    runs = []
    try:
        for n in (1, 4):
            orc.set_threads(n)
            r = orc.route(x, ref.W, ref.b, wl.top_k, wl.routed_scale, want_logits=True)
            f = orc.moe_forward(x, ref.W, ref.b, w4, rs, ref.shared[0], ref.shared[1], wl.hidden, wl.ffn,
                                wl.top_k, wl.routed_scale, intermediates=True)
            runs.append((r, f))
    finally:
        orc.set_threads(0)

    def flat(v):
        if isinstance(v, dict):
            return [a for key in sorted(v) for a in flat(v[key])]
        if isinstance(v, (tuple, list)):
            return [a for item in v for a in flat(item)]
        return [np.asarray(v)]

    a, b = flat(runs[0]), flat(runs[1])
    assert len(a) == len(b) and len(a) > 4
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u.view(np.uint8) if u.dtype.kind == "f" else u,
                                      v.view(np.uint8) if v.dtype.kind == "f" else v)



# --------------------------------------------------------------------------- #
# The int8 weight container (the pages' int8 head / int8 container)          #
# --------------------------------------------------------------------------- #
def test_int8_container_rule(orc):
    """s = max|row| / 127, q = clamp(lrintf(w / s), -127, 127): the largest
    element maps to +-127, every element is within s/2 of q*s, a zero row has
    s = 0 and zero codes, and a row of one repeated value is exact."""
    g = np.random.default_rng(21)
    w = (g.standard_normal((32, 256)) * 0.02).astype(np.float32)
    w[3] = 0.0
    w[4] = np.float32(0.5)
    q, s = orc.pack_int8_rows(w)
    assert q.dtype == np.int8 and np.all(np.abs(q.astype(np.int32)) <= 127)
    for r in range(32):
        if r == 3:
            assert s[r] == 0.0 and not np.any(q[r])
            continue
        assert s[r] == np.float32(np.float32(np.abs(w[r]).max()) / np.float32(127.0))
        k = int(np.argmax(np.abs(w[r])))
        assert abs(int(q[r, k])) == 127
        err = np.abs(w[r].astype(np.float64) - q[r].astype(np.float64) * float(s[r]))
        assert np.all(err <= float(s[r]) / 2 * (1 + 2 ** -20) + 1e-12)
    assert np.all(q[4] == 127)


def test_int8_block_dots_bruteforce(orc):
    g = np.random.default_rng(22)
    K = 512
    w8 = g.integers(-127, 128, (16, K)).astype(np.int8)
    w8[0] = -127
    q = g.integers(-127, 128, K).astype(np.int8)
    q[:32] = 127
    I = orc.block_dots_w8(w8, q)
    ref = (w8.astype(np.int64) * q.astype(np.int64)).reshape(16, K // 32, 32).sum(-1)
    np.testing.assert_array_equal(I, ref)
    assert I[0, 0] == -127 * 127 * 32


def test_int4_codes_in_the_int8_container_give_identical_bits(orc):
    """Container-equivalence pin of the oracle's two weight paths (a guard on
    the shared row-dot code, not a check of the pages' claim, which holds here
    by construction): an expert's int4 codes, widened into the int8 container
    with the same row scales, give the same block dots, the same expert
    outputs (g, u, h, the requantised h and y) and the same layer output, bit
    for bit, through the int8 path.  The GPU-side counterpart compares the
    device's int4 and int8-container kernels."""
    H, F = TINY.hidden, TINY.ffn
    g = np.random.default_rng(23)
    mats = [(g.standard_normal((F, H)) * 0.02).astype(np.float32),
            (g.standard_normal((F, H)) * 0.02).astype(np.float32),
            (g.standard_normal((H, F)) * 0.02).astype(np.float32)]
    packs = [orc.pack_int4_rows(m) for m in mats]
    ew4 = np.concatenate([p.ravel() for p, _ in packs])
    ew8 = np.concatenate([orc.unpack_int4_rows(p).ravel() for p, _ in packs])
    ers = np.concatenate([s for _, s in packs])
    x = g.standard_normal((3, H)).astype(np.float32)
    qx, dx = orc.q8_0(x)
    np.testing.assert_array_equal(orc.block_dots(packs[0][0], qx[0]),
                                  orc.block_dots_w8(orc.unpack_int4_rows(packs[0][0]), qx[0]))
    for t in range(3):
        r4 = orc.expert_ffn(ew4, ers, H, F, qx[t], dx[t], wbits=4)
        r8 = orc.expert_ffn(ew8, ers, H, F, qx[t], dx[t], wbits=8)
        for key in ("g", "u", "h", "qh", "dh", "y"):
            np.testing.assert_array_equal(r4[key].view(np.uint8), r8[key].view(np.uint8), err_msg=key)
    # the whole layer: E = 4 experts sharing this draw's pattern, plus a shared one
    E, k = 4, 2
    W = (g.standard_normal((E, H)) * 0.02).astype(np.float32)
    b = (g.standard_normal(E) * 0.01).astype(np.float32)
    out4 = orc.moe_forward(x, W, b, [ew4] * E, [ers] * E, ew4, ers, H, F, k, 2.5, wbits=4)
    out8 = orc.moe_forward(x, W, b, [ew8] * E, [ers] * E, ew8, ers, H, F, k, 2.5, wbits=8)
    np.testing.assert_array_equal(out4.view(np.uint32), out8.view(np.uint32))


def test_int8_expert_ffn_against_float_swiglu(orc):
    """Int8 weights: against double SwiGLU on the dequantised weights the error
    is the activation quantisers' alone, and against the unquantised weights
    the weight noise (~s/sqrt(12), 18x smaller than int4's) is added; both
    within twice the prediction, and well below the int4 container's error."""
    H, F = TINY.hidden, TINY.ffn
    g = np.random.default_rng(24)
    Ws = [(g.standard_normal((F, H)) * 0.02).astype(np.float32),
          (g.standard_normal((F, H)) * 0.02).astype(np.float32),
          (g.standard_normal((H, F)) * 0.02).astype(np.float32)]
    packs = [orc.pack_int8_rows(W) for W in Ws]
    ew8 = np.concatenate([q.ravel() for q, _ in packs])
    ers = np.concatenate([s for _, s in packs])
    D = [q.astype(np.float64) * s[:, None].astype(np.float64) for q, s in packs]
    p4 = [orc.pack_int4_rows(W) for W in Ws]
    ew4 = np.concatenate([p.ravel() for p, _ in p4])
    ers4 = np.concatenate([s for _, s in p4])
    for trial in range(4):
        x = g.standard_normal(H).astype(np.float32)
        qx, dx = orc.q8_0(x)
        r = orc.expert_ffn(ew8, ers, H, F, qx, dx, wbits=8)
        y_ref, _ = _swiglu64(D[0], D[1], D[2], x.astype(np.float64))
        ex = _rel_rms(qx * np.repeat(dx, 32).astype(np.float64), x.astype(np.float64))
        eh = _rel_rms(r["qh"] * np.repeat(r["dh"], 32).astype(np.float64), r["h"].astype(np.float64))
        pred = math.sqrt((2 * ex) ** 2 + eh ** 2)
        assert _rel_rms(r["y"].astype(np.float64), y_ref) <= 2 * pred
        y32, _ = _swiglu64(*(W.astype(np.float64) for W in Ws), x.astype(np.float64))
        ew = np.mean([_rel_rms(Dm, W.astype(np.float64)) for Dm, W in zip(D, Ws)])
        pred_w = math.sqrt(3 * ew ** 2 + pred ** 2)
        err8 = _rel_rms(r["y"].astype(np.float64), y32)
        assert err8 <= 2 * pred_w
        r4 = orc.expert_ffn(ew4, ers4, H, F, qx, dx, wbits=4)
        assert err8 < _rel_rms(r4["y"].astype(np.float64), y32)


def test_oracle_rejects_unsupported_weight_containers(orc):
    """Only the 4- and 8-bit containers exist: any other width, or a weight
    buffer whose size does not match the container, is refused before the C
    code could read past it."""
    H, F = TINY.hidden, TINY.ffn
    ers = np.ones(2 * F + H, np.float32)
    qx = np.zeros(H, np.int8)
    dx = np.zeros(H // 32, np.float32)
    for wbits in (2, 16, 0):
        with pytest.raises(ValueError):
            orc.expert_ffn(np.zeros(3 * F * H, np.uint8), ers, H, F, qx, dx, wbits=wbits)
    with pytest.raises(ValueError):
        orc.expert_ffn(np.zeros(3 * F * H // 2 - 1, np.uint8), ers, H, F, qx, dx, wbits=4)
    with pytest.raises(ValueError):
        orc.expert_ffn(np.zeros(3 * F * H // 2, np.uint8), ers, H, F, qx, dx, wbits=8)
