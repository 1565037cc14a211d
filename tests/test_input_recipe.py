"""The synthetic inputs follow their stated recipe.

The workloads stand in for data the method is measured on, so their
statistics are part of what the benchmark numbers mean: the prefill batch's
expert skew, the verify batch's token correlation and the sweep's
layer-to-layer routing correlation.  Routing here is the oracle's (CPU).
"""
import dataclasses

import numpy as np
import pytest

import synth


@pytest.mark.parametrize("seed", [10_000, 10_001])
def test_prefill_batch_has_the_stated_expert_skew(orc, seed):
    """2048 tokens routed by the oracle: per-expert counts run from a handful
    to several hundred ("from ~0 to several hundred tokens per expert", the
    reading the Zipf bias term was calibrated for), and every pair lands."""
    wl = synth.WORKLOADS["prefill"]
    W, b = synth.router(wl)
    x = synth.activations(wl, seed)
    idx, _ = orc.route(x, W, b, wl.top_k, wl.routed_scale)
    counts = np.bincount(idx.ravel(), minlength=wl.n_experts)
    assert counts.sum() == wl.n_tok * wl.top_k
    assert 200 <= counts.max() <= 800
    assert counts.min() <= 16
    assert 30 <= np.median(counts) <= 100


def test_batch_profile_fills_four_token_tiles_like_a_128_token_batch(orc):
    """The batch_profile case (64 experts, 32 tokens, the skewed bias) stands
    in for a 128-token batch over 256 experts in expert-kernel captures: four
    routed tokens per expert on average, and 4-token tiles about as full
    (0.73 at batch 128 over 256 experts)."""
    wl = synth.WORKLOADS["batch_profile"]
    W, b = synth.router(wl)
    x = synth.activations(wl, 0)
    idx, _ = orc.route(x, W, b, wl.top_k, wl.routed_scale)
    counts = np.bincount(idx.ravel(), minlength=wl.n_experts)
    assert counts.sum() == wl.n_tok * wl.top_k == 4 * wl.n_experts
    tiles = np.ceil(counts / 4).sum()
    assert 0.68 <= counts.sum() / (4 * tiles) <= 0.80
    assert (counts > 0).sum() >= 56


def test_prefill_tokens_have_norm_jitter():
    """x ~ N(0, 1) * U(0.5, 2) per token: row norms spread over a factor of
    about four around sqrt(H)."""
    wl = synth.WORKLOADS["prefill"]
    x = synth.activations(wl, 10_000)
    r = np.linalg.norm(x.astype(np.float64), axis=1) / np.sqrt(wl.hidden)
    assert 0.45 < r.min() < 0.6 and 1.9 < r.max() < 2.1


def test_verify_tokens_share_a_common_draw():
    """x_t = 0.7 x_0 + 0.3 N(0, 1) for t = 0..3, x_0 a fresh draw per forward
    (not itself one of the tokens): every pair of the four tokens correlates
    at 0.49 / (0.49 + 0.09) = 0.845."""
    wl = synth.WORKLOADS["verify"]
    for step in (7, 8):
        x = synth.activations(wl, step).astype(np.float64)
        assert x.shape == (4, wl.hidden)
        c = np.corrcoef(x)
        for t in range(4):
            for u in range(t + 1, 4):
                assert abs(c[t, u] - 0.845) < 0.02
    # forwards draw independent bases
    a, b = synth.activations(wl, 7)[0], synth.activations(wl, 8)[0]
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.05


def test_sweep_layers_route_alike_on_the_same_tokens(orc):
    """Each sweep layer's router rows are 0.97 x the previous layer's plus
    fresh noise: on the same (normalised) tokens about 70% of a layer's top-8
    are also in the previous layer's, and independent routers would share
    about 8/256 of them."""
    wl = synth.WORKLOADS["sweep"]
    xs = orc.rmsnorm(synth.activations(wl, 5))
    prev = None
    overlaps = []
    for layer in range(wl.layers):
        W, b = synth.router(wl, layer)
        idx, _ = orc.route(xs, W, b, wl.top_k, wl.routed_scale)
        if prev is not None:
            overlaps.append(np.mean([len(set(a) & set(p)) / wl.top_k for a, p in zip(idx, prev)]))
        prev = idx
    assert len(overlaps) == wl.layers - 1
    assert 0.6 <= float(np.mean(overlaps)) <= 0.8
    assert min(overlaps) > 0.55


def test_sweep_down_rows_are_the_draw_times_a_power_of_two():
    """The sweep's down rows are its N(0, 0.02) draw times 1/32 (a residual
    update of a few percent of the stream, as in a trained stack); gate and
    up rows are the draw itself.  A power of two: the scaled rows pack to the
    same int4 codes, with row scales divided by 32."""
    wl = synth.WORKLOADS["sweep"]
    assert wl.down_scale == 1.0 / 32
    plain = dataclasses.replace(wl, down_scale=1.0)
    F, H = wl.ffn, wl.hidden
    for e in (0, 17, wl.n_experts):
        a = synth.expert_f32_rows(wl, e, 3)
        b = synth.expert_f32_rows(plain, e, 3)
        np.testing.assert_array_equal(a[: 2 * F * H], b[: 2 * F * H])
        np.testing.assert_array_equal(a[2 * F * H:], b[2 * F * H:] / np.float32(32))
    gate, up, down = synth.expert_f32(wl, 5, 1)
    np.testing.assert_array_equal(down.ravel(), synth.expert_f32_rows(wl, 5, 1)[2 * F * H:])
