"""Seeded synthetic inputs for the quantized MoE layer.

This module draws random numbers and nothing else: it holds none of the layer's
arithmetic (no quantisation, routing or matmul).  Both the CUDA path and the
oracle take their inputs from here.  Every draw comes from numpy's PCG64 seeded
by a ``SeedSequence`` of (config seed, tensor id, index), so any tensor can be
regenerated alone, in any order, on any thread.

Workloads (GLM-5.2-shaped MoE layer: 256 routed experts, top-8, one shared
expert, SwiGLU experts, hidden 6144, expert FFN 2048):

* ``tiny``      hidden 256, FFN 128, 8 experts top-2, 4 tokens, seed 0
* ``decode``    the GLM-5.2 shape, 1 token per forward, seed 1
* ``verify``    the decode layer's weights, 4 correlated tokens per forward
                (x_t = 0.7 x_0 + 0.3 N(0,1)), activation seed 2
* ``prefill``   the decode layer's weights, 2048 tokens with per-token norm
                jitter U(0.5, 2) and a Zipf-skewed router bias, activation
                seed 3
* ``sweep``     8 stacked GLM-5.2-shaped layers (seeds 100..107), batches
                1, 8, 32, 128, Zipf-skewed bias, router rows of layer l drawn
                correlated with layer l-1's

Distributions: router weights N(0, 0.02), router bias N(0, 0.01), expert
weights N(0, 0.02) (F32, before the int4 container's quantiser), activations
N(0, 1).
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# tensor ids inside one seed's stream family
_T_ROUTER_W = 1
_T_ROUTER_B = 2
_T_EXPERT = 3
_T_X = 4
_T_X_NOISE = 5
_T_JITTER = 6
_T_ZIPF_PERM = 7
_T_ROUTER_W_FRESH = 8


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    ffn: int
    n_experts: int
    top_k: int
    n_tok: int
    seed: int
    routed_scale: float = 2.5
    correlated_tokens: bool = False      # verify: x_t = 0.7 x_0 + 0.3 N(0,1)
    norm_jitter: bool = False            # prefill: per-token factor U(0.5, 2)
    zipf_beta: float = 0.0               # Zipf-skewed bias amplitude (0 = none)
    zipf_s: float = 1.1
    layers: int = 1
    layer_corr: float = 0.0              # sweep: router rows correlated across layers
    down_scale: float = 1.0              # a power of two multiplying the down rows' draw
    batches: tuple = ()
    weight_seed: int | None = None       # seed of the layer's weights (default: seed)

    @property
    def expert_bytes(self) -> int:
        """Packed int4 bytes of one expert (gate, up, down)."""
        return 3 * self.ffn * self.hidden // 2

    @property
    def expert_scales(self) -> int:
        return 2 * self.ffn + self.hidden

    def layer_seed(self, layer: int) -> int:
        """Seed of the weights of layer ``layer``."""
        base = self.seed if self.weight_seed is None else self.weight_seed
        return base + layer

    def act_seed(self, layer: int) -> int:
        return self.seed + 1000 * layer


# Zipf amplitude of the prefill and sweep router bias.  Calibrated with the
# oracle's router on the prefill batch (2048 tokens): per-expert counts from 8
# to 472, median 55, so the busiest experts receive several hundred tokens and
# the quietest a handful ("from ~0 to several hundred").
ZIPF_BETA = 0.16
# Correlation of a sweep layer's router rows with the previous layer's.
# Calibrated with the oracle's router: on the same tokens, about 67-70% of a
# layer's top-8 choices are also in the previous layer's ("70% correlated";
# 69.6% in the calibration run, 0.67 on the 128 normalised tokens of the
# input-recipe test).
SWEEP_LAYER_CORR = 0.97
# The sweep's down rows are drawn at N(0, 0.02) x 1/32: each layer's residual
# update is then ~6% of the stream, as in a trained stack, so consecutive
# layers see nearly the same normalised input and route it alike (0.65 of the
# top-8 shared at 1/16, 0.68 at 1/64, 0.42 at full size, where every random
# layer rewrites the stream).  A power of two: the int4 codes are unchanged,
# only the row scales are.
SWEEP_DOWN_SCALE = 1.0 / 32

WORKLOADS = {
    "tiny": Workload("tiny", 256, 128, 8, 2, 4, 0),
    "decode": Workload("decode", 6144, 2048, 256, 8, 1, 1),
    "verify": Workload("verify", 6144, 2048, 256, 8, 4, 2, correlated_tokens=True,
                       weight_seed=1),
    "prefill": Workload("prefill", 6144, 2048, 256, 8, 2048, 3, norm_jitter=True,
                        zipf_beta=ZIPF_BETA, weight_seed=1),
    # the decode shape with 16 routed experts (~0.3 GB resident): a small case of
    # the same kernels for profiler captures; one forward still reads 170 MB
    "profile": Workload("profile", 6144, 2048, 16, 8, 1, 1),
    # the decode router's exact shape (hidden 6144, 256 experts, top-8, 1 token)
    # with a small expert FFN (~0.6 GB resident): a small case for capturing the
    # routing kernel
    "route_profile": Workload("route_profile", 6144, 256, 256, 8, 1, 1),
    # the verify batch (4 correlated tokens) on the decode shape with 16
    # routed experts: a small case for capturing the 4-token expert kernel
    "verify_profile": Workload("verify_profile", 6144, 2048, 16, 8, 4, 2, correlated_tokens=True,
                               weight_seed=1),
    # the prefill shape on 16 routed experts and 256 tokens (~0.3 GB of
    # weights, 128 tokens per expert on average): a small case for capturing
    # the grouped-GEMM kernels
    "prefill_profile": Workload("prefill_profile", 6144, 2048, 16, 8, 256, 3, norm_jitter=True,
                                weight_seed=1),
    # the decode shape with 64 routed experts and 32 tokens under the skewed
    # router bias (~1.2 GB resident): four tokens per expert on average, so the
    # 4-token tiles are about as full as those of a 128-token batch over 256
    # experts; a small case for capturing the expert kernel at that fill
    "batch_profile": Workload("batch_profile", 6144, 2048, 64, 8, 32, 100, zipf_beta=ZIPF_BETA),
    "sweep": Workload("sweep", 6144, 2048, 256, 8, 128, 100, zipf_beta=ZIPF_BETA, layers=8,
                      layer_corr=SWEEP_LAYER_CORR, down_scale=SWEEP_DOWN_SCALE, batches=(1, 8, 32, 128)),
}


def rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def normal(shape, std: float, *key: int) -> np.ndarray:
    """N(0, std^2) F32 draws by the Box-Muller transform of PCG64 uniforms
    (G. E. P. Box, M. E. Muller, 1958), in float32 throughout."""
    n = int(np.prod(shape))
    m = (n + 1) // 2
    g = rng(*key)
    u = g.random(m, dtype=np.float32)
    v = g.random(m, dtype=np.float32)
    np.subtract(np.float32(1.0), u, out=u)          # (0, 1]: log is finite
    np.log(u, out=u)
    np.multiply(u, np.float32(-2.0), out=u)
    np.sqrt(u, out=u)                               # radius
    np.multiply(v, np.float32(2.0 * np.pi), out=v)  # angle
    out = np.empty(2 * m, np.float32)
    np.cos(v, out=out[:m])                          # first half: r cos(theta)
    np.sin(v, out=out[m:])                          # second half: r sin(theta)
    out[:m] *= u
    out[m:] *= u
    a = out[:n].reshape(shape)
    if std != 1.0:
        a *= np.float32(std)
    return a


def router(wl: Workload, layer: int = 0):
    """Router weights [E][H] and bias [E] (F32) of one layer."""
    s = wl.layer_seed(layer)
    W = normal((wl.n_experts, wl.hidden), 0.02, s, _T_ROUTER_W)
    if wl.layer_corr and layer > 0:
        a = np.float32(wl.layer_corr)
        prev, _ = router(wl, layer - 1)
        fresh = normal((wl.n_experts, wl.hidden), 0.02, s, _T_ROUTER_W_FRESH)
        W = a * prev + np.float32(np.sqrt(1.0 - float(a) ** 2)) * fresh
        W = W.astype(np.float32)
    b = normal((wl.n_experts,), 0.01, s, _T_ROUTER_B)
    if wl.zipf_beta:
        perm = rng(s, _T_ZIPF_PERM).permutation(wl.n_experts)
        rank = np.empty(wl.n_experts, np.int64)
        rank[perm] = np.arange(wl.n_experts)
        b = (b + np.float32(wl.zipf_beta) * ((rank + 1.0) ** -wl.zipf_s).astype(np.float32))
        b = b.astype(np.float32)
    return W, b


def expert_f32(wl: Workload, e: int, layer: int = 0):
    """F32 weights of expert ``e`` (``e == n_experts`` is the shared expert):
    gate [F][H], up [F][H], down [H][F]."""
    a = expert_f32_rows(wl, e, layer)
    F, H = wl.ffn, wl.hidden
    return a[: F * H].reshape(F, H), a[F * H: 2 * F * H].reshape(F, H), a[2 * F * H:].reshape(H, F)


def expert_f32_rows(wl: Workload, e: int, layer: int = 0) -> np.ndarray:
    """Same draw as :func:`expert_f32`, as one [2F+H] list of rows in container
    order (gate rows, up rows, down rows); rows are ragged (H or F long), so this
    returns the flat F32 buffer."""
    s = wl.layer_seed(layer)
    a = normal((3 * wl.ffn * wl.hidden,), 0.02, s, _T_EXPERT, e)
    if wl.down_scale != 1.0:
        a[2 * wl.ffn * wl.hidden:] *= np.float32(wl.down_scale)
    return a


def activations(wl: Workload, step: int, n_tok: int | None = None, layer: int = 0) -> np.ndarray:
    """Input activations [T][H] (F32) of forward number ``step``."""
    T = wl.n_tok if n_tok is None else n_tok
    s = wl.act_seed(layer)
    x = normal((T, wl.hidden), 1.0, s, _T_X, step)
    if wl.correlated_tokens:
        noise = normal((T, wl.hidden), 1.0, s, _T_X_NOISE, step)
        x = (np.float32(0.7) * x[0:1] + np.float32(0.3) * noise).astype(np.float32)
    if wl.norm_jitter:
        j = rng(s, _T_JITTER, step).uniform(0.5, 2.0, size=(T, 1)).astype(np.float32)
        x = (x * j).astype(np.float32)
    return x


def parallel_map(fn, items, workers: int | None = None):
    """Map over items on a thread pool (numpy releases the GIL while drawing)."""
    workers = workers or min(16, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, items))
