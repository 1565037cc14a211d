"""Test-side helpers: oracle-packed experts from the seeded draws, and the
parity tolerance."""
from __future__ import annotations

import numpy as np

import synth


def oracle_expert(wl: synth.Workload, e: int, layer: int = 0, wbits: int = 4):
    """(weight bytes [3FH*wbits/8], row scales [2F+H]) of expert e (E =
    shared), packed by the oracle's own converter from the seeded F32 draw
    into the int4 (wbits 4) or int8 (wbits 8) container."""
    import oracle
    F, H = wl.ffn, wl.hidden
    flat = synth.expert_f32_rows(wl, e, layer)
    pack = oracle.pack_int4_rows if wbits == 4 else oracle.pack_int8_rows
    pg, sg = pack(flat[:F * H].reshape(F, H))
    pu, su = pack(flat[F * H:2 * F * H].reshape(F, H))
    pd, sd = pack(flat[2 * F * H:].reshape(H, F))
    return (np.concatenate([pg.ravel(), pu.ravel(), pd.ravel()]).view(np.uint8),
            np.concatenate([sg, su, sd]))


class OracleLayer:
    """Lazily packs only the experts a sample touches (several at a time, on
    a thread pool: the draws and the oracle's C packer release the GIL).

    ``cache``: an expert cache to share with other instances over the same
    weights (the decode, verify and prefill workloads share one layer's
    experts and differ only in the router bias)."""

    def __init__(self, wl: synth.Workload, layer: int = 0, cache: dict | None = None, wbits: int = 4):
        self.wl = wl
        self.layer = layer
        self.wbits = wbits
        self.W, self.b = synth.router(wl, layer)
        self._cache = {} if cache is None else cache
        self.shared = self.expert(wl.n_experts)

    def expert(self, e):
        if e not in self._cache:
            self._cache[e] = oracle_expert(self.wl, e, self.layer, self.wbits)
        return self._cache[e]

    def prefetch(self, experts):
        todo = sorted(set(int(e) for e in experts) - set(self._cache))
        if todo:
            packed = synth.parallel_map(lambda e: oracle_expert(self.wl, e, self.layer, self.wbits), todo)
            for e, v in zip(todo, packed):
                self._cache[e] = v

    def forward(self, x, intermediates=False):
        import oracle
        wl = self.wl
        idx, _ = oracle.route(x, self.W, self.b, wl.top_k, wl.routed_scale)
        need = set(int(v) for v in idx.ravel())
        self.prefetch(need)
        w4 = [None] * wl.n_experts
        rs = [None] * wl.n_experts
        for e in need:
            w4[e], rs[e] = self.expert(e)
        return oracle.moe_forward(x, self.W, self.b, w4, rs, self.shared[0], self.shared[1],
                                  wl.hidden, wl.ffn, wl.top_k, wl.routed_scale,
                                  intermediates=intermediates, wbits=self.wbits)


# Float outputs must agree within max|err| <= 1e-3 * rms(oracle output).
FLOAT_TOL = 1e-3


def assert_float_close(got, want, tol=FLOAT_TOL, what="out"):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    rms = float(np.sqrt(np.mean(want ** 2)))
    err = float(np.max(np.abs(got - want))) if want.size else 0.0
    assert err <= tol * rms, f"{what}: max|err| {err:.3e} > {tol} * rms {rms:.3e} ({err / max(rms, 1e-30):.2e})"
    return err / max(rms, 1e-30)
