"""The allocation-free router entry point, checked against the configured one
and against the oracle's router.

Callers that cannot allocate device memory (running under another runtime's
allocator, with all device memory reserved up front, or in loops that forbid
allocation) use coli_moe_route_noalloc: its scratch is a static device array of
the library.  This file is collected last so that a failure here cannot stop
the rest of the suite from running first; it also passes on its own, in a fresh
process.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("wl_name,T", [("decode", 1), ("verify", 4), ("prefill", 64), ("tiny", 3)])
def test_route_noalloc_matches_configured_router(wl_name, T):
    import int4_routed_expert_f32_gb300 as coli
    import oracle
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS[wl_name]
    W, b = synth.router(wl)
    Wd, bd = _cuda(W), _cuda(b)
    for call in range(2):   # two calls in a row share the static scratch
        xh = synth.activations(wl, 300 + call, n_tok=T)
        x = _cuda(xh)
        idx_s = torch.empty((T, wl.top_k), dtype=torch.int32, device="cuda")
        w_s = torch.empty((T, wl.top_k), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        coli.route_noalloc(x, Wd, bd, wl.hidden, wl.n_experts, wl.top_k, wl.routed_scale, idx=idx_s, w=w_s)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        if call == 1:
            # after the first call (which may commit the module's memory),
            # the entry point takes no device memory
            assert free1 == free0, (free0, free1)
        # the oracle's router on the same inputs: identical indices and weights
        ridx, rw = oracle.route(xh, W, b, wl.top_k, wl.routed_scale)
        np.testing.assert_array_equal(idx_s.cpu().numpy(), ridx)
        np.testing.assert_array_equal(w_s.cpu().numpy(), rw)
        coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, 64)
        idx_r, w_r = coli.dbg_route(x, Wd, bd, wl.top_k)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(idx_s.cpu().numpy(), idx_r.cpu().numpy())
        ws, wr = w_s.cpu().numpy().astype(np.float64), w_r.cpu().numpy().astype(np.float64)
        rms = float(np.sqrt(np.mean(wr ** 2)))
        assert float(np.max(np.abs(ws - wr))) <= 1e-3 * rms
        np.testing.assert_array_equal(ws, wr)      # same kernels, same order: identical


def test_route_noalloc_rejects_oversize():
    import int4_routed_expert_f32_gb300 as coli
    wl = synth.WORKLOADS["decode"]
    W, b = synth.router(wl)
    x = torch.zeros((coli.STATIC_MAX_TOK + 1, wl.hidden), dtype=torch.float32, device="cuda")
    with pytest.raises(coli.ColiError) as ei:
        coli.route_noalloc(x, _cuda(W), _cuda(b), wl.hidden, wl.n_experts, wl.top_k, wl.routed_scale)
    assert ei.value.code == coli.E_INVAL
