"""Multi-layer decode sweep: 8 stacked GLM-5.2-shaped layers (~39 GB of int4
experts resident), x <- x + MoE(RMSNorm(x)) between layers, Zipf-skewed routing
correlated with the previous layer's.  Every layer is checked against the
oracle fed the GPU's input of that layer, on every token of the batch."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import OracleLayer, assert_float_close

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module")
def stack():
    import int4_routed_expert_f32_gb300 as coli
    from synth.device import build_device_layer
    torch.cuda.set_device(0)
    wl = synth.WORKLOADS["sweep"]
    layers = [build_device_layer(wl, layer=l) for l in range(wl.layers)]
    yield coli, wl, layers
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [8, 128])
def test_sweep_stack_matches_oracle_per_layer(stack, B):
    coli, wl, layers = stack
    coli.configure(wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.routed_scale, max(wl.batches))
    x = torch.from_numpy(synth.activations(wl, 3, n_tok=B)).cuda()
    for l, L in enumerate(layers):
        nxt = layers[l + 1] if l + 1 < len(layers) else None
        # the stacked-decode forward with the next layer's router weights and
        # shared expert prefetched into L2: identical to the plain residual
        # forward
        out = coli.layer_forward_residual_prefetch(
            x, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"], L["shared_w4"], L["shared_rs"],
            nxt["router_w"] if nxt else None, nxt["shared_w4"] if nxt else None)
        plain = coli.layer_forward_residual(x, L["router_w"], L["router_b"], L["expert_w4"], L["expert_rs"],
                                            L["shared_w4"], L["shared_rs"])
        assert coli.get_device_status() == coli.OK
        assert torch.equal(out, plain)
        xs = x.cpu().numpy()
        ref = OracleLayer(wl, layer=l)     # one layer's experts at a time (host memory)
        want = (xs + ref.forward(oracle.rmsnorm(xs))).astype(np.float32)
        del ref
        got = out.cpu().numpy()
        assert_float_close(got, want, what=f"layer {l}")
        np.testing.assert_array_equal(got, want, err_msg=f"layer {l}")
        x = out
