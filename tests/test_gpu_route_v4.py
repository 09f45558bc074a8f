"""GPU parity of the DeepSeek-V4-shaped gate (sqrt-softplus score, group-limited or
plain top-k, with and without bias) and of hash routing, through the C ABI, against the
oracle: expert ids bit for bit, weights within 2e-6 relative; and a whole layer with
the sqrt-softplus gate (DeepSeek-V3 shapes, fp8 and bf16) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import synth
from moe_expert_dispatch_route_gb300 import workloads as W

from helpers import check_close, np_f32, np_weights, ocfg
from test_gpu_layer import Layer

pytestmark = pytest.mark.gpu
DEV = "cuda"

V4 = W.DSV3.with_(name="dsv4_shaped", gate="sqrt_softplus")
CASES = [V4.with_(T=2048), V4.with_(T=2048, routing="zipf"), V4.with_(T=512, n_group=1, topk_group=1),
         V4.with_(T=300, num_experts=64, n_group=4, topk_group=2, top_k=6, routed_scale=2.5, renormalize=False)]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: f"E{w.num_experts}-G{w.n_group}-{w.routing}-T{w.T}")
@pytest.mark.parametrize("with_bias", [False, True])
def test_sqrt_softplus_route_matches_oracle(wl, with_bias):
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed) * 3
    bias = synth.bias(wl.num_experts, 0.05, 13) if with_bias else None
    ids_ref, w_ref = oracle.route(ocfg(wl), logits.numpy(), None if bias is None else bias.numpy())
    ids = torch.empty(wl.T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    B.moe_route(cfg, wl.T, logits.to(DEV), None if bias is None else bias.to(DEV), ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


def test_hash_routing_matches_oracle():
    wl = V4.with_(T=1000)
    cfg = B.config_of(wl)
    rng = np.random.default_rng(3)
    V = 5000
    table = np.stack([rng.permutation(wl.num_experts)[:wl.top_k] for _ in range(V)]).astype(np.int32)
    table[11, 3] = wl.num_experts + 1  # out of range: passed on with weight 0
    tids = rng.integers(0, V, wl.T).astype(np.int32)
    tids[[5, 6]] = [-3, V + 2]  # token ids outside the table
    tids[7] = 11
    logits = synth.logits(wl.T, wl.num_experts, "uniform", 4)
    ids_ref, w_ref = oracle.route_hash(ocfg(wl), logits.numpy(), tids, table)
    ids = torch.empty(wl.T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    B.moe_route_hash(cfg, wl.T, logits.to(DEV), torch.as_tensor(tids, device=DEV), torch.as_tensor(table, device=DEV),
                     ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)
    # hash routing needs the sqrt-softplus gate
    with pytest.raises(B.MoeError):
        B.moe_route_hash(B.config_of(W.DSV3), wl.T, logits.to(DEV), torch.as_tensor(tids, device=DEV),
                         torch.as_tensor(table, device=DEV), ids, w)


@pytest.mark.parametrize("wl", [V4.with_(T=40, num_experts=64, n_group=8, topk_group=4),
                                # bf16 at this width: x scaled so that |y| < 4, where one bf16
                                # rounding step (2^-6) is inside the stated max-abs 2e-2
                                V4.with_(T=24, num_experts=32, n_group=4, topk_group=2, dtype="bf16", x_std=0.25),
                                V4.with_(T=128)],
                         ids=lambda w: f"{w.dtype}-E{w.num_experts}-T{w.T}")
def test_layer_with_sqrt_softplus_gate_matches_oracle(wl):
    L = Layer(wl)
    got = L.run().result()
    L.close()
    assert got["err"] == 0
    if wl.T <= 64:
        ref = oracle.moe_layer(ocfg(wl), np_f32(L.logits), np_f32(L.x), np_weights(L.W), split=wl.split, align=128)
        assert np.array_equal(got["ids"], ref["ids"])
        check_close(got["y"], ref["y"], wl.dtype, "y")
    else:  # full DeepSeek-V3 width: every id, and the weights
        ids_ref, w_ref = oracle.route(ocfg(wl), np_f32(L.logits))
        assert np.array_equal(got["ids"], ids_ref)
        np.testing.assert_allclose(got["w"], w_ref, rtol=2e-6, atol=1e-7)
