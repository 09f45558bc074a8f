"""Pins for the oracle's stack of layers: the residual combine reproduces
(k+S+1)*x with identity experts, the stand-in block equals a numpy matmul with
residual, a stack whose experts output zero is the iterated stand-in, and the
two-ubatch split changes nothing."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import synth


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _cfg(H=128, I=128, E=8, S=1, k=2, dtype=oracle.BF16):
    return oracle.Config(hidden=H, inter=I, num_experts=E, num_shared=S, top_k=k, dtype=dtype)


def test_combine_resid_identity_experts():
    rng = np.random.default_rng(0)
    T, H, E, k, S = 21, 128, 8, 3, 0
    cfg = _cfg(H=H, E=E, S=S, k=k)
    x = _bf16(rng.standard_normal((T, H)))
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    p = oracle.plan(cfg, ids, align=1)
    d = oracle.dispatch(cfg, x, p["slot_of"], p["rows"])
    y = oracle.combine_resid(cfg, d["xe"], np.ones((T, k)), p["slot_of"], x)
    assert np.array_equal(y, _bf16(4.0 * x.astype(np.float64)))  # (k + S + 1) = 4


def _standin_ref(x, wa):
    return _bf16(x.astype(np.float64) + x.astype(np.float64) @ wa.astype(np.float64).T)


def test_standin_is_matmul_plus_residual():
    rng = np.random.default_rng(1)
    T, H = 17, 256
    x = _bf16(rng.standard_normal((T, H)))
    wa = _bf16(rng.standard_normal((H, H)) * 0.02)
    a = oracle.standin(_cfg(H=H), x, wa)
    ref = _standin_ref(x, wa)
    assert np.all(np.abs(a - ref) <= np.abs(ref) * 2.0 ** -7)
    assert np.mean(a == ref) > 0.99


def _layers(L, cfg, T, seed, zero_w2=False):
    out = []
    for l in range(L):
        W = synth.weights(cfg.num_experts + cfg.num_shared, cfg.hidden, cfg.inter,
                          {oracle.BF16: "bf16", oracle.FP8: "fp8"}[cfg.dtype], seed=seed + l)
        W = {k: (v.float().numpy() if v.dtype == torch.bfloat16 else v.numpy()) for k, v in W.items()}
        if zero_w2:
            for k in ("w2", "w2_q"):
                if k in W:
                    W[k] = np.zeros_like(W[k])
        wa = _bf16(np.random.default_rng(seed + 100 + l).standard_normal((cfg.hidden, cfg.hidden)) * 0.02)
        out.append(dict(wa=wa, logits=synth.logits(T, cfg.num_experts, "uniform", seed + l).numpy(), **W))
    return out


def test_stack_with_silent_experts_is_iterated_standin():
    cfg = _cfg(H=128, I=128, E=8, S=1, k=2)
    T, L = 10, 3
    layers = _layers(L, cfg, T, 3, zero_w2=True)
    x0 = synth.hidden(T, cfg.hidden, "bf16", 1.0, 3).float().numpy()
    got = oracle.moe_stack(cfg, x0, layers, split=5, align=1)["y"]
    ref = x0
    for ly in layers:
        ref = oracle.standin(cfg, ref, ly["wa"])
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP8])
def test_stack_split_invariance_and_layer_composition(dtype):
    cfg = _cfg(H=256, I=128, E=8, S=1, k=2, dtype=dtype)
    T, L = 12, 2
    layers = _layers(L, cfg, T, 7)
    x0 = synth.hidden(T, cfg.hidden, "bf16", 1.0, 7).float().numpy()
    a = oracle.moe_stack(cfg, x0, layers, split=0, align=1)
    b = oracle.moe_stack(cfg, x0, layers, split=5, align=8)
    assert a["status"] == 0 and np.array_equal(a["y"], b["y"])
    # layer by layer through the oracle's own steps
    x = x0
    for ly in layers:
        h = oracle.standin(cfg, x, ly["wa"])
        ids, w = oracle.route(cfg, ly["logits"])
        p = oracle.plan(cfg, ids, align=1)
        d = oracle.dispatch(cfg, h, p["slot_of"], p["rows"])
        ye = oracle.expert_ffn(cfg, p["counts"], p["offsets"], xe=d.get("xe"), xe_q=d.get("xe_q"),
                               xe_s=d.get("xe_s"), weights=ly)
        x = oracle.combine_resid(cfg, ye, w, p["slot_of"], h)
    assert np.array_equal(a["y"], x)
