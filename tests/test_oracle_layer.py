"""Pins for the oracle's dispatch, expert FFN, combine and the whole layer:
identity experts reproduce (k+S)*x, E=1/k=1 reduces to a dense SwiGLU MLP computed
with numpy matmuls, the per-token brute force equals the permuted layer, the
micro-batch split and the capacity layout change nothing, and relabelling experts
changes nothing."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import synth

QG = 128


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _cfg(H, I, E, S, k, dtype, renorm=1):
    return oracle.Config(hidden=H, inter=I, num_experts=E, num_shared=S, top_k=k,
                         renormalize=renorm, dtype=dtype)


def _np_weights(w):
    return {k: v.cpu().numpy() if v.dtype != torch.bfloat16 else v.float().numpy()
            for k, v in w.items()}


def _dequant_weights(W, H, I):
    """Dense fp64 weights: fp8 codes decoded by torch's float8 view times block scales."""
    if "w13" in W:
        return W["w13"].astype(np.float64), W["w2"].astype(np.float64)
    dec = lambda q: torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    rep = lambda s: np.repeat(np.repeat(s, QG, axis=-2), QG, axis=-1)
    return dec(W["w13_q"]) * rep(W["w13_s"]), dec(W["w2_q"]) * rep(W["w2_s"])


@pytest.mark.parametrize("dtype,k,S", [(oracle.F32, 3, 0), (oracle.BF16, 2, 0), (oracle.BF16, 4, 0),
                                       (oracle.BF16, 2, 2)])
def test_dispatch_combine_identity_experts_give_k_times_x(dtype, k, S):
    rng = np.random.default_rng(1)
    T, H, E = 33, 256, 8
    cfg = _cfg(H, 128, E, S, k, dtype)
    x = rng.standard_normal((T, H)).astype(np.float32)
    if dtype == oracle.BF16:
        x = _bf16(x)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    p = oracle.plan(cfg, ids, align=4)
    d = oracle.dispatch(cfg, x, p["slot_of"], p["rows"])
    ye = d["xe"]  # identity experts
    y = oracle.combine(cfg, ye, np.ones((T, k)), p["slot_of"])
    ref = (k + S) * x.astype(np.float64)
    if dtype == oracle.F32:
        np.testing.assert_allclose(y, ref.astype(np.float32), rtol=0, atol=0)
    else:
        # one bf16 rounding of an exact sum; exact when k+S is a power of two
        if (k + S) & (k + S - 1) == 0:
            assert np.array_equal(y, _bf16(ref))
        else:
            np.testing.assert_allclose(y, ref, rtol=2.0 ** -8)


def test_dispatch_fp8_rows_are_per_token_quantisation():
    rng = np.random.default_rng(2)
    T, H, E, k = 9, 256, 4, 2
    cfg = _cfg(H, 128, E, 0, k, oracle.FP8)
    x = _bf16(rng.standard_normal((T, H)) * 4)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    p = oracle.plan(cfg, ids, align=1)
    d = oracle.dispatch(cfg, x, p["slot_of"], p["rows"])
    for t in range(T):
        q, s = oracle.quant_row_fp8(x[t])
        for j in range(k):
            r = p["slot_of"][t, j]
            assert np.array_equal(d["xe_q"][r], q) and np.array_equal(d["xe_s"][r], s)


def _dense_swiglu(x, w13, w2, I, dtype):
    """Textbook dense SwiGLU MLP with numpy matmuls: silu(x Wg^T) * (x Wu^T) then W2."""
    g = x @ w13[:I].T
    u = x @ w13[I:].T
    h = g / (1.0 + np.exp(-g)) * u
    if dtype == oracle.BF16:
        h = _bf16(h.astype(np.float32)).astype(np.float64)
    elif dtype == oracle.F32:
        h = h.astype(np.float32).astype(np.float64)
    else:
        hq = np.zeros_like(h)
        for t in range(h.shape[0]):
            q, s = oracle.quant_row_fp8(h[t].astype(np.float32))
            dec = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
            hq[t] = dec * np.repeat(s, QG)
        h = hq
    return h @ w2.T


@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16, oracle.FP8])
def test_single_expert_top1_is_dense_swiglu_mlp(dtype):
    T, H, I = 24, 256, 256
    dstr = {oracle.F32: "f32", oracle.BF16: "bf16", oracle.FP8: "fp8"}[dtype]
    W = _np_weights(synth.weights(1, H, I, dstr, seed=3))
    x = synth.hidden(T, H, "f32" if dtype == oracle.F32 else "bf16", seed=3).float().numpy()
    cfg = _cfg(H, I, 1, 0, 1, dtype)
    logits = np.zeros((T, 1), np.float32)
    out = oracle.moe_layer(cfg, logits, x, W, align=1)
    assert np.all(out["ids"] == 0) and np.allclose(out["w"], 1.0)
    w13, w2 = _dequant_weights(W, H, I)
    xin = x.astype(np.float64)
    if dtype == oracle.FP8:
        xin = np.zeros_like(xin)
        for t in range(T):
            q, s = oracle.quant_row_fp8(x[t])
            xin[t] = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy() * np.repeat(s, QG)
    ref = _dense_swiglu(xin, w13[0], w2[0], I, dtype)
    if dtype == oracle.F32:
        np.testing.assert_allclose(out["y"], ref, rtol=1e-6, atol=1e-9)
    else:
        refb = _bf16(ref.astype(np.float32))
        # at most one bf16 step apart (summation order inside double differs)
        step = np.abs(refb) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(out["y"] - refb) <= step)
        assert np.mean(out["y"] == refb) > 0.99


def test_shared_experts_add_their_dense_mlps():
    T, H, I, E, S, k = 10, 128, 128, 4, 2, 1
    W = _np_weights(synth.weights(E + S, H, I, "f32", seed=4))
    x = synth.hidden(T, H, "f32", seed=4).numpy()
    cfg = _cfg(H, I, E, S, k, oracle.F32)
    logits = synth.logits(T, E, seed=4).numpy()
    out = oracle.moe_layer(cfg, logits, x, W, align=1)
    w13, w2 = _dequant_weights(W, H, I)
    ref = np.zeros((T, H))
    for t in range(T):
        e = out["ids"][t, 0]
        ref[t] += out["w"][t, 0] * _dense_swiglu(x[t:t + 1].astype(np.float64), w13[e], w2[e], I,
                                                 oracle.F32)[0].astype(np.float32)
        for s in range(S):
            ref[t] += _dense_swiglu(x[t:t + 1].astype(np.float64), w13[E + s], w2[E + s], I,
                                    oracle.F32)[0].astype(np.float32)
    np.testing.assert_allclose(out["y"], ref, rtol=1e-6, atol=1e-9)


def _small_layer(dtype, T=40, H=256, I=256, E=8, S=1, k=2, routing="uniform", seed=5):
    dstr = {oracle.F32: "f32", oracle.BF16: "bf16", oracle.FP8: "fp8"}[dtype]
    W = _np_weights(synth.weights(E + S, H, I, dstr, seed=seed))
    x = synth.hidden(T, H, "f32" if dtype == oracle.F32 else "bf16", seed=seed).float().numpy()
    logits = synth.logits(T, E, routing, seed=seed).numpy()
    return _cfg(H, I, E, S, k, dtype), logits, x, W


@pytest.mark.parametrize("dtype", [oracle.F32, oracle.BF16, oracle.FP8])
def test_per_token_brute_force_equals_permuted_layer(dtype):
    cfg, logits, x, W = _small_layer(dtype)
    out = oracle.moe_layer(cfg, logits, x, W, align=16)
    for t in range(x.shape[0]):
        yt = oracle.token_output(cfg, x[t], out["ids"][t], out["w"][t], W)
        assert np.array_equal(yt, out["y"][t]), t


@pytest.mark.parametrize("dtype", [oracle.BF16, oracle.FP8])
def test_split_and_capacity_layout_do_not_change_output(dtype):
    cfg, logits, x, W = _small_layer(dtype, T=41, routing="zipf")
    base = oracle.moe_layer(cfg, logits, x, W, align=128)
    for split in (1, 20, 21, 40):
        s = oracle.moe_layer(cfg, logits, x, W, split=split, align=8)
        assert np.array_equal(s["y"], base["y"]) and np.array_equal(s["ids"], base["ids"])
    cap = oracle.moe_layer(cfg, logits, x, W, split=21, capacity=21)
    assert cap["status"] == oracle.OK and np.array_equal(cap["y"], base["y"])
    small = oracle.moe_layer(cfg, logits, x, W, capacity=3)
    assert small["status"] == oracle.CAPACITY


def test_expert_relabelling_leaves_output_unchanged():
    cfg, logits, x, W = _small_layer(oracle.BF16, S=0, seed=6)
    E = cfg.num_experts
    perm = np.random.default_rng(0).permutation(E)
    # expert e becomes expert perm[e]: move its logit column and its weights
    logits2 = np.empty_like(logits)
    logits2[:, perm] = logits
    W2 = {k: np.empty_like(v) for k, v in W.items()}
    for k_, v in W.items():
        W2[k_][perm] = v
    a = oracle.moe_layer(cfg, logits, x, W, align=1)
    b = oracle.moe_layer(cfg, logits2, x, W2, align=1)
    assert np.array_equal(b["ids"], perm[a["ids"]])
    assert np.array_equal(a["y"], b["y"])


def test_grouped_sigmoid_layer_runs_and_matches_brute_force():
    T, H, I, E, S, k = 6, 128, 128, 32, 1, 4
    cfg = oracle.Config(hidden=H, inter=I, num_experts=E, num_shared=S, top_k=k,
                        gate=oracle.GATE_SIGMOID_GROUPED, renormalize=1, n_group=4, topk_group=2,
                        routed_scale=2.5, dtype=oracle.FP8)
    W = _np_weights(synth.weights(E + S, H, I, "fp8", seed=8))
    x = synth.hidden(T, H, "bf16", seed=8).float().numpy()
    logits = synth.logits(T, E, "zipf", seed=8).numpy()
    out = oracle.moe_layer(cfg, logits, x, W, split=3, align=1)
    assert out["status"] == oracle.OK
    np.testing.assert_allclose(out["w"].sum(1), 2.5, rtol=1e-12)
    for t in range(T):
        assert np.array_equal(oracle.token_output(cfg, x[t], out["ids"][t], out["w"][t], W), out["y"][t])
