"""GPU parity of each step of the layer against the CPU oracle, through the C ABI.

Inputs are the seeded synthetic inputs of each workload (or oracle outputs used as
inputs for the later steps); the expected values come from the oracle only.
Indices, counts, permutations and quantised bytes are compared bit for bit; floating
point within the stated tolerances."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import synth
from moe_expert_dispatch_route_gb300 import workloads as W

from helpers import check_close, np_f32, np_weights, ocfg

pytestmark = pytest.mark.gpu
DEV = "cuda"

ROUTE_CASES = [W.TINY, W.QWEN3_DECODE, W.QWEN3_DECODE.with_(routing="zipf"), W.DSV2LITE,
               W.DSV2LITE.with_(T=4096), W.QWEN3_PREFILL, W.DSV3, W.DSV3.with_(routing="zipf"),
               W.DSV3.with_(T=16384)]


@pytest.mark.parametrize("wl", ROUTE_CASES, ids=lambda w: f"{w.name}-{w.T}-{w.routing}")
def test_route_matches_oracle(wl):
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
    ids_ref, w_ref = oracle.route(ocfg(wl), logits.numpy())
    ids = torch.empty(wl.T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    B.moe_route(cfg, wl.T, logits.to(DEV), None, ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


def test_route_grouped_with_bias_and_scale():
    wl = W.DSV3.with_(T=512, routed_scale=2.5, renormalize=True)
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, "uniform", 11)
    bias = synth.bias(wl.num_experts, 0.05, 11)
    ids_ref, w_ref = oracle.route(ocfg(wl), logits.numpy(), bias.numpy())
    ids = torch.empty(wl.T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    B.moe_route(cfg, wl.T, logits.to(DEV), bias.to(DEV), ids, w)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=2e-6, atol=1e-7)


def test_route_ties_pick_lower_id():
    wl = W.QWEN3_DECODE.with_(T=64)
    logits = torch.zeros(64, 128)
    logits[:, 5] = 1.0
    logits[:, 77] = 1.0
    ids = torch.empty(64, 8, dtype=torch.int32, device=DEV)
    w = torch.empty(64, 8, device=DEV)
    B.moe_route(B.config_of(wl), 64, logits.to(DEV), None, ids, w)
    ids_ref, _ = oracle.route(ocfg(wl), logits.numpy())
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert ids_ref[0].tolist() == [5, 77, 0, 1, 2, 3, 4, 6]


def _plan_gpu(wl, ids_np, T, capacity, align, ws_extra=0):
    cfg = B.config_of(wl)
    NE, kk = wl.num_experts + wl.num_shared, wl.top_k + wl.num_shared
    rows = B.moe_plan_rows(cfg, T, capacity, align)
    counts = torch.full((NE,), -5, dtype=torch.int32, device=DEV)
    offsets = torch.full((NE + 1,), -5, dtype=torch.int32, device=DEV)
    slot_of = torch.full((max(T, 1), kk), -5, dtype=torch.int32, device=DEV)
    token_of = torch.full((max(rows, 1),), -5, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = B.moe_plan_workspace_size(cfg, T)
    ws = torch.empty(max(wsb, 4) // 4 + ws_extra, dtype=torch.int32, device=DEV)
    B.moe_plan(cfg, T, torch.as_tensor(ids_np, device=DEV), capacity, align, counts, offsets, slot_of,
               token_of, err, ws, wsb)
    torch.cuda.synchronize()
    return dict(counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(), slot_of=slot_of.cpu().numpy()[:T],
                token_of=token_of.cpu().numpy(), err=int(err.item()))


PLAN_CASES = [(W.TINY, 0, 1), (W.QWEN3_DECODE, 0, 128), (W.QWEN3_DECODE, 128, 128), (W.DSV2LITE, 0, 128),
              (W.DSV2LITE.with_(T=4096), 0, 128), (W.DSV2LITE.with_(T=4096), 4096, 1),
              (W.QWEN3_PREFILL, 0, 128), (W.DSV3.with_(T=16384), 0, 128), (W.DSV3, 128, 1),
              (W.DSV3.with_(T=1), 0, 128), (W.QWEN3_DECODE.with_(T=1001, routing="zipf"), 0, 64)]


@pytest.mark.parametrize("wl,capacity,align", PLAN_CASES,
                         ids=lambda v: f"{v.name}-{v.T}" if hasattr(v, "name") else str(v))
def test_plan_matches_oracle_bit_exact(wl, capacity, align):
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
    ids, _ = oracle.route(ocfg(wl), logits.numpy())
    ref = oracle.plan(ocfg(wl), ids, capacity, align)
    got = _plan_gpu(wl, ids, wl.T, capacity, align)
    assert got["err"] == 0 and ref["status"] == 0
    assert np.array_equal(got["counts"], ref["counts"])
    assert np.array_equal(got["offsets"], ref["offsets"])
    assert np.array_equal(got["slot_of"], ref["slot_of"])
    assert np.array_equal(got["token_of"][: ref["rows"]], ref["token_of"])


def test_plan_empty_batch_writes_zero_counts():
    wl = W.DSV2LITE
    got = _plan_gpu(wl, np.zeros((0, wl.top_k), np.int32), 0, 0, 128)
    assert np.all(got["counts"] == 0) and np.all(got["offsets"] == 0) and got["err"] == 0


def test_plan_reports_capacity_overflow_and_bad_index():
    wl = W.QWEN3_DECODE
    logits = synth.logits(wl.T, wl.num_experts, "zipf", 3)
    ids, _ = oracle.route(ocfg(wl), logits.numpy())
    ref = oracle.plan(ocfg(wl), ids, capacity=8)
    got = _plan_gpu(wl, ids, wl.T, 8, 1)
    assert ref["status"] == oracle.CAPACITY and got["err"] == 6
    assert np.array_equal(got["slot_of"], ref["slot_of"])
    assert np.array_equal(got["counts"], ref["counts"])
    bad = ids.copy()
    bad[3, 2] = 128
    bad[17, 0] = -1
    ref = oracle.plan(ocfg(wl), bad, 0, 128)
    got = _plan_gpu(wl, bad, wl.T, 0, 128)
    assert ref["status"] == oracle.BAD_INDEX and got["err"] == 7
    assert np.array_equal(got["slot_of"], ref["slot_of"])
    assert np.array_equal(got["counts"], ref["counts"])


DISPATCH_CASES = [W.TINY, W.QWEN3_DECODE, W.DSV2LITE, W.QWEN3_PREFILL.with_(T=1024), W.DSV3]


@pytest.mark.parametrize("wl", DISPATCH_CASES, ids=lambda w: w.name)
def test_dispatch_matches_oracle_bit_exact(wl):
    cfg = B.config_of(wl)
    x = synth.hidden(wl.T, wl.hidden, wl.dtype, wl.x_std, wl.seed)
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
    ids, _ = oracle.route(ocfg(wl), logits.numpy())
    p = oracle.plan(ocfg(wl), ids, 0, 128)
    ref = oracle.dispatch(ocfg(wl), np_f32(x), p["slot_of"], p["rows"])
    rows = p["rows"]
    used = p["token_of"] >= 0
    H = wl.hidden
    if wl.dtype == "fp8":
        xe = torch.zeros(rows, H, dtype=torch.uint8, device=DEV)
        xs = torch.zeros(rows, H // 128, dtype=torch.float32, device=DEV)
        B.moe_dispatch(cfg, wl.T, x.to(DEV), torch.as_tensor(p["slot_of"], device=DEV), xe, xs)
        torch.cuda.synchronize()
        assert np.array_equal(xe.cpu().numpy()[used], ref["xe_q"][used])
        assert np.array_equal(xs.cpu().numpy()[used], ref["xe_s"][used])
        # column-major scales (the layer's internal layout), with a stride above rows
        ld = rows + 7
        xsc = torch.zeros(H // 128, ld, dtype=torch.float32, device=DEV)
        xe.zero_()
        B.moe_dispatch(cfg, wl.T, x.to(DEV), torch.as_tensor(p["slot_of"], device=DEV), xe, xsc, xe_scale_ld=ld)
        torch.cuda.synchronize()
        assert np.array_equal(xe.cpu().numpy()[used], ref["xe_q"][used])
        assert np.array_equal(xsc.cpu().numpy()[:, :rows].T[used], ref["xe_s"][used])
    else:
        tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        xe = torch.zeros(rows, H, dtype=tdt, device=DEV)
        B.moe_dispatch(cfg, wl.T, x.to(DEV), torch.as_tensor(p["slot_of"], device=DEV), xe)
        torch.cuda.synchronize()
        assert np.array_equal(np_f32(xe)[used], ref["xe"][used])


FFN_CASES = [W.TINY, W.QWEN3_DECODE.with_(T=48), W.DSV2LITE.with_(T=40), W.QWEN3_PREFILL.with_(T=40),
             W.DSV3.with_(T=6, num_experts=32, n_group=8, topk_group=4)]


def _ffn_inputs(wl, align=128, capacity=0):
    x = synth.hidden(wl.T, wl.hidden, wl.dtype, wl.x_std, wl.seed)
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
    W_ = synth.weights(wl.num_experts + wl.num_shared, wl.hidden, wl.inter, wl.dtype, wl.w_std, wl.seed)
    ids, w = oracle.route(ocfg(wl), logits.numpy())
    p = oracle.plan(ocfg(wl), ids, capacity, align)
    d = oracle.dispatch(ocfg(wl), np_f32(x), p["slot_of"], p["rows"])
    return x, W_, ids, w, p, d


def _run_ffn_gpu(wl, W_, p, d, max_ctas=0, scale_ld=0):
    cfg = B.config_of(wl)
    rows = p["rows"]
    H = wl.hidden
    if wl.dtype == "fp8":
        xe = torch.as_tensor(d["xe_q"], device=DEV)
        xs = torch.as_tensor(d["xe_s"], device=DEV)
        if scale_ld:  # column-major: scale(row, g) at g * scale_ld + row
            xsc = torch.zeros(H // 128, scale_ld, dtype=torch.float32, device=DEV)
            xsc[:, :rows] = xs.t()
            xs = xsc
        w13, w13s, w2, w2s = (W_[k].to(DEV) for k in ("w13_q", "w13_s", "w2_q", "w2_s"))
        ye = torch.zeros(rows, H, dtype=torch.bfloat16, device=DEV)
    else:
        tdt = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        xe = torch.as_tensor(d["xe"], device=DEV).to(tdt)
        xs = None
        w13, w2 = W_["w13"].to(DEV), W_["w2"].to(DEV)
        w13s = w2s = None
        ye = torch.zeros(rows, H, dtype=tdt, device=DEV)
    wsb = B.moe_ffn_workspace_size(cfg, rows)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.moe_expert_ffn(cfg, torch.as_tensor(p["counts"], device=DEV), torch.as_tensor(p["offsets"], device=DEV),
                     rows, xe, xs, w13, w13s, w2, w2s, ye, ws, wsb, err, max_ctas, xe_scale_ld=scale_ld)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return np_f32(ye)


@pytest.mark.parametrize("wl", [w for w in FFN_CASES if w.dtype == "fp8"], ids=lambda w: w.name)
def test_expert_ffn_scale_layouts_agree(wl):
    """Row-major and column-major activation scales give the same ye, bit for bit."""
    x, W_, ids, w, p, d = _ffn_inputs(wl)
    a = _run_ffn_gpu(wl, W_, p, d)
    b = _run_ffn_gpu(wl, W_, p, d, scale_ld=p["rows"] + 5)
    used = p["token_of"] >= 0
    assert np.array_equal(a[used], b[used])


@pytest.mark.parametrize("wl", FFN_CASES, ids=lambda w: w.name)
def test_expert_ffn_matches_oracle(wl):
    x, W_, ids, w, p, d = _ffn_inputs(wl)
    ye = _run_ffn_gpu(wl, W_, p, d)
    ref = oracle.expert_ffn(ocfg(wl), p["counts"], p["offsets"], xe=d.get("xe"), xe_q=d.get("xe_q"),
                            xe_s=d.get("xe_s"), weights=np_weights(W_))
    used = p["token_of"] >= 0
    check_close(ye[used], ref[used], wl.dtype, "ye")


def test_expert_ffn_capacity_layout_and_sm_budget():
    wl = W.DSV2LITE.with_(T=24)
    x, W_, ids, w, p, d = _ffn_inputs(wl, capacity=24)
    ye = _run_ffn_gpu(wl, W_, p, d, max_ctas=7)
    ref = oracle.expert_ffn(ocfg(wl), p["counts"], p["offsets"], xe=d.get("xe"), weights=np_weights(W_))
    used = p["token_of"] >= 0
    check_close(ye[used], ref[used], wl.dtype, "ye")


COMBINE_CASES = [W.TINY, W.QWEN3_DECODE, W.DSV2LITE, W.DSV3]


@pytest.mark.parametrize("wl", COMBINE_CASES, ids=lambda w: w.name)
def test_combine_matches_oracle(wl):
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
    ids, w = oracle.route(ocfg(wl), logits.numpy())
    p = oracle.plan(ocfg(wl), ids, 0, 128)
    io = "f32" if wl.dtype == "f32" else "bf16"
    ye = synth.hidden(p["rows"], wl.hidden, io, 1.0, wl.seed + 100)
    w32 = w.astype(np.float32)
    ref = oracle.combine(ocfg(wl), np_f32(ye), w32.astype(np.float64), p["slot_of"])
    y = torch.zeros(wl.T, wl.hidden, dtype=ye.dtype, device=DEV)
    B.moe_combine(cfg, wl.T, ye.to(DEV), torch.as_tensor(w32, device=DEV),
                  torch.as_tensor(p["slot_of"], device=DEV), y)
    torch.cuda.synchronize()
    got = np_f32(y)
    if wl.dtype == "f32":
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)
    else:
        # one bf16 rounding (one step of the result) plus the fp32 accumulation error
        # over k+S terms (bounded by 2^-20 of the sum of the terms' magnitudes)
        Y = np_f32(ye).astype(np.float64)
        kk = p["slot_of"].shape[1]
        absum = sum(np.abs((w32[:, j, None] if j < wl.top_k else 1.0) * Y[p["slot_of"][:, j]]) for j in range(kk))
        bound = np.abs(ref) * 2.0 ** -7 + absum * 2.0 ** -20
        assert np.all(np.abs(got - ref) <= bound)


def test_combine_skips_unplaced_entries():
    wl = W.QWEN3_DECODE.with_(T=32)
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, "zipf", 9)
    ids, w = oracle.route(ocfg(wl), logits.numpy())
    p = oracle.plan(ocfg(wl), ids, capacity=2)
    assert p["status"] == oracle.CAPACITY
    ye = synth.hidden(p["rows"], wl.hidden, "bf16", 1.0, 5)
    ref = oracle.combine(ocfg(wl), np_f32(ye), w, p["slot_of"])
    y = torch.zeros(wl.T, wl.hidden, dtype=torch.bfloat16, device=DEV)
    B.moe_combine(cfg, wl.T, ye.to(DEV), torch.as_tensor(w.astype(np.float32), device=DEV),
                  torch.as_tensor(p["slot_of"], device=DEV), y)
    torch.cuda.synchronize()
    check_close(np_f32(y), ref, "bf16", "y")


def test_plan_without_token_of_gives_the_same_plan():
    wl = W.DSV2LITE.with_(T=4096)
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
    ids, _ = oracle.route(ocfg(wl), logits.numpy())
    ref = _plan_gpu(wl, ids, wl.T, 0, 128)
    NE, kk = wl.num_experts + wl.num_shared, wl.top_k + wl.num_shared
    counts = torch.zeros(NE, dtype=torch.int32, device=DEV)
    offsets = torch.zeros(NE + 1, dtype=torch.int32, device=DEV)
    slot_of = torch.zeros(wl.T, kk, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    wsb = B.moe_plan_workspace_size(cfg, wl.T)
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    B.moe_plan(cfg, wl.T, torch.as_tensor(ids, device=DEV), 0, 128, counts, offsets, slot_of, None, err, ws, wsb)
    torch.cuda.synchronize()
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(slot_of.cpu().numpy(), ref["slot_of"])


@pytest.mark.parametrize("wl", [W.QWEN3_DECODE.with_(T=64), W.DSV3.with_(T=64)], ids=lambda w: w.name)
def test_route_nan_logits_give_valid_ids(wl):
    """Rows of NaN logits (and partly NaN rows) still select k distinct experts in
    [0, E): the gates rank a NaN as -inf, so no id can leave the range (the weights of
    such rows are unspecified)."""
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, "uniform", 5)
    logits[: wl.T // 2] = float("nan")
    logits[wl.T // 2:, ::3] = float("nan")
    ids = torch.full((wl.T, wl.top_k), -1, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    B.moe_route(cfg, wl.T, logits.to(DEV), None, ids, w)
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    assert got.min() >= 0 and got.max() < wl.num_experts
    assert all(len(set(r)) == wl.top_k for r in got.tolist())
    # the partly-NaN rows choose among their finite logits
    assert np.all(got[wl.T // 2:] % 3 != 0)
