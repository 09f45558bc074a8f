"""The staged combine kernel (bulk async copies of the expert-output rows through
shared-memory stages) and the dispatch kernels on the shapes that exercise their
bookkeeping, against the oracle, through the C ABI:

* rows cut into several column chunks with a ragged last chunk (bf16, fp32, and fp8,
  whose 1024-element dispatch slices leave a ragged last slice of whole 1x128 groups);
* 32 entries per token (the most a combine stage holds; the most a scale-store pass of
  the fp8 dispatch covers is 16, so two rounds);
* CTA budgets of 1 and 3 (each combine CTA's unit range wraps its stage ring many times;
  each dispatch warp walks many items) and fewer units than CTAs: results bit-identical
  to the default grid;
* the failure path: with the wait-injection hook on, moe_combine leaves its work undone
  and reports MOE_ERR_TIMEOUT through moe_comm_error; the next call gives the same bytes
  as before."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import synth
from moe_expert_dispatch_route_gb300 import workloads as W

from helpers import np_f32, ocfg

pytestmark = pytest.mark.gpu
DEV = "cuda"
TIMEOUT = 8  # MOE_ERR_TIMEOUT

CASES = [
    # combine: 16528-byte rows -> 5 chunks of 3312 bytes, the last 3280; dispatch: 8
    # slices of 1024 elements and a last one of 72 (9 vectors)
    W.Workload("chunks_bf16", T=70, hidden=8264, inter=128, num_experts=16, num_shared=1, top_k=4, dtype="bf16",
               seed=41),
    # fp32 rows of 8368 bytes -> 3 chunks, the last ragged
    W.Workload("chunks_f32", T=33, hidden=2092, inter=128, num_experts=9, num_shared=0, top_k=3, dtype="f32",
               seed=42),
    # fp8: 65 groups -> 8 slices of 8 groups and one of 1 group (one half-warp)
    W.Workload("chunks_fp8", T=45, hidden=8320, inter=128, num_experts=24, num_shared=1, top_k=5, dtype="fp8",
               seed=43),
    # 32 entries per token
    W.Workload("kk32", T=50, hidden=256, inter=128, num_experts=64, num_shared=2, top_k=30, dtype="bf16", seed=44),
    W.Workload("kk32_fp8", T=21, hidden=384, inter=128, num_experts=40, num_shared=0, top_k=32, dtype="fp8",
               seed=45),
]


def _plan(wl):
    logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
    ids, w = oracle.route(ocfg(wl), logits.numpy())
    return w.astype(np.float32), oracle.plan(ocfg(wl), ids, 0, 128)


def _dispatch(wl, p, x, max_ctas=0, scale_ld=0):
    cfg = B.config_of(wl)
    rows, H = p["rows"], wl.hidden
    slot = torch.as_tensor(p["slot_of"], device=DEV)
    if wl.dtype == "fp8":
        xe = torch.zeros(rows, H, dtype=torch.uint8, device=DEV)
        xs = (torch.zeros(H // 128, scale_ld, dtype=torch.float32, device=DEV) if scale_ld
              else torch.zeros(rows, H // 128, dtype=torch.float32, device=DEV))
        B.moe_dispatch(cfg, wl.T, x, slot, xe, xs, max_ctas, xe_scale_ld=scale_ld)
        torch.cuda.synchronize()
        s = xs.cpu().numpy()
        return xe.cpu().numpy(), (s[:, :rows].T if scale_ld else s)
    xe = torch.zeros(rows, H, dtype=torch.float32 if wl.dtype == "f32" else torch.bfloat16, device=DEV)
    B.moe_dispatch(cfg, wl.T, x, slot, xe, None, max_ctas)
    torch.cuda.synchronize()
    return np_f32(xe), None


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_dispatch_bit_exact_on_any_grid(wl):
    _, p = _plan(wl)
    x = synth.hidden(wl.T, wl.hidden, wl.dtype, wl.x_std, wl.seed)
    ref = oracle.dispatch(ocfg(wl), np_f32(x), p["slot_of"], p["rows"])
    used = p["token_of"] >= 0
    xd = x.to(DEV)
    for max_ctas in (0, 1, 3):
        xe, xs = _dispatch(wl, p, xd, max_ctas)
        if wl.dtype == "fp8":
            assert np.array_equal(xe[used], ref["xe_q"][used]), max_ctas
            assert np.array_equal(xs[used], ref["xe_s"][used]), max_ctas
        else:
            assert np.array_equal(xe[used], ref["xe"][used]), max_ctas
    if wl.dtype == "fp8":  # column-major scales with a stride above rows
        xe, xs = _dispatch(wl, p, xd, 0, scale_ld=p["rows"] + 5)
        assert np.array_equal(xe[used], ref["xe_q"][used])
        assert np.array_equal(xs[used], ref["xe_s"][used])


def _combine(wl, ye, w32, p, max_ctas=0):
    cfg = B.config_of(wl)
    y = torch.zeros(wl.T, wl.hidden, dtype=ye.dtype, device=DEV)
    B.moe_combine(cfg, wl.T, ye, torch.as_tensor(w32, device=DEV), torch.as_tensor(p["slot_of"], device=DEV), y,
                  max_ctas)
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("wl", CASES, ids=lambda w: w.name)
def test_staged_combine_matches_oracle_on_any_grid(wl):
    w32, p = _plan(wl)
    io = "f32" if wl.dtype == "f32" else "bf16"
    ye = synth.hidden(p["rows"], wl.hidden, io, 1.0, wl.seed + 100)
    ref = oracle.combine(ocfg(wl), np_f32(ye), w32.astype(np.float64), p["slot_of"])
    yd = ye.to(DEV)
    y0 = _combine(wl, yd, w32, p)
    got = np_f32(y0)
    if wl.dtype == "f32":
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6)
    else:
        # one bf16 rounding plus the fp32 accumulation error over k+S terms
        Y = np_f32(ye).astype(np.float64)
        kk = p["slot_of"].shape[1]
        absum = sum(np.abs((w32[:, j, None] if j < wl.top_k else 1.0) * Y[p["slot_of"][:, j]]) for j in range(kk))
        assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + absum * 2.0 ** -20)
    for max_ctas in (1, 3, 1000):
        assert torch.equal(_combine(wl, yd, w32, p, max_ctas), y0), max_ctas


def test_combine_reports_timeout_then_recovers():
    wl = CASES[0]
    w32, p = _plan(wl)
    ye = synth.hidden(p["rows"], wl.hidden, "bf16", 1.0, wl.seed + 100).to(DEV)
    y0 = _combine(wl, ye, w32, p)
    assert B.moe_comm_error(clear=True) == 0
    try:
        B.moe_debug_inject_wait(True, 2_000_000)
        _combine(wl, ye, w32, p)
        assert B.moe_comm_error(clear=True) == TIMEOUT
    finally:
        B.moe_debug_inject_wait(False)
    assert B.moe_comm_error() == 0
    assert torch.equal(_combine(wl, ye, w32, p), y0)
    assert B.moe_comm_error() == 0
