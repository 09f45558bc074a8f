"""moe_plan_noalloc: the plan entry point for callers that cannot allocate device
memory -- code inside a CUDA-graph capture whose memory pool is locked, under an
allocator that owns the whole device, or in a plugin that is handed tensor pointers
only.  Its scratch is a fixed array inside the library.

Checked through the C ABI against moe_plan with a caller-provided workspace, byte
for byte, on two calls in a row with different routings (the second call must not
be affected by what the first left in the shared array), in exact and capacity
layouts (with and without overflow), on a batch exactly at the array's limit and
on one just past it (rejected before anything is enqueued).  This file is collected
last so that a failure here does not hide any other test's result."""
import ctypes

import pytest
import torch

from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import synth
from moe_expert_dispatch_route_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_INTS = 65536  # the built-in array: 256 KiB of per-chunk expert histograms


def _route(wl, routing, seed, T=None):
    T = wl.T if T is None else T
    cfg = B.config_of(wl)
    logits = synth.logits(T, wl.num_experts, routing, seed, DEV)
    ids = torch.empty(T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(T, wl.top_k, dtype=torch.float32, device=DEV)
    B.moe_route(cfg, T, logits, None, ids, w)
    return ids


def _outputs(wl, T, rows):
    NE, kk = wl.num_experts + wl.num_shared, wl.top_k + wl.num_shared
    return dict(counts=torch.full((NE,), -9, dtype=torch.int32, device=DEV),
                offsets=torch.full((NE + 1,), -9, dtype=torch.int32, device=DEV),
                slot_of=torch.full((T, kk), -9, dtype=torch.int32, device=DEV),
                token_of=torch.full((rows,), -9, dtype=torch.int32, device=DEV),
                err=torch.zeros(1, dtype=torch.int32, device=DEV))


def _compare(wl, T, ids, capacity, align):
    """moe_plan (workspace) vs moe_plan_noalloc on the same ids: every output and the
    error flag equal."""
    cfg = B.config_of(wl)
    rows = B.moe_plan_rows(cfg, T, capacity, align)
    ref = _outputs(wl, T, rows)
    wsb = B.moe_plan_workspace_size(cfg, T)
    ws = torch.empty(max(wsb, 16), dtype=torch.uint8, device=DEV)
    B.moe_plan(cfg, T, ids, capacity, align, ref["counts"], ref["offsets"], ref["slot_of"], ref["token_of"],
               ref["err"], ws, wsb)
    got = _outputs(wl, T, rows)
    B.moe_plan_noalloc(cfg, T, ids, capacity, align, got["counts"], got["offsets"], got["slot_of"],
                       got["token_of"], got["err"])
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    return int(got["err"].item())


def test_plan_noalloc_matches_plan_on_two_calls():
    wl = W.DSV2LITE.with_(T=4096)
    cfg = B.config_of(wl)
    assert B.moe_plan_workspace_size(cfg, wl.T) > 0  # this batch needs the scratch
    for routing, seed in (("uniform", 21), ("zipf", 22)):
        assert _compare(wl, wl.T, _route(wl, routing, seed), 0, 128) == 0


@pytest.mark.parametrize("capacity,expect", [(4096, 0), (300, 6)], ids=["fits", "overflows"])
def test_plan_noalloc_capacity_layout(capacity, expect):
    """Worst-token layout: with room for every entry (capacity = T: the shared experts
    receive every token) nothing is flagged; with too little, entries past the capacity
    get slot -1 and MOE_ERR_CAPACITY, as moe_plan."""
    wl = W.DSV2LITE.with_(T=4096)
    assert _compare(wl, wl.T, _route(wl, "zipf", 23), capacity, 1) == expect


def test_plan_noalloc_at_the_scratch_limit():
    """The largest DeepSeek-V3-shaped batch whose histograms fill the array (the last
    chunk's histogram ends at its final entries), then two more calls in a row."""
    wl = W.DSV3
    cfg = B.config_of(wl)
    NE = wl.num_experts + wl.num_shared
    T = 0
    while B.moe_plan_workspace_size(cfg, T + 1) <= 4 * SCRATCH_INTS:
        T += 1 if T > 20000 else 1000
    while B.moe_plan_workspace_size(cfg, T) > 4 * SCRATCH_INTS:
        T -= 1
    need = B.moe_plan_workspace_size(cfg, T)
    assert need <= 4 * SCRATCH_INTS and need > 4 * (SCRATCH_INTS - NE)
    for seed in (24, 25):
        assert _compare(wl, T, _route(wl, "uniform", seed, T), 0, 128) == 0


def test_plan_noalloc_rejects_batches_beyond_its_scratch():
    """One token past the limit: MOE_ERR_WORKSPACE before anything is enqueued (real
    buffers of the batch's sizes, so a regressed check would show as changed outputs,
    never as a kernel on an invalid address)."""
    wl = W.DSV3
    cfg = B.config_of(wl)
    T = 0
    while B.moe_plan_workspace_size(cfg, T + 1) <= 4 * SCRATCH_INTS:
        T += 1 if T > 20000 else 1000
    T += 1
    assert B.moe_plan_workspace_size(cfg, T) > 4 * SCRATCH_INTS
    ids = _route(wl, "uniform", 26, T)
    out = _outputs(wl, T, B.moe_plan_rows(cfg, T, 0, 128))
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = B.lib().moe_plan_noalloc(ctypes.byref(cfg), T, P(ids), 0, 128, P(out["counts"]), P(out["offsets"]),
                                  P(out["slot_of"]), P(out["token_of"]), P(out["err"]), 0, None)
    torch.cuda.synchronize()
    assert st == 4  # MOE_ERR_WORKSPACE
    assert int(out["err"].item()) == 0
    for k in ("counts", "offsets", "slot_of", "token_of"):
        assert bool((out[k] == -9).all()), k
