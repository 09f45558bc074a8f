"""moe_plan_noalloc: the plan entry point for callers that cannot allocate device
memory (its scratch is a fixed array inside the library).  Checked through the C
ABI against moe_plan with a caller-provided workspace, on two calls in a row with
different routings -- the second call must not be affected by what the first left
in the shared array -- on a batch large enough to need the scratch.  This file is
collected last so that a failure here does not hide any other test's result."""
import numpy as np
import pytest
import torch

from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import synth
from moe_expert_dispatch_route_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route(wl, routing, seed):
    cfg = B.config_of(wl)
    logits = synth.logits(wl.T, wl.num_experts, routing, seed, DEV)
    ids = torch.empty(wl.T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.empty(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    B.moe_route(cfg, wl.T, logits, None, ids, w)
    return ids


def _outputs(wl, rows):
    NE, kk = wl.num_experts + wl.num_shared, wl.top_k + wl.num_shared
    return dict(counts=torch.full((NE,), -9, dtype=torch.int32, device=DEV),
                offsets=torch.full((NE + 1,), -9, dtype=torch.int32, device=DEV),
                slot_of=torch.full((wl.T, kk), -9, dtype=torch.int32, device=DEV),
                token_of=torch.full((rows,), -9, dtype=torch.int32, device=DEV),
                err=torch.zeros(1, dtype=torch.int32, device=DEV))


def test_plan_noalloc_matches_plan_on_two_calls():
    wl = W.DSV2LITE.with_(T=4096)
    cfg = B.config_of(wl)
    assert B.moe_plan_workspace_size(cfg, wl.T) > 0  # this batch needs the scratch
    rows = B.moe_plan_rows(cfg, wl.T, 0, 128)
    for routing, seed in (("uniform", 21), ("zipf", 22)):
        ids = _route(wl, routing, seed)
        ref = _outputs(wl, rows)
        wsb = B.moe_plan_workspace_size(cfg, wl.T)
        ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
        B.moe_plan(cfg, wl.T, ids, 0, 128, ref["counts"], ref["offsets"], ref["slot_of"], ref["token_of"],
                   ref["err"], ws, wsb)
        got = _outputs(wl, rows)
        B.moe_plan_noalloc(cfg, wl.T, ids, 0, 128, got["counts"], got["offsets"], got["slot_of"],
                           got["token_of"], got["err"])
        torch.cuda.synchronize()
        for k in ref:
            assert torch.equal(got[k], ref[k]), (routing, k)
        assert int(got["err"].item()) == 0


def test_plan_noalloc_rejects_batches_beyond_its_scratch():
    wl = W.DSV3
    cfg = B.config_of(wl)
    T = 2_000_000  # needs far more than the built-in 256 KiB of histograms
    L = B.lib()
    import ctypes
    st = L.moe_plan_noalloc(ctypes.byref(cfg), T, 16, 0, 128, 16, 16, 16, 16, 16, 0, None)
    assert st == 4  # MOE_ERR_WORKSPACE, before anything is enqueued
