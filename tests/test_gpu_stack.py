"""GPU parity of the stack of layers (moe_stack_dbo) against the oracle's stack:
every element of a small stack, bit-identical results for the two event placements,
for the split and the unsplit run, and for a replayed CUDA graph."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import synth
from moe_expert_dispatch_route_gb300 import workloads as W

from helpers import TOL_STACK, check_close, np_f32, np_weights, ocfg

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layers(wl, L, T, device):
    out = []
    for l in range(L):
        g = torch.Generator(device=device)
        g.manual_seed(9000 + l)
        wa = (torch.randn(wl.hidden, wl.hidden, generator=g, device=device) * 0.01).to(torch.bfloat16)
        ly = dict(logits=synth.logits(T, wl.num_experts, wl.routing, wl.seed + 10 * l, device), wa=wa)
        ly.update(synth.weights(wl.num_experts + wl.num_shared, wl.hidden, wl.inter, wl.dtype, wl.w_std,
                                wl.seed + 10 * l, device))
        out.append(ly)
    return out


class Stack:
    def __init__(self, wl, L, T, capacity=0):
        self.wl, self.L, self.T, self.cap = wl, L, T, capacity
        self.cfg = B.config_of(wl)
        self.layers = _layers(wl, L, T, DEV)
        self.x = synth.hidden(T, wl.hidden, "bf16", 1.0, wl.seed, DEV)
        self.out = torch.zeros_like(self.x)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.ws = torch.empty(B.moe_stack_workspace_size(self.cfg, T, capacity, 128), dtype=torch.uint8, device=DEV)
        self.args = B.StackArgs(self.x, self.out, self.layers, self.ws, None, self.err)
        self.h = B.moe_dbo_create()
        self.comm = torch.cuda.Stream()

    def run(self, split=0, before=1, comm_sms=16):
        B.moe_stack_dbo(self.h, self.cfg, self.args, self.T, split, 4, self.cap, 128, comm_sms, before,
                        torch.cuda.current_stream(), self.comm)
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0
        return np_f32(self.out)

    def oracle(self, split):
        lys = []
        for ly in self.layers:
            d = np_weights({k: v for k, v in ly.items() if k.startswith("w") and k != "wa"})
            d["wa"] = np_f32(ly["wa"])
            d["logits"] = np_f32(ly["logits"])
            lys.append(d)
        return oracle.moe_stack(ocfg(self.wl), np_f32(self.x), lys, split=split, capacity=self.cap, align=128)

    def close(self):
        B.moe_dbo_destroy(self.h)


@pytest.mark.parametrize("wl,L", [(W.QWEN3_DECODE.with_(T=64), 3), (W.DSV2LITE.with_(T=48), 2),
                                  (W.QWEN3_PREFILL.with_(T=64), 2)], ids=lambda v: getattr(v, "name", str(v)))
def test_stack_matches_oracle(wl, L):
    S = Stack(wl, L, wl.T)
    got = S.run()
    ref = S.oracle(wl.split)
    assert ref["status"] == 0
    tol = dict(TOL_STACK, rel_l2=3e-2) if wl.dtype == "fp8" else TOL_STACK
    check_close(got, ref["y"], wl.dtype, f"stack of {L}", tol)
    S.close()


def test_stack_schedules_agree_bit_for_bit():
    wl = W.QWEN3_DECODE
    S = Stack(wl, 2, wl.T)
    base = S.run(split=wl.T)
    for kw in (dict(split=0, before=1), dict(split=0, before=0), dict(split=100, before=1), dict(comm_sms=0)):
        assert np.array_equal(S.run(**kw), base), kw
    # graph capture of the whole stack
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            B.moe_stack_dbo(S.h, S.cfg, S.args, S.T, 0, 4, 0, 128, 16, 1, torch.cuda.current_stream(), S.comm)
    S.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(np_f32(S.out), base)
    S.close()
