"""The fused layer (moe_layer_dbo_ex with MOE_LAYER_FUSED_GATHER and / or _COMBINE): the
expert FFN gathers its A rows from x by token, its down kernel forms y in the epilogue.
Each option and both must give the
unfused layer's result bit for bit -- same routing, same operands, the combine's fixed
order and arithmetic -- on all five workloads (at full size for the prefill shapes, in
the benchmark's launch configuration), in capacity layout, unsplit, and replayed as a
CUDA graph; and it is checked against the oracle directly on a small layer."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import workloads as W

from helpers import check_close, np_f32, np_weights, ocfg
from test_gpu_layer import COMM_SMS, Layer

pytestmark = pytest.mark.gpu


def run_ex(L: Layer, flags, split=0, comm_sms=COMM_SMS):
    L.y.fill_(float("nan"))  # every row must be written
    L.err.zero_()
    B.moe_layer_dbo_ex(L.handle, L.cfg, L.args, L.T, split, 4, L.capacity, L.align, comm_sms, flags,
                       torch.cuda.current_stream(), L.comm)
    return L.result()


CASES = [W.TINY, W.QWEN3_DECODE, W.QWEN3_DECODE.with_(routing="zipf"), W.DSV2LITE, W.DSV2LITE.with_(T=4096),
         W.QWEN3_PREFILL, W.DSV3, W.DSV3.with_(T=16384), W.Workload("odd_tc", T=45, hidden=768, inter=384,
                                                                    num_experts=33, num_shared=0, top_k=5,
                                                                    dtype="bf16", seed=32),
         W.Workload("odd_fp8", T=19, hidden=384, inter=256, num_experts=40, num_shared=1, top_k=4, dtype="fp8",
                    seed=34)]


@pytest.mark.parametrize("wl", CASES, ids=lambda w: f"{w.name}-{w.T}-{w.routing}")
def test_fused_equals_unfused_bit_for_bit(wl):
    L = Layer(wl)
    ref = run_ex(L, 0)
    for flags in (B.LAYER_FUSED_GATHER, B.LAYER_FUSED_COMBINE, B.LAYER_FUSED):
        got = run_ex(L, flags)
        assert ref["err"] == 0 and got["err"] == 0, flags
        assert np.array_equal(got["ids"], ref["ids"])
        assert np.array_equal(got["w"], ref["w"])
        assert not np.isnan(got["y"]).any(), flags
        assert np.array_equal(got["y"], ref["y"]), flags
    L.close()


@pytest.mark.parametrize("wl", [W.QWEN3_DECODE, W.DSV2LITE.with_(T=512), W.QWEN3_PREFILL.with_(T=1024)],
                         ids=lambda w: w.name)
def test_fused_unsplit_capacity_and_budgets(wl):
    L = Layer(wl)
    base = run_ex(L, 0, split=wl.T)["y"]
    for kw in (dict(split=wl.T), dict(split=0), dict(split=0, comm_sms=0), dict(split=1)):
        got = run_ex(L, B.LAYER_FUSED, **kw)
        assert got["err"] == 0 and np.array_equal(got["y"], base), kw
    L.close()
    C = Layer(wl, capacity=wl.T)  # worst-token layout: every ubatch fits
    got = run_ex(C, B.LAYER_FUSED)
    assert got["err"] == 0 and np.array_equal(got["y"], base)
    C.close()


def test_fused_matches_oracle_every_element():
    wl = W.QWEN3_PREFILL.with_(T=64)
    L = Layer(wl)
    got = run_ex(L, B.LAYER_FUSED)
    ref = oracle.moe_layer(ocfg(wl), np_f32(L.logits), np_f32(L.x), np_weights(L.W), split=wl.split, align=128)
    L.close()
    assert got["err"] == 0 and np.array_equal(got["ids"], ref["ids"])
    check_close(got["y"], ref["y"], wl.dtype, "fused y")


def test_fused_graph_replay_equals_eager():
    wl = W.QWEN3_DECODE
    L = Layer(wl)
    eager = run_ex(L, B.LAYER_FUSED)["y"]
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            B.moe_layer_dbo_ex(L.handle, L.cfg, L.args, L.T, 0, 4, 0, 128, COMM_SMS, B.LAYER_FUSED,
                               torch.cuda.current_stream(), L.comm)
    torch.cuda.synchronize()
    for _ in range(3):
        L.y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(np_f32(L.y), eager)
    L.close()


def test_fused_rejects_unknown_flags():
    wl = W.QWEN3_DECODE.with_(T=8)
    L = Layer(wl)
    with pytest.raises(B.MoeError):
        B.moe_layer_dbo_ex(L.handle, L.cfg, L.args, L.T, 0, 4, 0, 128, 0, 6, torch.cuda.current_stream(), L.comm)
    L.close()
