"""Edge cases on the GPU against the oracle: shapes off every tile size (experts not
a multiple of 32, odd k, hidden / intermediate sizes that take the CUDA-core FFN),
ragged and tiny batches, a grouped gate with one group kept, and the independent
CUDA-core implementation of the FFN (MOE_FFN_IMPL=simt) for bf16 and fp8 layers."""
import os
import subprocess
import sys

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
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_layer(wl, capacity=0, align=128, split=0, comm_sms=16):
    cfg = B.config_of(wl)
    inp = synth.workload_inputs(wl, "cpu")
    Wt = {k: v for k, v in inp.items() if k.startswith("w")}
    d = {k: v.to(DEV) for k, v in Wt.items()}
    io = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    y = torch.zeros(wl.T, wl.hidden, dtype=io, device=DEV)
    ids = torch.zeros(wl.T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.zeros(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(B.moe_layer_workspace_size(cfg, wl.T, capacity, align), dtype=torch.uint8, device=DEV)
    args = B.layer_args(inp["logits"].to(DEV), inp["x"].to(DEV), d, y, ids, w, ws, None, err)
    h = B.moe_dbo_create()
    comm = torch.cuda.Stream()
    B.moe_layer_dbo(h, cfg, args, wl.T, split, 4, capacity, align, comm_sms, torch.cuda.current_stream(), comm)
    torch.cuda.synchronize()
    B.moe_dbo_destroy(h)
    s = split if split else (wl.T + 1) // 2
    ref = oracle.moe_layer(ocfg(wl), inp["logits"].numpy(), np_f32(inp["x"]), np_weights(Wt),
                           split=s if wl.T >= 4 else 0, capacity=capacity, align=align)
    return dict(y=np_f32(y), ids=ids.cpu().numpy(), err=int(err.item())), ref


ODD = [
    W.Workload("odd_bf16", T=37, hidden=384, inter=200, num_experts=37, num_shared=1, top_k=3, dtype="bf16", seed=31),
    W.Workload("odd_tc", T=45, hidden=768, inter=384, num_experts=33, num_shared=0, top_k=5, dtype="bf16", seed=32),
    W.Workload("odd_f32", T=29, hidden=96, inter=80, num_experts=5, num_shared=2, top_k=1, dtype="f32",
               x_std=0.02, seed=33),
    W.Workload("odd_fp8", T=19, hidden=384, inter=256, num_experts=40, num_shared=1, top_k=4, dtype="fp8", seed=34),
    W.Workload("grouped_one", T=23, hidden=512, inter=256, num_experts=64, num_shared=0, top_k=6,
               gate="sigmoid_grouped", n_group=4, topk_group=1, dtype="bf16", seed=35),
    # the tensor-core kernels with one or two k-blocks per tile and several tiles per CTA
    # (160 experts: the FP8 down kernel has ~640 tiles of a single k-block), so the FP8
    # scale staging looks ahead across many tile boundaries
    W.Workload("short_k_fp8", T=400, hidden=512, inter=128, num_experts=160, num_shared=1, top_k=4, dtype="fp8",
               seed=36),
    W.Workload("short_k_bf16", T=400, hidden=512, inter=128, num_experts=160, num_shared=1, top_k=4, dtype="bf16",
               seed=37),
]


@pytest.mark.parametrize("wl", ODD, ids=lambda w: w.name)
@pytest.mark.parametrize("align", [1, 128])
def test_odd_shapes(wl, align):
    got, ref = run_layer(wl, align=align)
    assert got["err"] == 0 and ref["status"] == 0
    assert np.array_equal(got["ids"], ref["ids"])
    check_close(got["y"], ref["y"], wl.dtype, wl.name)


@pytest.mark.parametrize("T,split", [(1, 0), (2, 0), (3, 0), (4, 0), (5, 0), (5, 1), (5, 4), (9, 2)])
def test_tiny_and_ragged_batches(T, split):
    wl = W.QWEN3_DECODE.with_(T=T)
    got, ref = run_layer(wl, split=split)
    assert np.array_equal(got["ids"], ref["ids"])
    check_close(got["y"], ref["y"], wl.dtype, f"T={T} split={split}")


def test_capacity_equal_to_ubatch_never_overflows():
    wl = W.DSV2LITE.with_(T=33, routing="zipf")
    got, ref = run_layer(wl, capacity=17)
    assert got["err"] == 0 and ref["status"] == 0
    check_close(got["y"], ref["y"], wl.dtype, "capacity")


SIMT_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_gpu_edges as t
from moe_expert_dispatch_route_gb300 import workloads as W
from helpers import check_close
for wl in (W.QWEN3_DECODE.with_(T=24), W.QWEN3_PREFILL.with_(T=24)):
    got, ref = t.run_layer(wl)
    assert np.array_equal(got["ids"], ref["ids"])
    check_close(got["y"], ref["y"], wl.dtype, "simt " + wl.name)
print("simt ok")
"""


def test_cuda_core_ffn_implementation_matches_oracle():
    env = dict(os.environ, MOE_FFN_IMPL="simt")
    code = SIMT_SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "simt ok" in r.stdout
