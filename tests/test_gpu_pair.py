"""The expert FFN on CTA pairs (tcgen05.mma.cta_group::2, 256 x 256 tiles) against the
oracle, through the C ABI.

* Forced onto small and odd shapes (MOE_FFN_TILE=pair, in a child process because the
  choice is read once per process): experts with fewer rows than a CTA (the peer CTA of
  the pair idle), a shared expert whose last pair tile is ragged in the peer's half,
  one-k-block tiles, several tiles per pair, capacity layout; every output element
  against the oracle.  The same shapes with MOE_FFN_TILE=single must agree too.
* At full size, in the benchmark's launch configuration (prefill ubatches: the FFN on
  every SM, no split of the GPU) and the kernels the library picks: every row of the busiest Zipf-routed
  expert of the Qwen3-30B-A3B prefill layer (fp8) and of the DeepSeek-V2-Lite layer at
  T=4096 (bf16: CTA-pair tiles), and for the DeepSeek-V3 prefill layer rows from every
  256-row block (both halves, the block edges) of the busiest routed expert and of the
  shared expert; each against the oracle's FFN of that single expert.  The Qwen3
  check is repeated with the fp8 CTA-pair kernels forced."""
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

from helpers import check_close, np_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
COMM_SMS = 0  # the benchmark's SM budget at prefill-sized ubatches: no split

FORCED_SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_gpu_edges as t
from moe_expert_dispatch_route_gb300 import workloads as W
from helpers import check_close
cases = [
    (W.QWEN3_DECODE.with_(T=48), 0),                     # ~3 rows per expert
    (W.DSV2LITE.with_(T=300), 0),                        # shared experts: 150 rows per ubatch
    (W.DSV2LITE.with_(T=300), 150),                      # capacity layout
    (W.QWEN3_PREFILL.with_(T=600), 0),                   # fp8
    (W.DSV3.with_(T=300, num_experts=32, n_group=8, topk_group=4), 0),
    (W.Workload("short_k_fp8", T=400, hidden=512, inter=128, num_experts=160, num_shared=1, top_k=4,
                dtype="fp8", seed=36), 0),               # down tiles of one k-block
    (W.Workload("short_k_bf16", T=400, hidden=512, inter=128, num_experts=160, num_shared=1, top_k=4,
                dtype="bf16", seed=37), 0),
    (W.Workload("odd_tc", T=45, hidden=768, inter=384, num_experts=33, num_shared=0, top_k=5, dtype="bf16",
                seed=32), 0),
]
for wl, cap in cases:
    got, ref = t.run_layer(wl, capacity=cap)
    assert got["err"] == 0 and ref["status"] == 0, (wl.name, got["err"])
    assert np.array_equal(got["ids"], ref["ids"])
    check_close(got["y"], ref["y"], wl.dtype, wl.name)
print("forced ok")
"""


@pytest.mark.parametrize("tile", ["pair", "single"])
def test_forced_tile_family_matches_oracle(tile):
    env = dict(os.environ, MOE_FFN_TILE=tile)
    code = FORCED_SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "forced ok" in r.stdout


def _ubatch0_ffn(wl):
    """Route, plan, dispatch and the expert FFN of the first ubatch through the C ABI, in
    the layer's launch configuration (fp8: column-major activation scales; the FFN on
    sms - COMM_SMS CTAs)."""
    cfg = B.config_of(wl)
    fp8 = wl.dtype == "fp8"
    T0 = wl.split
    E, S, k = wl.num_experts, wl.num_shared, wl.top_k
    NE, kk = E + S, k + S
    inp = synth.workload_inputs(wl, DEV)
    logits, x = inp["logits"][:T0].contiguous(), inp["x"][:T0].contiguous()
    rows = B.moe_plan_rows(cfg, T0, 0, 128)
    ids = torch.empty(T0, k, dtype=torch.int32, device=DEV)
    w = torch.empty(T0, k, dtype=torch.float32, device=DEV)
    counts = torch.empty(NE, dtype=torch.int32, device=DEV)
    offsets = torch.empty(NE + 1, dtype=torch.int32, device=DEV)
    slot_of = torch.empty(T0, kk, dtype=torch.int32, device=DEV)
    token_of = torch.empty(rows, dtype=torch.int32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pws = torch.empty(max(B.moe_plan_workspace_size(cfg, T0), 16), dtype=torch.uint8, device=DEV)
    xe = torch.zeros(rows, wl.hidden, dtype=torch.uint8 if fp8 else torch.bfloat16, device=DEV)
    xs = torch.zeros(wl.hidden // 128, rows, dtype=torch.float32, device=DEV) if fp8 else None
    ld = rows if fp8 else 0
    ye = torch.zeros(rows, wl.hidden, dtype=torch.bfloat16, device=DEV)
    fws = torch.empty(B.moe_ffn_workspace_size(cfg, rows), dtype=torch.uint8, device=DEV)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    W_ = [inp.get(key) for key in (("w13_q", "w13_s", "w2_q", "w2_s") if fp8 else ("w13", "w13_s", "w2", "w2_s"))]
    B.moe_route(cfg, T0, logits, None, ids, w)
    B.moe_plan(cfg, T0, ids, 0, 128, counts, offsets, slot_of, token_of, err, pws, pws.numel())
    B.moe_dispatch(cfg, T0, x, slot_of, xe, xs, xe_scale_ld=ld)
    B.moe_expert_ffn(cfg, counts, offsets, rows, xe, xs, *W_, ye, fws, fws.numel(), err, sms - COMM_SMS,
                     xe_scale_ld=ld)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return dict(inp=inp, counts=counts.cpu().numpy(), offsets=offsets.cpu().numpy(), xe=xe, xs=xs, ye=ye)


def _check_expert_rows(wl, r, e, sel):
    """ye of expert e at the given rows (relative to its segment) against the oracle's
    FFN of that expert alone."""
    inp = r["inp"]
    fp8 = wl.dtype == "fp8"
    base = int(r["offsets"][e])
    rows = torch.as_tensor(base + np.asarray(sel), dtype=torch.long, device=DEV)
    n = len(sel)
    c1 = oracle.Config(hidden=wl.hidden, inter=wl.inter, num_experts=1, num_shared=0, top_k=1,
                       dtype=oracle.FP8 if fp8 else oracle.BF16)
    cnt, off = np.array([n], np.int32), np.array([0, n], np.int32)
    if fp8:
        xe_q = r["xe"].index_select(0, rows).cpu().numpy()
        xe_s = r["xs"].index_select(1, rows).t().contiguous().cpu().numpy()
        Wn = {key: inp[key][e:e + 1].cpu().numpy() for key in ("w13_q", "w13_s", "w2_q", "w2_s")}
        ref = oracle.expert_ffn(c1, cnt, off, xe_q=xe_q, xe_s=xe_s, weights=Wn)
    else:
        Wn = {key: np_f32(inp[key][e:e + 1]) for key in ("w13", "w2")}
        ref = oracle.expert_ffn(c1, cnt, off, xe=np_f32(r["xe"].index_select(0, rows)), weights=Wn)
    got = np_f32(r["ye"].index_select(0, rows))
    check_close(got, ref, wl.dtype, f"expert {e} ({n} rows)")


def _block_sample(count, rng, per_block=8):
    """Rows of every 256-row block: both edges, both CTAs' halves around row 128, and
    random ones."""
    sel = set()
    for b in range(0, count, 256):
        hi = min(count, b + 256)
        for rr in (b, b + 1, b + 127, b + 128, hi - 2, hi - 1):
            if b <= rr < hi:
                sel.add(rr)
        sel.update(int(v) for v in rng.integers(b, hi, per_block))
    return sorted(sel)


def check_qwen3_prefill_busiest_expert():
    wl = W.QWEN3_PREFILL.with_(routing="zipf")
    r = _ubatch0_ffn(wl)
    e = int(np.argmax(r["counts"][: wl.num_experts]))
    count = int(r["counts"][e])
    assert count > 512  # several 256-row blocks
    _check_expert_rows(wl, r, e, list(range(count)))


def test_qwen3_prefill_busiest_zipf_expert_every_row():
    check_qwen3_prefill_busiest_expert()


def test_dsv3_prefill_every_block_of_busiest_and_shared_expert():
    wl = W.DSV3.with_(T=16384, routing="zipf")
    r = _ubatch0_ffn(wl)
    rng = np.random.default_rng(7)
    e = int(np.argmax(r["counts"][: wl.num_experts]))
    _check_expert_rows(wl, r, e, _block_sample(int(r["counts"][e]), rng))
    shared = wl.num_experts  # every token of the ubatch: 32 blocks of 256 rows
    _check_expert_rows(wl, r, shared, _block_sample(int(r["counts"][shared]), rng, per_block=4))


def test_dsv2lite_prefill_pair_tiles_busiest_expert_every_row():
    """bf16 at T=4096: the library's own choice is the CTA-pair kernel."""
    wl = W.DSV2LITE.with_(T=4096, routing="zipf")
    r = _ubatch0_ffn(wl)
    e = int(np.argmax(r["counts"][: wl.num_experts]))
    assert int(r["counts"][e]) > 512
    _check_expert_rows(wl, r, e, list(range(int(r["counts"][e]))))
    rng = np.random.default_rng(8)
    shared = wl.num_experts
    _check_expert_rows(wl, r, shared, _block_sample(int(r["counts"][shared]), rng, per_block=4))


FORCED_FULL_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_gpu_pair as t
t.check_qwen3_prefill_busiest_expert()
print("forced full ok")
"""


def test_forced_fp8_pair_tiles_qwen3_prefill_busiest_expert():
    """The FP8 CTA-pair kernels (chosen only when forced) at full size, every row of the
    busiest Zipf expert."""
    env = dict(os.environ, MOE_FFN_TILE="pair")
    code = FORCED_FULL_SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "forced full ok" in r.stdout
