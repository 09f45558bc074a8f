"""The failure path of the bounded device waits, made to happen on purpose without
faulting or hanging anything: with the test hook moe_debug_inject_wait on, each
expert-FFN kernel first waits, for a short time chosen here, on a barrier nothing
completes (before it issues any copy).  The wait runs out, the kernel stores
MOE_ERR_TIMEOUT in the caller's error flag and returns; the next normal call on the
same GPU must give the result it gave before, bit for bit, with the flag clear.

Covered: the one-CTA kernels (bf16 and fp8), the CTA-pair kernels (bf16 as the library
chooses them, fp8 forced in a child process), and the whole DBO layer."""
import os
import subprocess
import sys

import pytest
import torch

import oracle
from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import synth
from moe_expert_dispatch_route_gb300 import workloads as W

from helpers import np_f32, ocfg

pytestmark = pytest.mark.gpu
DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIMIT_NS = 2_000_000  # 2 ms: the injected wait's limit
TIMEOUT = 8           # MOE_ERR_TIMEOUT


class Ffn:
    """One moe_expert_ffn call's inputs and outputs on the GPU."""

    def __init__(self, wl):
        self.wl, self.cfg = wl, B.config_of(wl)
        x = synth.hidden(wl.T, wl.hidden, wl.dtype, wl.x_std, wl.seed)
        logits = synth.logits(wl.T, wl.num_experts, wl.routing, wl.seed)
        Wt = synth.weights(wl.num_experts + wl.num_shared, wl.hidden, wl.inter, wl.dtype, wl.w_std, wl.seed, DEV)
        ids, _ = oracle.route(ocfg(wl), logits.numpy())
        p = oracle.plan(ocfg(wl), ids, 0, 128)
        d = oracle.dispatch(ocfg(wl), np_f32(x), p["slot_of"], p["rows"])
        self.rows = p["rows"]
        self.counts = torch.as_tensor(p["counts"], device=DEV)
        self.offsets = torch.as_tensor(p["offsets"], device=DEV)
        if wl.dtype == "fp8":
            self.xe = torch.as_tensor(d["xe_q"], device=DEV)
            self.xs = torch.as_tensor(d["xe_s"], device=DEV)
            self.w = [Wt[k] for k in ("w13_q", "w13_s", "w2_q", "w2_s")]
        else:
            self.xe = torch.as_tensor(d["xe"], device=DEV).to(torch.bfloat16)
            self.xs = None
            self.w = [Wt["w13"], None, Wt["w2"], None]
        self.ye = torch.zeros(self.rows, wl.hidden, dtype=torch.bfloat16, device=DEV)
        self.wsb = B.moe_ffn_workspace_size(self.cfg, self.rows)
        self.ws = torch.empty(self.wsb, dtype=torch.uint8, device=DEV)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.used = torch.as_tensor(p["token_of"] >= 0, device=DEV)

    def run(self):
        self.err.zero_()
        self.ye.zero_()
        w13, w13s, w2, w2s = self.w
        B.moe_expert_ffn(self.cfg, self.counts, self.offsets, self.rows, self.xe, self.xs, w13, w13s, w2, w2s,
                         self.ye, self.ws, self.wsb, self.err)
        torch.cuda.synchronize()
        return int(self.err.item()), self.ye[self.used].clone()


CASES = [
    ("single-bf16", W.QWEN3_DECODE.with_(T=40)),
    ("single-fp8", W.QWEN3_PREFILL.with_(T=40)),
    ("pair-bf16", W.DSV2LITE.with_(T=2048)),  # bf16, >= 128 rows per expert: the library picks CTA pairs
]


@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_bounded_wait_runs_out_and_reports_timeout(name, wl):
    check_timeout_and_recovery(wl)


FORCED_PAIR_SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import test_gpu_failure as t
from moe_expert_dispatch_route_gb300 import workloads as W
t.check_timeout_and_recovery(W.QWEN3_PREFILL.with_(T=2048))
print("pair fp8 ok")
"""


def test_bounded_wait_runs_out_in_forced_fp8_pair_tiles():
    """The FP8 CTA-pair kernels (chosen only when forced) take the same failure path."""
    env = dict(os.environ, MOE_FFN_TILE="pair")
    code = FORCED_PAIR_SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "pair fp8 ok" in r.stdout


def check_timeout_and_recovery(wl):
    f = Ffn(wl)
    err0, ref = f.run()
    assert err0 == 0
    try:
        B.moe_debug_inject_wait(True, LIMIT_NS)
        err1, _ = f.run()
    finally:
        B.moe_debug_inject_wait(False)
    assert err1 == TIMEOUT
    err2, again = f.run()  # the same GPU context, the next normal call
    assert err2 == 0
    assert torch.equal(again, ref)


def test_layer_reports_timeout_then_recovers():
    wl = W.QWEN3_DECODE.with_(T=64)
    cfg = B.config_of(wl)
    inp = synth.workload_inputs(wl, DEV)
    Wd = {k: v for k, v in inp.items() if k.startswith("w")}
    y = torch.zeros(wl.T, wl.hidden, dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros(wl.T, wl.top_k, dtype=torch.int32, device=DEV)
    w = torch.zeros(wl.T, wl.top_k, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(B.moe_layer_workspace_size(cfg, wl.T, 0, 128), dtype=torch.uint8, device=DEV)
    args = B.layer_args(inp["logits"], inp["x"], Wd, y, ids, w, ws, None, err)
    h = B.moe_dbo_create()
    comm = torch.cuda.Stream()

    def run():
        B.moe_layer_dbo(h, cfg, args, wl.T, 0, 4, 0, 128, 16, torch.cuda.current_stream(), comm)
        torch.cuda.synchronize()
        return int(err.item()), y.clone()

    try:
        e0, y0 = run()
        assert e0 == 0
        try:
            B.moe_debug_inject_wait(True, LIMIT_NS)
            e1, _ = run()
        finally:
            B.moe_debug_inject_wait(False)
        assert e1 == TIMEOUT
        e2, y2 = run()
        assert e2 == 0 and torch.equal(y2, y0)
    finally:
        B.moe_dbo_destroy(h)


def test_inject_wait_rejects_a_nonpositive_limit():
    with pytest.raises(B.MoeError):
        B.moe_debug_inject_wait(True, 0)
    B.moe_debug_inject_wait(False)
