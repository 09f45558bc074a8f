"""GPU parity of the whole layer (moe_layer_dbo) against the CPU oracle.

Small batches are checked on every output element; the five workloads at their
full sizes -- in the launch configuration the benchmark times (two ubatches, an SM
budget for the comm kernels, exact layout with 128-row alignment) -- are checked
bit-exactly on routing for every token and within tolerance on a seeded sample of
tokens, each computed by the oracle's per-token brute force.  The two-ubatch
output must equal the unsplit output bit for bit, and a replayed CUDA graph must
equal the eager call bit for bit."""
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
COMM_SMS = 16  # an SM budget for the comm-side kernels (the benchmark's at decode-sized ubatches)


class Layer:
    """Inputs, outputs and workspace of one layer call (all on the GPU)."""

    def __init__(self, wl, capacity=0, align=128, T=None, inputs=None):
        self.wl = wl
        self.T = wl.T if T is None else T
        self.cfg = B.config_of(wl)
        self.capacity, self.align = capacity, align
        inp = inputs or synth.workload_inputs(wl, DEV, T=self.T)
        self.logits, self.x, self.bias = inp["logits"], inp["x"], inp["bias"]
        self.W = {k: v for k, v in inp.items() if k.startswith("w")}
        io = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        self.y = torch.zeros(self.T, wl.hidden, dtype=io, device=DEV)
        self.ids = torch.zeros(self.T, wl.top_k, dtype=torch.int32, device=DEV)
        self.w = torch.zeros(self.T, wl.top_k, dtype=torch.float32, device=DEV)
        self.err = torch.zeros(1, dtype=torch.int32, device=DEV)
        self.ws = torch.empty(B.moe_layer_workspace_size(self.cfg, self.T, capacity, align), dtype=torch.uint8,
                              device=DEV)
        self.args = B.layer_args(self.logits, self.x, self.W, self.y, self.ids, self.w, self.ws, self.bias,
                                 self.err)
        self.handle = B.moe_dbo_create()
        self.comm = torch.cuda.Stream()

    def run(self, split=0, comm_sms=COMM_SMS, same_stream=False, min_tokens=4):
        comm = torch.cuda.current_stream() if same_stream else self.comm
        B.moe_layer_dbo(self.handle, self.cfg, self.args, self.T, split, min_tokens, self.capacity, self.align,
                        comm_sms, torch.cuda.current_stream(), comm)
        return self

    def result(self):
        torch.cuda.synchronize()
        return dict(y=np_f32(self.y), ids=self.ids.cpu().numpy(), w=self.w.cpu().numpy(),
                    err=int(self.err.item()))

    def close(self):
        B.moe_dbo_destroy(self.handle)


def token_ref(wl, x_t, ids_t, w_t, W_dev):
    """Oracle brute force for one token, copying only that token's experts to the host:
    the chosen routed experts become experts 0..k-1 of a k-expert layer, shared after."""
    E, S, k = wl.num_experts, wl.num_shared, wl.top_k
    sel = [int(e) for e in ids_t] + [E + s for s in range(S)]
    idx = torch.as_tensor(sel, dtype=torch.long, device=DEV)
    sub = {}
    for key, v in W_dev.items():
        t = v.index_select(0, idx).cpu()
        sub[key] = t.float().numpy() if t.dtype == torch.bfloat16 else t.numpy()
    c = ocfg(wl)
    c = oracle.Config(**{**c.__dict__, "num_experts": k, "gate": oracle.GATE_SOFTMAX, "n_group": 1,
                         "topk_group": 1})
    return oracle.token_output(c, x_t, np.arange(k, dtype=np.int32), w_t, sub)


SMALL = [W.TINY, W.QWEN3_DECODE.with_(T=64), W.QWEN3_DECODE.with_(T=50, routing="zipf"),
         W.DSV2LITE.with_(T=64), W.QWEN3_PREFILL.with_(T=64)]


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: f"{w.name}-{w.T}-{w.routing}")
@pytest.mark.parametrize("capacity", [0, -1], ids=["exact", "capacity"])
def test_small_layer_every_element(wl, capacity):
    cap = (wl.T + 1) // 2 if capacity < 0 else 0
    L = Layer(wl, capacity=cap)
    got = L.run().result()
    L.close()
    ref = oracle.moe_layer(ocfg(wl), np_f32(L.logits), np_f32(L.x), np_weights(L.W), split=wl.split,
                           capacity=cap, align=128)
    assert ref["status"] == 0 and got["err"] == 0
    assert np.array_equal(got["ids"], ref["ids"])
    np.testing.assert_allclose(got["w"], ref["w"], rtol=2e-6, atol=1e-7)
    check_close(got["y"], ref["y"], wl.dtype, "y")


FULL = [W.TINY, W.QWEN3_DECODE, W.QWEN3_DECODE.with_(routing="zipf"), W.DSV2LITE.with_(T=64),
        W.DSV2LITE, W.DSV2LITE.with_(T=4096), W.DSV2LITE.with_(T=4096, capacity=2048),
        W.QWEN3_PREFILL, W.DSV3, W.DSV3.with_(routing="zipf"), W.DSV3.with_(T=16384)]


@pytest.mark.parametrize("wl", FULL, ids=lambda w: f"{w.name}-{w.T}-{w.routing}-c{w.capacity}")
def test_full_size_layer_sampled_tokens(wl):
    L = Layer(wl, capacity=wl.capacity)
    got = L.run().result()
    ids_ref, w_ref = oracle.route(ocfg(wl), np_f32(L.logits))
    assert got["err"] == 0
    assert np.array_equal(got["ids"], ids_ref)
    np.testing.assert_allclose(got["w"], w_ref, rtol=2e-6, atol=1e-7)
    rng = np.random.default_rng(wl.seed)
    n = 4 if wl.hidden > 4096 else 8
    sample = sorted(set([0, wl.split - 1, wl.split, wl.T - 1] + list(rng.integers(0, wl.T, n))))
    x = np_f32(L.x)
    yref = np.stack([token_ref(wl, x[t], ids_ref[t], w_ref[t], L.W) for t in sample])
    check_close(got["y"][sample], yref, wl.dtype, "y[sample]")
    # two ubatches == one batch, bit for bit (the unsplit batch needs a capacity of T:
    # every shared expert receives every token)
    y_split = got["y"].copy()
    U = L if not wl.capacity else Layer(wl, capacity=wl.T, inputs=dict(logits=L.logits, x=L.x, bias=None, **L.W))
    got1 = U.run(split=wl.T).result()
    assert got1["err"] == 0
    assert np.array_equal(got1["y"], y_split)
    L.close()
    if U is not L:
        U.close()


@pytest.mark.parametrize("wl", [W.QWEN3_DECODE, W.DSV2LITE.with_(T=512, capacity=256), W.QWEN3_PREFILL.with_(T=1024)],
                         ids=lambda w: w.name)
def test_dbo_variants_bit_identical(wl):
    L = Layer(wl, capacity=wl.capacity)
    U = Layer(wl, capacity=wl.T if wl.capacity else 0, inputs=dict(logits=L.logits, x=L.x, bias=None, **L.W))
    base = U.run(split=wl.T).result()["y"]
    U.close()
    for kw in (dict(split=0), dict(split=1), dict(split=wl.T - 3), dict(split=0, comm_sms=0),
               dict(split=0, same_stream=True), dict(split=0, comm_sms=40)):
        if wl.capacity and kw.get("split", 0) in (1, wl.T - 3):
            continue  # ubatches larger than the capacity would overflow by design
        y = L.run(**kw).result()
        assert y["err"] == 0
        assert np.array_equal(y["y"], base), kw
    L.close()


def test_graph_replay_equals_eager():
    wl = W.QWEN3_DECODE
    L = Layer(wl)
    eager = L.run().result()["y"]
    L.y.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            B.moe_layer_dbo(L.handle, L.cfg, L.args, L.T, 0, 4, 0, 128, COMM_SMS, torch.cuda.current_stream(),
                            L.comm)
    torch.cuda.synchronize()
    for _ in range(3):
        L.y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(np_f32(L.y), eager)
    # new inputs written in place are picked up by the replay
    L.x.copy_(synth.hidden(wl.T, wl.hidden, wl.dtype, 1.0, 77, DEV))
    g.replay()
    torch.cuda.synchronize()
    replayed = np_f32(L.y)
    assert np.array_equal(replayed, L.run().result()["y"])
    L.close()


def test_layer_capacity_overflow_sets_flag():
    wl = W.QWEN3_DECODE.with_(routing="zipf")
    L = Layer(wl, capacity=4)
    got = L.run().result()
    assert got["err"] == 6  # MOE_ERR_CAPACITY
    # the flag is reset by the next call
    L2 = Layer(wl, capacity=128, inputs=dict(logits=L.logits, x=L.x, bias=None, **L.W))
    assert L2.run().result()["err"] == 0
    L.close()
    L2.close()


def test_single_token_and_tiny_batches_run_unsplit():
    for T in (1, 2, 3):
        wl = W.DSV2LITE.with_(T=T)
        L = Layer(wl)
        got = L.run().result()
        ref = oracle.moe_layer(ocfg(wl), np_f32(L.logits), np_f32(L.x), np_weights(L.W), align=128)
        assert np.array_equal(got["ids"], ref["ids"])
        check_close(got["y"], ref["y"], wl.dtype, f"y T={T}")
        L.close()
