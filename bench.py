#!/usr/bin/env python3
"""Benchmark of the single-GPU MoE layer with Dual-Batch Overlap.

One step = one pass of the whole layer -- route, plan, dispatch, expert FFN and
combine on two ubatches overlapped on a compute and a comm stream
(moe_layer_dbo) -- over one batch of synthetic input, replayed as a CUDA graph.
Default workload: the largest configuration that fits one GPU, the DeepSeek-V3
shaped prefill layer (T=16384 split 8192/8192, hidden 7168, 256 routed + 1 shared
experts, grouped sigmoid gate 8 groups -> top-4 groups -> top-8, intermediate 2048,
fp8 e4m3 with 128-block scales, uniform routing, ~11 GB of expert weights).

Timing: K graph replays between CUDA events on the compute stream form one block,
bracketed by a barrier and a synchronize; blocks are repeated until at least
--min-seconds of timed work have passed and the median block's time per step is
reported (with the spread), so the clock sampler sees the GPU under load for
several seconds.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload on its own GPU (the layer has no cross-GPU step), so the
scaling is weak and the value is the tokens of all ranks over the slowest rank's
time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from moe_expert_dispatch_route_gb300 import workloads as W  # noqa: E402

METRIC = "MoE-layer tokens/s (route->dispatch->GEMM->combine, DBO) at 1 GB300; % roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# SMs given to the comm-side steps while they overlap an FFN.  Measured on GB300 (0, 8,
# 16, 24, 32 SMs): decode-sized ubatches gain from 16, where the FFN streams weights and
# the comm kernels are latency-bound; prefill ubatches are fastest with no split at all,
# because there the FFN is held by a GPU-wide limit and kernels beside it only take
# bandwidth from it (DeepSeek-V3 T=16384: 8.41 ms with no split, 8.73 with 16 SMs).
COMM_SMS_DECODE = 16
DECODE_UBATCH_MAX = 512


def default_comm_sms(wl) -> int:
    ub = wl.split if (wl.T >= 4 and 0 < wl.split < wl.T) else wl.T
    return COMM_SMS_DECODE if ub <= DECODE_UBATCH_MAX else 0
DEFAULT_WORKLOAD = ("dsv3", 16384)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=None, choices=sorted(W.ALL),
                    help=f"default: {DEFAULT_WORKLOAD[0]} at T={DEFAULT_WORKLOAD[1]}")
    ap.add_argument("--T", type=int, default=None)
    ap.add_argument("--experts", type=int, default=None, help="routed experts (a scaled-down shape for profiling)")
    ap.add_argument("--min-seconds", type=float, default=3.0,
                    help="repeat blocks of --steps timed steps until this much timed work has passed")
    ap.add_argument("--routing", default=None, choices=[None, "uniform", "zipf"])
    ap.add_argument("--capacity", type=int, default=None,
                    help="rows per expert per ubatch (worst-token layout); -1 = the ubatch size")
    ap.add_argument("--comm-sms", type=int, default=None,
                    help="SM budget of the comm-side steps beside an FFN (default: 16 for ubatches of at "
                         "most 512 tokens, else 0 = no split)")
    ap.add_argument("--fused", default="none", choices=["none", "gather", "combine", "both"],
                    help="time the layer with the gather fused into the expert GEMM and / or the combine into "
                         "its epilogue; every other mode is timed beside it")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the DBO-gain and e2e legs")
    ap.add_argument("--stack", type=int, default=0,
                    help="time a stack of this many layers (stand-in block + MoE layer each) instead of one layer")
    return ap.parse_args()


def workload(args):
    if args.workload is None:
        wl = W.ALL[DEFAULT_WORKLOAD[0]].with_(T=DEFAULT_WORKLOAD[1])
    else:
        wl = W.ALL[args.workload]
    if args.T:
        wl = wl.with_(T=args.T)
    if args.experts:
        wl = wl.with_(num_experts=args.experts)
    if args.routing:
        wl = wl.with_(routing=args.routing)
    if args.capacity is not None:
        wl = wl.with_(capacity=wl.split if args.capacity < 0 else args.capacity)
    return wl


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every 100 ms (read-only queries).  stop() summarises the
    samples whose timestamps fall inside the timed window."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            self.sel = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                   "-f", self.path]
            if self.sel:
                cmd[1:1] = ["-i", self.sel]
            self.proc = subprocess.Popen(cmd, stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    @staticmethod
    def _when(text: str):
        for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
            try:
                return datetime.datetime.strptime(text.strip(), fmt)
            except ValueError:
                pass
        return None

    def stop(self, window=None):
        """window: (start, end) local datetimes of the timed region."""
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "samples_under_load": 0}
        if not self.proc:
            return out
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        try:
            with open(self.path) as f:
                rows = [ln.strip().split(",") for ln in f if ln.strip()]
            os.unlink(self.path)
        except Exception:
            return out
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        parsed = []
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 10:
                continue
            try:
                parsed.append((self._when(r[0]), float(r[2]), float(r[3]), float(r[4]),
                               [n for n, v in zip(names, r[6:10]) if v.lower() == "active"]))
            except ValueError:
                continue
        if not parsed:
            return out
        inside = [p for p in parsed if window and p[0] and window[0] <= p[0] <= window[1]]
        use = inside or parsed
        reasons = sorted({n for p in use for n in p[4]})
        out.update(sm_mhz=statistics.median(p[1] for p in use), sm_max_mhz=max(p[2] for p in parsed),
                   power_w_median=statistics.median(p[3] for p in use), reasons=reasons, samples=len(parsed),
                   samples_under_load=len(inside))
        return out


# --------------------------------------------------------------------------- helpers
def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """The slowest rank's time (every rank gets it)."""
    if world == 1:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def launches_per_step(wl, split_two: bool, fused: str = "none", tc: bool = True) -> int:
    """Kernels this library launches for one layer call, per ubatch: route; plan and
    dispatch (one fused kernel when the plan is a single chunk; route, plan and dispatch
    in one clustered kernel for a small batch that runs alone: the unsplit batch or
    ubatch 0); the two FFN kernels; combine."""
    kk = wl.top_k + wl.num_shared
    tpc = max(1, 4096 // kk)
    sizes = [wl.split, wl.T - wl.split] if split_two else [wl.T]
    n = 0
    for u, Tu in enumerate(sizes):
        chunks = max(1, math.ceil(Tu / tpc))
        if fused != "none" and tc:  # route, plan (count + assign when chunked), gather step, FFN, combine
            gather = fused in ("gather", "both")
            n += 1 + (1 if chunks == 1 else 2)
            n += (1 if wl.dtype == "fp8" else 0) if gather else 1  # quantisation | dispatch
            n += 2 + (0 if fused in ("combine", "both") else 1)
            continue
        alone = u == 0
        if chunks == 1 and alone and Tu <= 128:
            head = 1
        else:
            head = 1 + (1 if chunks == 1 else 3)  # route + (plan/dispatch fused | count, assign, dispatch)
        n += head + 2 + 1
    return n


def code_only(text: str) -> str:
    """C/C++ source without comments, whitespace runs collapsed (the sources hold no
    comment markers inside string literals)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def ffn_source_hash() -> str:
    """Hash of the code (comments aside) of the FFN kernels' device sources: a
    profile's DRAM counters apply only while it is unchanged."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_expert_dispatch_route_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.startswith("ffn") or name in ("common.cuh", "tc_ptx.cuh"):
            with open(os.path.join(csrc, name)) as f:
                h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag: str, wl):
    """DRAM bytes per launch recorded from an ncu capture in profiles/ (for this workload
    and batch size), only if the FFN sources are unchanged since the capture."""
    p = os.path.join(ROOT, "profiles", f"{kernel_tag}_{wl.name}_T{wl.T}.txt")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for ln in f:
            if ":" in ln:
                k, v = ln.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("ffn_source_hash") != ffn_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    from moe_expert_dispatch_route_gb300 import binding as B
    from moe_expert_dispatch_route_gb300 import synth

    wl = workload(args)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = B.config_of(wl)
    T, H, E, k = wl.T, wl.hidden, wl.num_experts, wl.top_k
    io = torch.float32 if wl.dtype == "f32" else torch.bfloat16
    inp = synth.workload_inputs(wl, dev)
    Wd = {kk_: v for kk_, v in inp.items() if kk_.startswith("w")}
    logits, x = inp["logits"], inp["x"]
    y = torch.zeros(T, H, dtype=io, device=dev)
    ids = torch.zeros(T, k, dtype=torch.int32, device=dev)
    w = torch.zeros(T, k, dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    cap, align = wl.capacity, wl.align
    ws = torch.empty(B.moe_layer_workspace_size(cfg, T, cap, align), dtype=torch.uint8, device=dev)
    args_c = B.layer_args(logits, x, Wd, y, ids, w, ws, None, err)
    handle = B.moe_dbo_create()
    comm = torch.cuda.Stream(device=dev)
    compute = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()  # inputs and zeroed buffers were made on the current stream
    comm_sms = args.comm_sms if args.comm_sms is not None else default_comm_sms(wl)

    modes = {"none": 0, "gather": B.LAYER_FUSED_GATHER, "combine": B.LAYER_FUSED_COMBINE, "both": B.LAYER_FUSED}
    flags = modes[args.fused]

    def enqueue(split=0, same=False, a=args_c, cs=None, fl=None):
        cs = cs or torch.cuda.current_stream()
        B.moe_layer_dbo_ex(handle, cfg, a, T, split, 4, cap, align, comm_sms, flags if fl is None else fl, cs,
                           cs if same else comm)

    def capture(**kw):  # split, same, a, fl
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(compute):
            enqueue(**kw)  # eager warm call (also builds any per-device state)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=compute):
                enqueue(**kw, cs=compute)
        torch.cuda.synchronize()
        return g

    def time_graph(g, steps, warmup):
        """Mean time per step over one block of `steps` replays."""
        for _ in range(warmup):
            g.replay()
        return time_block(g, steps)

    def time_block(g, steps):
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(compute):
            e0.record(compute)
            for _ in range(steps):
                g.replay()
            e1.record(compute)
        torch.cuda.synchronize()
        barrier(world)
        return e0.elapsed_time(e1) / steps

    g_dbo = capture(split=0)
    for _ in range(args.warmup):
        g_dbo.replay()
    # blocks of exactly K steps, each bracketed by barrier + synchronize, repeated until
    # at least --min-seconds of timed work (the same number of blocks on every rank)
    first = max_over_ranks(time_block(g_dbo, args.steps), world)
    n_blocks = max(3, math.ceil(args.min_seconds * 1e3 / max(first * args.steps, 1e-3)))
    n_blocks = int(max_over_ranks(float(n_blocks), world))
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    g_dbo.replay()  # the GPU is busy when the window opens
    torch.cuda.synchronize()
    t_open = datetime.datetime.now()
    wall0 = time.perf_counter()
    blocks = [max_over_ranks(time_block(g_dbo, args.steps), world) for _ in range(n_blocks)]
    timed_s = time.perf_counter() - wall0
    clocks = sampler.stop((t_open, datetime.datetime.now()))
    ms = statistics.median(blocks)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error flag {int(err.item())}"
    timing = {"blocks": n_blocks, "steps_per_block": args.steps, "timed_seconds": round(timed_s, 3),
              "ms_per_step_median": round(ms, 5), "ms_per_step_min": round(min(blocks), 5),
              "ms_per_step_max": round(max(blocks), 5),
              "how": "each block: barrier + synchronize, K CUDA-graph replays between CUDA events on the compute "
                     "stream, synchronize + barrier; max over ranks per block; median over blocks"}
    ids_host = ids.cpu().numpy()

    res = {}
    two = T >= 4 and 0 < wl.split < T
    if not args.no_extras:
        # DBO gain: the same two ubatches serialised on one stream, and the unsplit layer
        g_serial = capture(split=0, same=True)
        ms_serial = max_over_ranks(time_graph(g_serial, args.steps, args.warmup), world)
        g_unsplit = capture(split=T)
        ms_unsplit = max_over_ranks(time_graph(g_unsplit, args.steps, args.warmup), world)
        res["dbo"] = {"ms_dbo": round(ms, 5), "ms_two_ubatches_one_stream": round(ms_serial, 5),
                      "ms_unsplit_one_stream": round(ms_unsplit, 5),
                      "gain_vs_two_ubatches_one_stream": round(ms_serial / ms, 4),
                      "gain_vs_unsplit": round(ms_unsplit / ms, 4), "comm_sms": comm_sms}
        del g_serial, g_unsplit
        # the other modes: the gather fused into the expert GEMM and / or the combine into its
        # epilogue, against dispatched rows and the combine kernel
        times = {args.fused: ms}
        for name, fl in modes.items():
            if name not in times and wl.dtype != "f32":
                g_other = capture(split=0, fl=fl)
                times[name] = max_over_ranks(time_graph(g_other, args.steps, args.warmup), world)
                del g_other
        if len(times) > 1:
            res["fused"] = {"timed_mode": args.fused, "ms": {k: round(v, 5) for k, v in times.items()},
                            "gain_vs_unfused": {k: round(times["none"] / v, 4) for k, v in times.items()},
                            "bytes_saved_by_gather_per_step": fused_bytes_saved(wl, two)}

    # ---- roofline of the dominant kernel: moe_expert_ffn on ubatch 0, timed alone
    roof = ffn_roofline(B, wl, cfg, inp, dev, args, comm_sms, compute)
    # ---- roofline of the whole layer (the metric's "% roofline")
    layer_roof = layer_roofline(wl, ids_host, ms, two)

    # ---- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_extras:
        e2e = run_e2e(B, wl, cfg, inp, args_c, handle, comm, compute, enqueue, logits, x, y, args, world)

    value = T * world / (ms / 1e3)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"f32": "f32", "bf16": "bf16", "fp8": "fp8e4m3"}[wl.dtype],
        "data": "synthetic (seeded N(0,1) logits / hidden states, N(0,0.02) weights)",
        "config": {"workload": wl.describe() + ("" if args.fused == "none" else f" fused-{args.fused}"), "T": T,
                   "hidden": H,
                   "inter": wl.inter, "experts": E,
                   "shared": wl.num_shared, "top_k": k, "ubatches": 2 if two else 1, "split": wl.split,
                   "layout": f"capacity {cap}" if cap else f"exact, align {align}", "comm_sms": comm_sms,
                   "graph": "CUDA graph replay", "l2": "inputs larger than L2 (expert weights "
                   f"{weights_bytes(wl) / 1e9:.2f} GB > 129 MB L2)", "parallelism": f"replicas x{world}"},
        "gpu_launches": launches_per_step(wl, two, args.fused, wl.dtype != "f32") * args.steps * n_blocks,
        "timing": timing,
        "clocks": clocks,
        "roofline": roof,
        "layer_roofline": layer_roof,
        "e2e": e2e,
    }
    out.update(res)
    B.moe_dbo_destroy(handle)
    return out, wl, inp


def run_stack(args, rank, world, local):
    """A stack of L layers (moe_stack_dbo): tokens/s through all layers, with the events
    recorded before the yield (the fix) and after it (the old placement), and unsplit."""
    from moe_expert_dispatch_route_gb300 import binding as B
    from moe_expert_dispatch_route_gb300 import synth

    wl = workload(args)
    L = args.stack
    comm_sms = args.comm_sms if args.comm_sms is not None else default_comm_sms(wl)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = B.config_of(wl)
    T = wl.T
    layers = []
    for l in range(L):
        g = torch.Generator(device=dev)
        g.manual_seed(9000 + l)
        ly = dict(logits=synth.logits(T, wl.num_experts, wl.routing, wl.seed + 10 * l, dev),
                  wa=(torch.randn(wl.hidden, wl.hidden, generator=g, device=dev) * 0.01).to(torch.bfloat16))
        ly.update(synth.weights(wl.num_experts + wl.num_shared, wl.hidden, wl.inter, wl.dtype, wl.w_std,
                                wl.seed + 10 * l, dev))
        layers.append(ly)
    x = synth.hidden(T, wl.hidden, "bf16", 1.0, wl.seed, dev)
    out = torch.zeros_like(x)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(B.moe_stack_workspace_size(cfg, T, wl.capacity, wl.align), dtype=torch.uint8, device=dev)
    sa = B.StackArgs(x, out, layers, ws, None, err)
    h = B.moe_dbo_create()
    comm = torch.cuda.Stream(device=dev)
    compute = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()  # inputs and zeroed buffers were made on the current stream

    def graph(split, before):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(compute):
            B.moe_stack_dbo(h, cfg, sa, T, split, 4, wl.capacity, wl.align, comm_sms, before, compute, comm)
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=compute):
                B.moe_stack_dbo(h, cfg, sa, T, split, 4, wl.capacity, wl.align, comm_sms, before, compute, comm)
        torch.cuda.synchronize()
        return g

    def timed(g, sample=False):
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        barrier(world)
        sampler = ClockSampler(local) if sample else None
        if sampler:
            sampler.start()
            time.sleep(0.3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(compute):
            e0.record(compute)
            for _ in range(args.steps):
                g.replay()
            e1.record(compute)
        torch.cuda.synchronize()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1) / args.steps, world), (sampler.stop() if sampler else None)

    ms_fix, clocks = timed(graph(0, 1), sample=True)
    ms_old, _ = timed(graph(0, 0))
    ms_unsplit, _ = timed(graph(T, 1))
    assert int(err.item()) == 0
    B.moe_dbo_destroy(h)
    out = {"metric": f"MoE stack tokens/s ({L} layers of stand-in block + MoE layer, DBO) at 1 GB300",
           "value": round(T * world / (ms_fix / 1e3), 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms_fix, 5), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": {"f32": "f32", "bf16": "bf16", "fp8": "fp8e4m3"}[wl.dtype],
           "data": "synthetic", "config": {"workload": wl.describe(), "layers": L, "comm_sms": comm_sms},
           "clocks": clocks,
           "stack": {"ms_event_before_yield": round(ms_fix, 5), "ms_event_after_yield": round(ms_old, 5),
                     "gain_of_event_before_yield": round(ms_old / ms_fix, 4),
                     "ms_unsplit": round(ms_unsplit, 5), "gain_vs_unsplit": round(ms_unsplit / ms_fix, 4)}}
    return out


def fused_bytes_saved(wl, two: bool) -> dict:
    """DRAM bytes the fused layer does not move, per step (model): dispatch's reads of x
    and writes of xe (+ scales), the gate/up kernel's reads of xe, and the combine's
    re-reads of ye; it adds the per-token quantisation of x for fp8 (reads x, writes x_q),
    the gathers' reads of x / x_q (once per token: the rows of a ubatch stay in L2) and the
    combine's reads of ye inside the down kernel (counted the same as the kernel's)."""
    T, H, kk = wl.T, wl.hidden, wl.top_k + wl.num_shared
    io, elt = (4, 4) if wl.dtype == "f32" else (2, 2 if wl.dtype == "bf16" else 1)
    rows = T * kk
    scales = rows * (H // 128) * 4 if wl.dtype == "fp8" else 0
    dispatch = T * H * io + rows * H * elt + scales
    xe_read = rows * H * elt + scales
    fused_in = (T * H * io + T * H * elt + T * (H // 128) * 4 if wl.dtype == "fp8" else 0) + T * H * elt
    return {"model_bytes": int(dispatch + xe_read - fused_in),
            "note": "dispatch (x read, xe written) + xe read by the gate/up GEMM, less the per-token quantisation "
                    "and one gathered read of x per token"}


def weights_bytes(wl) -> float:
    NE = wl.num_experts + wl.num_shared
    elt = {"f32": 4, "bf16": 2, "fp8": 1}[wl.dtype]
    return NE * 3 * wl.hidden * wl.inter * elt


def expert_weight_bytes(wl) -> int:
    """Bytes of one expert's weights (W13 + W2, with the fp8 block scales)."""
    H, I = wl.hidden, wl.inter
    elt = {"f32": 4, "bf16": 2, "fp8": 1}[wl.dtype]
    scales = ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128)) * 4 if wl.dtype == "fp8" else 0
    return 3 * H * I * elt + scales


def layer_roofline(wl, ids, ms: float, two: bool) -> dict:
    """The layer's roofline: the slower of the grouped-GEMM FLOPs at the tensor peak and
    the weight + activation bytes at HBM bandwidth, against the measured step time.
    Weights are counted per ubatch (each ubatch's expert GEMMs read every expert it
    touches, as the DBO method must) and, for comparison, once (the unsplit layer's
    bound).  The step is timed over seconds, so the tensor peak is the sustained one."""
    pk, src = peaks()
    T, H, E, S, k = wl.T, wl.hidden, wl.num_experts, wl.num_shared, wl.top_k
    fp8 = wl.dtype == "fp8"
    io = 4 if wl.dtype == "f32" else 2
    NE = E + S
    bounds = [(0, wl.split), (wl.split, T)] if two else [(0, T)]

    def touched(lo, hi):
        c = np.bincount(ids[lo:hi].reshape(-1), minlength=E)[:E]
        return int((c > 0).sum()) + (S if hi > lo else 0)

    t_dbo = sum(touched(lo, hi) for lo, hi in bounds)
    t_once = touched(0, T)
    wb = expert_weight_bytes(wl)
    act = T * E * 4 + T * H * io + T * H * io + T * k * 8  # logits, x, y, ids + weights
    flops = 2.0 * T * (k + S) * 3 * H * wl.inter
    bw = pk["hbm_gbs"] * 1e9
    sustained = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    tf = sustained * 1e12 * (2.0 if fp8 else 1.0)
    t = ms / 1e3
    out = {"flops": flops, "bytes_weights_per_ubatch": t_dbo * wb + act, "bytes_weights_once": t_once * wb + act,
           "experts_touched_per_ubatch": t_dbo, "experts_touched_once": t_once,
           "achieved_tflops": round(flops / t / 1e12, 2), "tensor_peak_tflops": round(tf / 1e12, 2),
           "hbm_peak_gbs": pk["hbm_gbs"],
           "peak_source": f"{src} (HBM copy; {'fp8 = 2x ' if fp8 else ''}sustained bf16 GEMM)"}
    for key, nbytes in (("frac", t_dbo * wb + act), ("frac_vs_unsplit_bound", t_once * wb + act)):
        t_min = max(flops / tf, nbytes / bw)
        out[key] = round(t_min / t, 4)
    out["bound"] = "tensor" if flops / tf > (t_dbo * wb + act) / bw else "hbm"
    out["note"] = ("frac = roofline time / measured step; frac_vs_unsplit_bound counts every touched expert's "
                   "weights once (the bound of the layer run as one batch)")
    return out


def ffn_roofline(B, wl, cfg, inp, dev, args, comm_sms, compute):
    pk, src = peaks()
    T0 = wl.split if (wl.T >= 4 and 0 < wl.split < wl.T) else wl.T
    H, I, E, S, k = wl.hidden, wl.inter, wl.num_experts, wl.num_shared, wl.top_k
    NE, kk = E + S, k + S
    fp8 = wl.dtype == "fp8"
    elt = {"f32": 4, "bf16": 2, "fp8": 1}[wl.dtype]
    io = 4 if wl.dtype == "f32" else 2
    rows = B.moe_plan_rows(cfg, T0, wl.capacity, wl.align)
    ids = torch.zeros(T0, k, dtype=torch.int32, device=dev)
    w = torch.zeros(T0, k, dtype=torch.float32, device=dev)
    counts = torch.zeros(NE, dtype=torch.int32, device=dev)
    offsets = torch.zeros(NE + 1, dtype=torch.int32, device=dev)
    slot_of = torch.zeros(T0, kk, dtype=torch.int32, device=dev)
    token_of = torch.zeros(rows, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pws = torch.empty(max(B.moe_plan_workspace_size(cfg, T0), 4), dtype=torch.uint8, device=dev)
    xe = torch.zeros(rows, H * elt, dtype=torch.uint8, device=dev)
    # fp8 row scales column-major (scale(row, g) at g * rows + row), as the layer keeps them
    xs = torch.zeros(H // 128, rows, dtype=torch.float32, device=dev) if fp8 else None
    xs_ld = rows if fp8 else 0
    ye = torch.zeros(rows, H * io, dtype=torch.uint8, device=dev)
    fws = torch.empty(B.moe_ffn_workspace_size(cfg, rows), dtype=torch.uint8, device=dev)
    w13 = inp.get("w13", inp.get("w13_q"))
    w2 = inp.get("w2", inp.get("w2_q"))
    torch.cuda.synchronize()  # the buffers above were zeroed on the current stream
    with torch.cuda.stream(compute):
        B.moe_route(cfg, T0, inp["logits"], None, ids, w, 0, compute)
        B.moe_plan(cfg, T0, ids, wl.capacity, wl.align, counts, offsets, slot_of, token_of, err, pws,
                   pws.numel(), 0, compute)
        B.moe_dispatch(cfg, T0, inp["x"], slot_of, xe, xs, 0, compute, xe_scale_ld=xs_ld)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ffn_ctas = max(1, sms - comm_sms)

    def call():
        B.moe_expert_ffn(cfg, counts, offsets, rows, xe, xs, w13, inp.get("w13_s"), w2, inp.get("w2_s"), ye,
                         fws, fws.numel(), err, ffn_ctas, compute, xe_scale_ld=xs_ld)

    with torch.cuda.stream(compute):
        for _ in range(max(3, args.warmup)):
            call()
    torch.cuda.synchronize()
    n = max(10, args.steps)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(compute):
        e0.record(compute)
        for _ in range(n):
            call()
        e1.record(compute)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) / n / 1e3
    c = counts.cpu().numpy().astype(np.int64)
    touched = int((c > 0).sum())
    used = int(c.sum())
    wbytes_e = expert_weight_bytes(wl)
    act_bytes = used * (H * elt + 2 * I * elt + H * io) + (used * (H // 128 + 2 * (I // 128)) * 4 if fp8 else 0)
    bytes_alg = touched * wbytes_e + act_bytes
    flops_alg = 2.0 * used * 3 * H * I
    bw = pk["hbm_gbs"] * 1e9
    tf = pk["bf16_tflops"] * 1e12 * (2.0 if fp8 else 1.0)   # fp8 peak = bf16 measured x nominal 2x
    bound = "tensor" if flops_alg / tf > bytes_alg / bw else "hbm"
    if bound == "hbm":
        achieved, peak, unit = bytes_alg / t / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = flops_alg / t / 1e12, tf / 1e12, "TFLOP/s"
    traffic = profiled_traffic("ffn", wl) if wl.num_experts == W.ALL[wl.name].num_experts else None

    # the comm-side kernels of the same ubatch, each timed alone on the whole GPU, one
    # call at a time between CUDA events with L2 flushed before each call (their
    # working sets can be smaller than L2).  The flush READS a 256 MB buffer: it leaves
    # L2 full of clean lines, so the timed kernel pays no write-back of the flush's data
    flush = torch.ones(256 << 18, dtype=torch.int32, device=dev)

    def time_call(fn, n_iter):
        with torch.cuda.stream(compute):
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_iter)]
        with torch.cuda.stream(compute):
            for a0, a1 in evs:
                flush.sum()
                a0.record(compute)
                fn()
                a1.record(compute)
        torch.cuda.synchronize()
        return sum(a0.elapsed_time(a1) for a0, a1 in evs) / n_iter / 1e3

    y0 = torch.zeros(T0, H * io, dtype=torch.uint8, device=dev)
    n_iter = max(20, args.steps)
    kern = {}
    specs = {
        "route": (lambda: B.moe_route(cfg, T0, inp["logits"], None, ids, w, 0, compute),
                  T0 * E * 4 + T0 * k * 8),
        "plan": (lambda: B.moe_plan(cfg, T0, ids, wl.capacity, wl.align, counts, offsets, slot_of, token_of, err,
                                    pws, pws.numel(), 0, compute),
                 T0 * k * 4 + T0 * kk * 4 + rows * 4 + (2 * NE + 1) * 4),
        "dispatch": (lambda: B.moe_dispatch(cfg, T0, inp["x"], slot_of, xe, xs, 0, compute, xe_scale_ld=xs_ld),
                     T0 * H * io + T0 * kk * 4 + used * H * elt + (used * (H // 128) * 4 if fp8 else 0)),
        "combine": (lambda: B.moe_combine(cfg, T0, ye, w, slot_of, y0, 0, compute),
                    used * H * io + T0 * H * io + T0 * kk * 4 + T0 * k * 4),
    }
    for name, (fn, nbytes) in specs.items():
        tk = time_call(fn, n_iter)
        kern[name] = {"us": round(tk * 1e6, 3), "algorithmic_bytes": int(nbytes),
                      "achieved_gbs": round(nbytes / tk / 1e9, 1), "frac_hbm": round(nbytes / tk / bw, 4)}
    torch.cuda.synchronize()

    # dispatch and combine back to back, as the layer runs them: each call on its own
    # buffer set (inputs, slots, weights and outputs cloned), cycling through enough sets
    # that a set's data has left L2 before it comes round again (sets x bytes >= 3 x L2)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 129 << 20) or (129 << 20)

    def time_rotating(make_set, nbytes):
        n_sets = max(2, math.ceil(3 * l2 / nbytes))
        sets = [make_set() for _ in range(n_sets)]
        # the clones ran on the current stream; the calls run on `compute`, a stream that
        # does not wait for it
        torch.cuda.synchronize()
        calls = max(3 * n_sets, 24)
        with torch.cuda.stream(compute):
            for fn in sets:
                fn()
            flush.sum()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(compute):
            e0.record(compute)
            for i in range(calls):
                sets[i % n_sets]()
            e1.record(compute)
        torch.cuda.synchronize()
        del sets
        return e0.elapsed_time(e1) / calls / 1e3, n_sets

    def dispatch_set():
        xi, si = inp["x"][:T0].clone(), slot_of.clone()
        xei, xsi = torch.empty_like(xe), (torch.empty_like(xs) if xs is not None else None)
        return lambda: B.moe_dispatch(cfg, T0, xi, si, xei, xsi, 0, compute, xe_scale_ld=xs_ld)

    def combine_set():
        yei, wi, si, yi = ye.clone(), w.clone(), slot_of.clone(), torch.empty_like(y0)
        return lambda: B.moe_combine(cfg, T0, yei, wi, si, yi, 0, compute)

    for name, make_set in (("dispatch", dispatch_set), ("combine", combine_set)):
        nbytes = kern[name]["algorithmic_bytes"]
        tk, n_sets = time_rotating(make_set, nbytes)
        kern[name]["back_to_back"] = {"us": round(tk * 1e6, 3), "achieved_gbs": round(nbytes / tk / 1e9, 1),
                                      "frac_hbm": round(nbytes / tk / bw, 4), "buffer_sets": n_sets}
    torch.cuda.synchronize()
    return {"kernel": "moe_expert_ffn (gate/up + SwiGLU, down) on ubatch 0", "bound": bound,
            "achieved": round(achieved, 2), "peak": round(peak, 2), "unit": unit,
            "frac": round(achieved / peak, 4), "peak_source": f"{src} ({'fp8 = 2x bf16 nominal ratio' if fp8 and bound == 'tensor' else 'burst'})",
            "traffic": traffic, "algorithmic_bytes": int(bytes_alg), "algorithmic_flops": flops_alg,
            "us_per_launch": round(t * 1e6, 3), "rows": used, "experts_touched": touched,
            "ctas": ffn_ctas, "comm_kernels": kern,
            "comm_kernels_note": ("us / frac_hbm: each call timed alone, whole GPU, L2 flushed (by reading 256 MB) "
                                  "before it; back_to_back: calls enqueued one after another, each on its own "
                                  "buffer set, the sets together at least 3x L2, so every call reads from HBM")}


def run_e2e(B, wl, cfg, inp, args_c, handle, comm, compute, enqueue, logits, x, y, args, world):
    """Same metric with host buffers, as a serving loop runs it: every step copies its
    logits and x from pinned host memory, runs the layer through the C ABI and copies y
    back.  Uploads and downloads run on streams of their own with two device buffer
    sets, so step i+1's inputs go up while layer i computes and step i's y comes down
    while layer i+1 computes; the timed region holds every step's copies.  The layer
    call of each buffer set is captured once into a CUDA graph, as a serving loop does
    for decode."""
    h_logits = logits.cpu().pin_memory()
    h_x = x.cpu().pin_memory()
    h_y = [torch.empty(y.shape, dtype=y.dtype, pin_memory=True) for _ in range(2)]
    Wd = {k: v for k, v in inp.items() if k.startswith("w")}
    lg2, x2, y2 = logits.clone(), x.clone(), torch.empty_like(y)  # the warm-up call reads them
    torch.cuda.synchronize()  # cloned on the current stream, read on `compute`
    ws2 = torch.empty(0, dtype=torch.uint8, device=logits.device)
    # the second buffer set shares the workspace: layers run one after another
    a2 = B.layer_args(lg2, x2, Wd, y2, None, None, ws2)
    for f in ("topk_ids", "topk_w", "err_flag", "workspace", "workspace_bytes"):
        setattr(a2, f, getattr(args_c, f))
    sets = [(logits, x, y, args_c), (lg2, x2, y2, a2)]
    graphs = []
    for _, _, _, a_b in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(compute):
            enqueue(a=a_b, cs=compute)  # eager warm call
            torch.cuda.synchronize()
            with torch.cuda.graph(g, stream=compute):
                enqueue(a=a_b, cs=compute)
        torch.cuda.synchronize()
        graphs.append(g)
    up = torch.cuda.Stream(device=logits.device)
    down = torch.cuda.Stream(device=logits.device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_out:
        e.record(down)

    def step(i):
        b = i % 2
        lg_b, x_b, y_b, a_b = sets[b]
        up.wait_event(ev_out[b])  # y of step i-2 is down: buffer set b is free
        with torch.cuda.stream(up):
            lg_b.copy_(h_logits, non_blocking=True)
            x_b.copy_(h_x, non_blocking=True)
        ev_in[b].record(up)
        compute.wait_event(ev_in[b])
        with torch.cuda.stream(compute):
            graphs[b].replay()
        ev_done[b].record(compute)
        down.wait_event(ev_done[b])
        with torch.cuda.stream(down):
            h_y[b].copy_(y_b, non_blocking=True)
        ev_out[b].record(down)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    up.wait_event(e0)
    for i in range(args.steps):
        step(i)
    compute.wait_event(ev_out[(args.steps - 1) % 2])  # the last y is on the host
    e1.record(compute)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    bi = h_logits.numel() * h_logits.element_size() + h_x.numel() * h_x.element_size()
    bo = h_y[0].numel() * h_y[0].element_size()
    return {"value": round(wl.T * world / (ms / 1e3), 1), "unit": "tokens/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": round(ms, 5),
            "pipeline": "uploads and downloads on streams of their own, two buffer sets, the layer replayed "
                        "as a CUDA graph per set"}


# --------------------------------------------------------------------------- oracle legs
def _ocfg(wl):
    import oracle
    return oracle.Config(hidden=wl.hidden, inter=wl.inter, num_experts=wl.num_experts,
                         num_shared=wl.num_shared, top_k=wl.top_k,
                         gate={"softmax": oracle.GATE_SOFTMAX, "sigmoid_grouped": oracle.GATE_SIGMOID_GROUPED,
                               "sqrt_softplus": oracle.GATE_SQRT_SOFTPLUS}[wl.gate],
                         renormalize=int(wl.renormalize), n_group=wl.n_group, topk_group=wl.topk_group,
                         routed_scale=wl.routed_scale,
                         dtype={"f32": oracle.F32, "bf16": oracle.BF16, "fp8": oracle.FP8}[wl.dtype])


def oracle_inputs(wl, device, inp=None):
    from moe_expert_dispatch_route_gb300 import synth

    if inp is None:
        inp = synth.workload_inputs(wl, device)
    Wn = {k: (v.cpu().float().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy())
          for k, v in inp.items() if k.startswith("w")}
    return inp["logits"].cpu().float().numpy(), inp["x"].cpu().float().numpy(), Wn


def oracle_sample(wl, n_tokens: int, inputs) -> float:
    """Seconds the single-threaded CPU oracle takes for the first n_tokens of the
    workload, run as two ubatches like the layer."""
    import oracle

    lg, xx, Wn = inputs
    half = (n_tokens + 1) // 2
    t0 = time.perf_counter()
    oracle.moe_layer(_ocfg(wl), lg[:n_tokens], xx[:n_tokens], Wn, split=half,
                     capacity=min(wl.capacity, half) if wl.capacity else 0, align=wl.align)
    return time.perf_counter() - t0


def sample_size(wl, seconds: float) -> int:
    per_token = 2 * (wl.top_k + wl.num_shared) * 3 * wl.hidden * wl.inter  # flops
    # the oracle's plain double-precision loops run near 2.5 GFLOP/s on one core
    return int(max(2, min(wl.T, seconds * 2.5e9 / per_token)))


def cpu_baseline(wl, inp=None, seconds: float = 12.0):
    """The oracle on about `seconds` of CPU work: the first n tokens of the workload, or
    the whole workload repeated when one pass takes less than that."""
    n = sample_size(wl, seconds)
    inputs = oracle_inputs(wl, "cuda", inp)
    secs = oracle_sample(wl, n, inputs)
    reps = 1
    while n == wl.T and secs < 0.8 * seconds:
        secs += oracle_sample(wl, n, inputs)
        reps += 1
    what = f"first {n} of {wl.T} tokens" if n < wl.T else f"all {n} tokens x {reps}"
    return {"value": round(n * reps / secs, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{what}, two ubatches {(n + 1) // 2}/{n - (n + 1) // 2}, "
                      f"single-threaded C oracle, {secs:.1f} s"}


def run_reference(args, rank, world, local):
    """The reference arm: the CPU oracle as it stands, a bounded sample per step."""
    wl = workload(args)
    if rank != 0:
        return None, wl
    n = sample_size(wl, 90.0 / max(1, args.steps + args.warmup))
    inputs = oracle_inputs(wl, "cuda" if torch.cuda.is_available() else "cpu")
    for _ in range(args.warmup):
        oracle_sample(wl, n, inputs)
    t = 0.0
    for _ in range(args.steps):
        t += oracle_sample(wl, n, inputs)
    value = n * args.steps / t
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": wl.describe()},
           "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                            "sample": f"first {n} of {wl.T} tokens per step, single-threaded C oracle"},
           "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return out, wl


def main():
    args = parse()
    rank, world, local = dist_info()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        out, _ = run_reference(args, rank, world, local)
        if out is not None:
            print(json.dumps(out), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    if args.stack > 0:
        out = run_stack(args, rank, world, local)
        if rank == 0:
            print(json.dumps(out), flush=True)
        if world > 1:
            torch.distributed.barrier()
            torch.distributed.destroy_process_group()
        return
    out, wl, inp = run_ours(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(wl, inp)
    del inp
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
