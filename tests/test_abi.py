"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every symbol moe.h declares, rejects bad arguments before touching a
device, sizes its workspaces, and its Dual-Batch Overlap schedule keeps the
dependency rules."""
import ctypes
import os
import re

import pytest

from moe_expert_dispatch_route_gb300 import binding as B
from moe_expert_dispatch_route_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["moe_route", "moe_plan", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_layer_dbo",
              "moe_dbo_create", "moe_dbo_destroy", "moe_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    L = B.lib()
    declared = _declared()
    for n in declared:
        assert hasattr(L, n), n
    assert set(declared) <= set(B.EXPORTS)


def test_status_strings():
    assert B.moe_status_string(0) == "ok"
    assert "capacity" in B.moe_status_string(6)
    assert B.moe_status_string(99) == "unknown status"


class _Buffers:
    """Pointers for the rejection tests.  With a GPU they point into one real, zeroed
    device buffer large enough for every shape below (so that, if a host check ever
    regressed, a kernel would touch valid memory and the status assertion would fail
    instead of a kernel running on a made-up address); without one they are small
    integers (no kernel can launch)."""

    def __init__(self, nbytes=1 << 30):
        import torch

        self.t = None
        if torch.cuda.is_available():
            self.t = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
            self.base = self.t.data_ptr()
        else:
            self.base = 0
        self.next = 1 << 20

    def __call__(self, misalign=0):
        """A distinct 16-byte aligned pointer (plus `misalign` bytes), 16 MB apart."""
        p = self.base + self.next + misalign
        self.next += 16 << 20
        assert self.t is None or self.next <= self.t.numel()
        return p

    def handle(self):
        return ctypes.c_void_p(B.moe_dbo_create()) if self.t is not None else ctypes.c_void_p(1)

    def close(self, h):
        if self.t is not None:
            B.moe_dbo_destroy(h.value)


def test_invalid_arguments_rejected_on_host():
    L = B.lib()
    P = _Buffers()
    cfg = B.config_of(W.QWEN3_DECODE)
    bad = B.config_of(W.QWEN3_DECODE)
    bad.top_k = 0
    assert L.moe_route(ctypes.byref(bad), 4, P(), None, P(), P(), 0, None) == 1
    assert L.moe_route(ctypes.byref(cfg), 4, None, None, P(), P(), 0, None) == 1
    assert L.moe_route(ctypes.byref(cfg), 0, None, None, None, None, 0, None) == 0  # empty batch
    assert L.moe_dispatch(ctypes.byref(cfg), 4, P(8), P(), P(), None, 0, 0, None) == 3     # misaligned x
    assert L.moe_dispatch(ctypes.byref(cfg), 4, P(), P(), P(), None, -1, 0, None) == 1     # negative scale ld
    g = B.config_of(W.DSV3)
    g.n_group = 7  # 256 % 7 != 0
    assert L.moe_route(ctypes.byref(g), 4, P(), None, P(), P(), 0, None) == 1
    f = B.config_of(W.QWEN3_PREFILL)
    f.hidden = 2000  # fp8 needs multiples of 128
    assert L.moe_dispatch(ctypes.byref(f), 4, P(), P(), P(), P(), 0, 0, None) == 3
    # expert FFN: a column-major scale stride must cover max_rows (and not be negative)
    f8 = B.config_of(W.QWEN3_PREFILL)
    ffn = lambda ld: L.moe_expert_ffn(ctypes.byref(f8), P(), P(), 100, P(), P(), ld, P(), P(), P(), P(), P(), P(),
                                      1 << 20, None, 0, None)
    assert ffn(5) == 1 and ffn(-1) == 1
    # plan: workspace required when the batch spans several chunks (ids / slots of
    # 100000 tokens would not fit the test buffer: the call must return first)
    assert B.moe_plan_workspace_size(cfg, 100000) > 0
    assert L.moe_plan(ctypes.byref(cfg), 100000, P(), 0, 128, P(), P(), P(), P(), P(), None, 0, 0, None) == 4
    # layer: workspace too small (the tiny layer: every buffer fits a 16 MB slot)
    tiny = B.config_of(W.TINY)
    h = P.handle()
    args = B.MoeLayerArgs(P(), None, P(), P(), None, P(), None, P(), P(), P(), None, P(), 1024)
    assert L.moe_layer_dbo(h, ctypes.byref(tiny), ctypes.byref(args), 64, 0, 4, 0, 128, 0, None, None) == 4
    P.close(h)
    if P.t is not None:  # nothing was written
        import torch

        torch.cuda.synchronize()
        assert int(P.t.count_nonzero().item()) == 0


def test_plan_rows_and_workspace_sizes():
    cfg = B.config_of(W.DSV2LITE)
    NE, kk = 66, 8
    assert B.moe_plan_rows(cfg, 512, 0, 128) == 512 * kk + NE * 127
    assert B.moe_plan_rows(cfg, 512, 256, 128) == NE * 256
    assert B.moe_plan_rows(cfg, 512, 0, 1) == 512 * kk
    assert B.moe_plan_workspace_size(cfg, 64) == 0   # one chunk: no scratch
    ws = B.moe_layer_workspace_size(cfg, 4096, 0, 128)
    assert ws > 2 * B.moe_plan_rows(cfg, 4096, 0, 128) * 2048 * 2 * 2  # xe + ye per ubatch
    assert B.moe_ffn_workspace_size(B.config_of(W.QWEN3_PREFILL), 1000) >= 1000 * 768


def _events(sched):
    """For each event id: (stream, position) of its record."""
    return {ev: (st, i) for i, (st, op, ub, ev) in enumerate(sched) if op == 5}


def test_dbo_schedule_dependencies():
    s = B.moe_dbo_schedule(True)
    ops = [(st, B.OPS[op], ub, ev) for st, op, ub, ev in s]
    rec = _events(s)

    def pos(name, ub):
        return next(i for i, o in enumerate(ops) if o[1] == name and o[2] == ub)

    # dispatch/route/plan and combine on the comm stream, experts on compute
    for name in ("route", "plan", "dispatch", "combine"):
        for ub in (0, 1):
            assert ops[pos(name, ub)][0] == 1
    assert ops[pos("ffn", 0)][0] == 0 and ops[pos("ffn", 1)][0] == 0

    def waits_before(i, stream):
        return [o[3] for o in ops[:i] if o[0] == stream and o[1] == "wait"]

    # ffn(u) waits for dispatch(u): the event it waits on is recorded right after dispatch(u)
    for ub in (0, 1):
        evs = waits_before(pos("ffn", ub), 0)
        ev = evs[-1]
        st, at = rec[ev]
        assert st == 1 and ops[at - 1][1] == "dispatch" and ops[at - 1][2] == ub
    # combine(0) waits on an event recorded right after ffn(0) -- BEFORE ffn(1) is
    # enqueued, so it does not cover the other ubatch's compute
    ev = waits_before(pos("combine", 0), 1)[-1]
    st, at = rec[ev]
    assert st == 0 and ops[at - 1][1] == "ffn" and ops[at - 1][2] == 0
    assert at < pos("ffn", 1)
    # the comm-side work of ubatch 1 is not behind ffn(0): no wait on the comm stream
    # between the fork and dispatch(1) refers to a compute-stream event other than the fork
    for e in waits_before(pos("dispatch", 1), 1):
        assert rec[e][1] < pos("ffn", 0)
    # join: the last op makes the compute stream wait for the comm stream's last record
    last = ops[-1]
    assert last[0] == 0 and last[1] == "wait" and rec[last[3]][0] == 1
    assert max(i for i, o in enumerate(ops) if o[0] == 1) == rec[last[3]][1]
    # every ubatch runs the same steps (the two ubatches perform equal numbers of yields)
    for name in ("route", "plan", "dispatch", "ffn", "combine"):
        assert sum(1 for o in ops if o[1] == name) == 2


def test_unsplit_schedule_is_one_stream():
    s = B.moe_dbo_schedule(False)
    assert [B.OPS[o[1]] for o in s] == ["route", "plan", "dispatch", "ffn", "combine"]
    assert all(o[0] == 0 for o in s)


def _graph(sched):
    """Dependency edges of an enqueue schedule: stream order plus event waits (a wait
    depends on the op recorded just before the latest record of that event)."""
    ops = [(st, B.OPS[op], ub, ev) for st, op, ub, ev in sched]
    deps = {i: set() for i in range(len(ops))}
    last_on = {}
    last_rec = {}
    for i, (st, name, ub, ev) in enumerate(ops):
        if st in last_on:
            deps[i].add(last_on[st])
        if name == "wait":
            deps[i].add(last_rec[ev])
        if name == "record":
            last_rec[ev] = i
        last_on[st] = i
    return ops, deps


def _ancestors(deps, i):
    seen, todo = set(), [i]
    while todo:
        j = todo.pop()
        for d in deps[j]:
            if d not in seen:
                seen.add(d)
                todo.append(d)
    return seen


def _find(ops, name, ub, nth=0):
    return [i for i, o in enumerate(ops) if o[1] == name and o[2] == ub][nth]


def test_stack_schedule_overlap_rule_and_prefix_variant():
    L = 3
    for before in (True, False):
        ops, deps = _graph(B.moe_stack_schedule(L, True, before))
        for l in range(L):
            a0, a1 = _find(ops, "standin", 0, l), _find(ops, "standin", 1, l)
            d0 = _find(ops, "dispatch", 0, l)
            f0, f1 = _find(ops, "ffn", 0, l), _find(ops, "ffn", 1, l)
            c0, c1 = _find(ops, "combine", 0, l), _find(ops, "combine", 1, l)
            anc_d0, anc_c0 = _ancestors(deps, d0), _ancestors(deps, c0)
            # data dependencies hold in both placements
            assert a0 in anc_d0 and d0 in _ancestors(deps, f0) and f0 in anc_c0
            assert f1 in _ancestors(deps, c1)
            if l + 1 < L:
                assert c0 in _ancestors(deps, _find(ops, "standin", 0, l + 1))
            # the fix: dispatch(0) does not wait for the other ubatch's stand-in, and
            # combine(0) not for the other ubatch's experts; the old placement does
            assert (a1 not in anc_d0) == before
            assert (f1 not in anc_c0) == before
        # everything joins back to the compute stream
        assert ops[-1][0] == 0 and ops[-1][1] == "wait"
    assert all(o[0] == 0 for o in B.moe_stack_schedule(2, False, True))


def test_fused_schedule_has_no_combine_and_keeps_the_overlap():
    s = B.moe_dbo_schedule(True, B.LAYER_FUSED)
    ops, deps = _graph(s)
    assert not any(o[1] == "combine" for o in ops)
    for ub in (0, 1):
        for name in ("route", "plan", "dispatch"):
            assert ops[_find(ops, name, ub)][0] == 1  # comm stream
        f = _find(ops, "ffn", ub)
        assert ops[f][0] == 0 and _find(ops, "dispatch", ub) in _ancestors(deps, f)
    # ubatch 1's route/plan/dispatch do not wait for ubatch 0's experts
    assert _find(ops, "ffn", 0) not in _ancestors(deps, _find(ops, "dispatch", 1))
    # joined back to the compute stream
    assert ops[-1][0] == 0 and ops[-1][1] == "wait"
    assert [B.OPS[o[1]] for o in B.moe_dbo_schedule(False, B.LAYER_FUSED)] == ["route", "plan", "dispatch", "ffn"]
