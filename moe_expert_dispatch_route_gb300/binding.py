"""Python binding of libmoe_gb300 (ctypes): the C ABI's calls under the same names.

Argument marshalling only -- every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory and
streams); a call returns after enqueueing, like the C call.  A non-zero
``moe_status`` raises :class:`MoeError`.  Importing this module loads the in-tree
shared library and fails loudly when it is missing or cannot be built.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

F32, BF16, FP8_E4M3 = 0, 1, 2
GATE_SOFTMAX, GATE_SIGMOID_GROUPED, GATE_SQRT_SOFTPLUS = 0, 1, 2
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_ALIGNMENT",
          4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA", 6: "MOE_ERR_CAPACITY", 7: "MOE_ERR_BAD_INDEX",
          8: "MOE_ERR_TIMEOUT"}
OPS = {0: "route", 1: "plan", 2: "dispatch", 3: "ffn", 4: "combine", 5: "record", 6: "wait", 7: "standin"}


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)}")


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("num_shared", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("routed_scale", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


class MoeStackArgs(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("out", ctypes.c_void_p), ("logits", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("wa", ctypes.c_void_p), ("w13", ctypes.c_void_p),
                ("w13_scale", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("w2_scale", ctypes.c_void_p),
                ("err_flag", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


class MoeLayerArgs(ctypes.Structure):
    _fields_ = [("logits", ctypes.c_void_p), ("bias", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("w13", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p), ("w2", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("y", ctypes.c_void_p), ("topk_ids", ctypes.c_void_p),
                ("topk_w", ctypes.c_void_p), ("err_flag", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


def config(hidden, inter, num_experts, num_shared, top_k, gate=GATE_SOFTMAX, renormalize=1,
           n_group=1, topk_group=1, routed_scale=1.0, dtype=BF16) -> MoeConfig:
    return MoeConfig(hidden, inter, num_experts, num_shared, top_k, gate, int(renormalize), n_group,
                     topk_group, float(routed_scale), dtype)


def config_of(wl) -> MoeConfig:
    """MoeConfig of a workloads.Workload."""
    gate = {"softmax": GATE_SOFTMAX, "sigmoid_grouped": GATE_SIGMOID_GROUPED, "sqrt_softplus": GATE_SQRT_SOFTPLUS}
    return config(wl.hidden, wl.inter, wl.num_experts, wl.num_shared, wl.top_k, gate[wl.gate],
                  int(wl.renormalize), wl.n_group, wl.topk_group, wl.routed_scale,
                  {"f32": F32, "bf16": BF16, "fp8": FP8_E4M3}[wl.dtype])


_P, _I32, _I64, _SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_CFG = ctypes.POINTER(MoeConfig)
_SIGS = {
    "moe_route": (_I32, [_CFG, _I32, _P, _P, _P, _P, _I32, _P]),
    "moe_route_hash": (_I32, [_CFG, _I32, _P, _P, _P, _I32, _P, _P, _I32, _P]),
    "moe_plan_rows": (_SZ, [_CFG, _I32, _I32, _I32]),
    "moe_plan_workspace_size": (_SZ, [_CFG, _I32]),
    "moe_plan": (_I32, [_CFG, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P, _P, _SZ, _I32, _P]),
    "moe_plan_noalloc": (_I32, [_CFG, _I32, _P, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P]),
    "moe_dispatch": (_I32, [_CFG, _I32, _P, _P, _P, _P, _I64, _I32, _P]),
    "moe_ffn_workspace_size": (_SZ, [_CFG, _I64]),
    "moe_expert_ffn": (_I32, [_CFG, _P, _P, _I64, _P, _P, _I64, _P, _P, _P, _P, _P, _P, _SZ, _P, _I32, _P]),
    "moe_combine": (_I32, [_CFG, _I32, _P, _P, _P, _P, _I32, _P]),
    "moe_dbo_create": (_I32, [ctypes.POINTER(_P)]),
    "moe_dbo_destroy": (None, [_P]),
    "moe_layer_workspace_size": (_SZ, [_CFG, _I32, _I32, _I32]),
    "moe_layer_dbo": (_I32, [_P, _CFG, ctypes.POINTER(MoeLayerArgs), _I32, _I32, _I32, _I32, _I32, _I32,
                             _P, _P]),
    "moe_dbo_schedule": (_I32, [_I32, _P, _I32]),
    "moe_layer_dbo_ex": (_I32, [_P, _CFG, ctypes.POINTER(MoeLayerArgs), _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                                _P, _P]),
    "moe_dbo_schedule_ex": (_I32, [_I32, _I32, _P, _I32]),
    "moe_stack_workspace_size": (_SZ, [_CFG, _I32, _I32, _I32]),
    "moe_stack_dbo": (_I32, [_P, _CFG, ctypes.POINTER(MoeStackArgs), _I32, _I32, _I32, _I32, _I32, _I32, _I32,
                             _I32, _P, _P]),
    "moe_stack_schedule": (_I32, [_I32, _I32, _I32, _P, _I32]),
    "moe_status_string": (ctypes.c_char_p, [_I32]),
    "moe_debug_inject_wait": (_I32, [_I32, _I64]),
    "moe_comm_error": (_I32, [_P, _I32]),
}
EXPORTS = tuple(_SIGS)

_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmoe_gb300 (built in-tree on first use if stale or missing)."""
    global _lib
    if _lib is None:
        path = _build.build()
        if not os.path.exists(path):
            raise ImportError(f"libmoe_gb300 not found at {path}")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(st: int, where: str):
    if st != 0:
        raise MoeError(st, where)


def moe_route(cfg, T, logits, bias, topk_ids, topk_w, max_ctas=0, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg), T, _ptr(logits), _ptr(bias), _ptr(topk_ids), _ptr(topk_w),
                           max_ctas, _stream(stream)), "moe_route")


def moe_route_hash(cfg, T, logits, token_ids, table, topk_ids, topk_w, max_ctas=0, stream=None):
    vocab = table.shape[0] if table is not None else 0
    _check(lib().moe_route_hash(ctypes.byref(cfg), T, _ptr(logits), _ptr(token_ids), _ptr(table), vocab,
                                _ptr(topk_ids), _ptr(topk_w), max_ctas, _stream(stream)), "moe_route_hash")


def moe_plan_rows(cfg, T, capacity=0, align=1) -> int:
    return int(lib().moe_plan_rows(ctypes.byref(cfg), T, capacity, align))


def moe_plan_workspace_size(cfg, T) -> int:
    return int(lib().moe_plan_workspace_size(ctypes.byref(cfg), T))


def moe_plan(cfg, T, topk_ids, capacity, align, counts, offsets, slot_of, token_of, err_flag, ws=None,
             ws_bytes=0, max_ctas=0, stream=None):
    if ws is not None and not ws_bytes:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().moe_plan(ctypes.byref(cfg), T, _ptr(topk_ids), capacity, align, _ptr(counts), _ptr(offsets),
                          _ptr(slot_of), _ptr(token_of), _ptr(err_flag), _ptr(ws), ws_bytes, max_ctas,
                          _stream(stream)), "moe_plan")


def moe_plan_noalloc(cfg, T, topk_ids, capacity, align, counts, offsets, slot_of, token_of, err_flag,
                     max_ctas=0, stream=None):
    """moe_plan without a workspace (scratch lives in the library; see moe.h for the limit)."""
    _check(lib().moe_plan_noalloc(ctypes.byref(cfg), T, _ptr(topk_ids), capacity, align, _ptr(counts),
                                  _ptr(offsets), _ptr(slot_of), _ptr(token_of), _ptr(err_flag), max_ctas,
                                  _stream(stream)), "moe_plan_noalloc")


def moe_dispatch(cfg, T, x, slot_of, xe, xe_scale=None, max_ctas=0, stream=None, xe_scale_ld=0):
    _check(lib().moe_dispatch(ctypes.byref(cfg), T, _ptr(x), _ptr(slot_of), _ptr(xe), _ptr(xe_scale),
                              xe_scale_ld, max_ctas, _stream(stream)), "moe_dispatch")


def moe_ffn_workspace_size(cfg, max_rows) -> int:
    return int(lib().moe_ffn_workspace_size(ctypes.byref(cfg), max_rows))


def moe_expert_ffn(cfg, counts, offsets, max_rows, xe, xe_scale, w13, w13_scale, w2, w2_scale, ye, ws,
                   ws_bytes=0, err_flag=None, max_ctas=0, stream=None, xe_scale_ld=0):
    if ws is not None and not ws_bytes:
        ws_bytes = ws.numel() * ws.element_size()
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _ptr(counts), _ptr(offsets), max_rows, _ptr(xe),
                                _ptr(xe_scale), xe_scale_ld, _ptr(w13), _ptr(w13_scale), _ptr(w2), _ptr(w2_scale),
                                _ptr(ye), _ptr(ws), ws_bytes, _ptr(err_flag), max_ctas, _stream(stream)),
           "moe_expert_ffn")


def moe_combine(cfg, T, ye, topk_w, slot_of, y, max_ctas=0, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), T, _ptr(ye), _ptr(topk_w), _ptr(slot_of), _ptr(y), max_ctas,
                             _stream(stream)), "moe_combine")


def moe_dbo_create() -> int:
    h = ctypes.c_void_p()
    _check(lib().moe_dbo_create(ctypes.byref(h)), "moe_dbo_create")
    return h.value


def moe_dbo_destroy(h: int):
    lib().moe_dbo_destroy(h)


def moe_layer_workspace_size(cfg, T, capacity=0, align=128) -> int:
    return int(lib().moe_layer_workspace_size(ctypes.byref(cfg), T, capacity, align))


def moe_layer_dbo(handle, cfg, args: MoeLayerArgs, T, split=0, min_tokens=4, capacity=0, align=128,
                  comm_sms=0, compute=None, comm=None):
    cs = _stream(compute)
    ms = _stream(comm) if comm is not None else cs
    _check(lib().moe_layer_dbo(handle, ctypes.byref(cfg), ctypes.byref(args), T, split, min_tokens, capacity,
                               align, comm_sms, cs, ms), "moe_layer_dbo")


LAYER_FUSED_GATHER, LAYER_FUSED_COMBINE, LAYER_FUSED = 1, 2, 3


def moe_layer_dbo_ex(handle, cfg, args: MoeLayerArgs, T, split=0, min_tokens=4, capacity=0, align=128,
                     comm_sms=0, flags=0, compute=None, comm=None):
    cs = _stream(compute)
    ms = _stream(comm) if comm is not None else cs
    _check(lib().moe_layer_dbo_ex(handle, ctypes.byref(cfg), ctypes.byref(args), T, split, min_tokens, capacity,
                                  align, comm_sms, flags, cs, ms), "moe_layer_dbo_ex")


def moe_dbo_schedule(two_ubatches: bool, flags: int = 0):
    n = lib().moe_dbo_schedule_ex(int(two_ubatches), flags, None, 0)
    buf = (ctypes.c_int32 * (4 * n))()
    lib().moe_dbo_schedule_ex(int(two_ubatches), flags, buf, n)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]


def moe_debug_inject_wait(enable: bool, timeout_ns: int = 0):
    """Test hook: FFN and combine kernels launched while enabled let a bounded wait run
    out (see moe.h)."""
    _check(lib().moe_debug_inject_wait(int(enable), int(timeout_ns)), "moe_debug_inject_wait")


def moe_comm_error(clear: bool = False) -> int:
    """The sticky error word of moe_combine (synchronises the device)."""
    code = ctypes.c_int32(0)
    _check(lib().moe_comm_error(ctypes.byref(code), int(clear)), "moe_comm_error")
    return int(code.value)


def moe_status_string(st: int) -> str:
    return lib().moe_status_string(st).decode()


def layer_args(logits, x, weights: dict, y, topk_ids, topk_w, workspace, bias=None, err_flag=None):
    """MoeLayerArgs from tensors (weights: {"w13","w2"} or {"w13_q","w13_s","w2_q","w2_s"})."""
    w13 = weights.get("w13", weights.get("w13_q"))
    w2 = weights.get("w2", weights.get("w2_q"))
    return MoeLayerArgs(_ptr(logits), _ptr(bias), _ptr(x), _ptr(w13), _ptr(weights.get("w13_s")), _ptr(w2),
                        _ptr(weights.get("w2_s")), _ptr(y), _ptr(topk_ids), _ptr(topk_w), _ptr(err_flag),
                        _ptr(workspace), workspace.numel() * workspace.element_size())


def moe_stack_workspace_size(cfg, T, capacity=0, align=128) -> int:
    return int(lib().moe_stack_workspace_size(ctypes.byref(cfg), T, capacity, align))


class StackArgs:
    """moe_stack_args from tensors; keeps the host pointer arrays alive.
    layers: list of dicts with "logits", "wa" and the weights ({"w13","w2"} or fp8 keys)."""

    def __init__(self, x, out, layers, workspace, bias=None, err_flag=None):
        L = len(layers)
        arr = lambda vals: (ctypes.c_void_p * L)(*[_ptr(v) for v in vals])
        self._keep = [arr([ly["logits"] for ly in layers]), arr([ly["wa"] for ly in layers]),
                      arr([ly.get("w13", ly.get("w13_q")) for ly in layers]),
                      arr([ly.get("w13_s") for ly in layers]),
                      arr([ly.get("w2", ly.get("w2_q")) for ly in layers]),
                      arr([ly.get("w2_s") for ly in layers])]
        lg, wa, w13, w13s, w2, w2s = self._keep
        self.c = MoeStackArgs(_ptr(x), _ptr(out), ctypes.cast(lg, ctypes.c_void_p), _ptr(bias),
                              ctypes.cast(wa, ctypes.c_void_p), ctypes.cast(w13, ctypes.c_void_p),
                              ctypes.cast(w13s, ctypes.c_void_p), ctypes.cast(w2, ctypes.c_void_p),
                              ctypes.cast(w2s, ctypes.c_void_p), _ptr(err_flag), _ptr(workspace),
                              workspace.numel() * workspace.element_size())
        self.L = L


def moe_stack_dbo(handle, cfg, args: StackArgs, T, split=0, min_tokens=4, capacity=0, align=128, comm_sms=0,
                  event_before_yield=1, compute=None, comm=None):
    cs = _stream(compute)
    ms = _stream(comm) if comm is not None else cs
    _check(lib().moe_stack_dbo(handle, ctypes.byref(cfg), ctypes.byref(args.c), args.L, T, split, min_tokens,
                               capacity, align, comm_sms, int(event_before_yield), cs, ms), "moe_stack_dbo")


def moe_stack_schedule(layers: int, two_ubatches: bool = True, event_before_yield: bool = True):
    n = lib().moe_stack_schedule(layers, int(two_ubatches), int(event_before_yield), None, 0)
    buf = (ctypes.c_int32 * (4 * n))()
    lib().moe_stack_schedule(layers, int(two_ubatches), int(event_before_yield), buf, n)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]
