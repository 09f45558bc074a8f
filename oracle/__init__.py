"""CPU oracle for the MoE layer -- TEST INFRASTRUCTURE ONLY.

A thin ctypes wrapper (argument marshalling only) around ``moe_oracle.c``: a plain,
single-threaded C definition of route -> plan -> dispatch -> expert FFN -> combine,
in double precision, optionally run as two micro-batches.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It shares no code with the CUDA library and never calls it.

Functions that follow a page of the Dual-Batch Overlap (DBO) material cite it in
``moe_oracle.c``; every arithmetic choice the pages leave open is a "reading"
stated there.  Parity of every function here is pinned by ``tests/test_oracle_*``
(brute force, closed forms, invariants and library routines); nothing here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, FP8 = 0, 1, 2
GATE_SOFTMAX, GATE_SIGMOID_GROUPED, GATE_SQRT_SOFTPLUS = 0, 1, 2
OK, BAD_INDEX, CAPACITY = 0, 1, 2
QG = 128


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into _liboracle.so (gcc, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("inter", ctypes.c_int32),
                ("num_experts", ctypes.c_int32), ("num_shared", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("routed_scale", ctypes.c_double),
                ("dtype", ctypes.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            L.orc_bf16_round.argtypes = [ctypes.c_float]
            L.orc_bf16_round.restype = ctypes.c_float
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_encode.argtypes = [ctypes.c_double]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_fp8_scale_exp.argtypes = [ctypes.c_float]
            L.orc_fp8_scale_exp.restype = i32
            L.orc_spec_exp.argtypes = [ctypes.c_float]
            L.orc_spec_exp.restype = ctypes.c_float
            L.orc_spec_sigmoid.argtypes = [ctypes.c_float]
            L.orc_spec_sigmoid.restype = ctypes.c_float
            L.orc_spec_log1p.argtypes = [ctypes.c_float]
            L.orc_spec_log1p.restype = ctypes.c_float
            L.orc_spec_sqrt_softplus.argtypes = [ctypes.c_float]
            L.orc_spec_sqrt_softplus.restype = ctypes.c_float
            L.orc_route_hash.argtypes = [P, i32, P, P, P, i32, P, P]
            L.orc_route_hash.restype = None
            L.orc_route.argtypes = [P, i32, P, P, P, P]
            L.orc_route.restype = None
            L.orc_plan.argtypes = [i32, i32, i32, i32, P, i32, i32, P, P, P, P]
            L.orc_plan.restype = i32
            L.orc_quant_row_fp8.argtypes = [i32, P, P, P]
            L.orc_quant_row_fp8.restype = None
            L.orc_dispatch.argtypes = [P, i32, P, P, P, P, P]
            L.orc_dispatch.restype = None
            L.orc_expert_ffn.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P]
            L.orc_expert_ffn.restype = None
            L.orc_combine.argtypes = [P, i32, P, P, P, P]
            L.orc_combine.restype = None
            L.orc_token_output.argtypes = [P, P, P, P, P, P, P, P, P, P, P]
            L.orc_token_output.restype = None
            L.orc_max_rows.argtypes = [P, i32, i32, i32]
            L.orc_max_rows.restype = ctypes.c_int64
            L.orc_moe_layer.argtypes = [P, i32, i32, P, P, P, P, P, P, P, P, P, i32, i32, P, P, P]
            L.orc_moe_layer.restype = i32
            L.orc_combine_resid.argtypes = [P, i32, P, P, P, P, P]
            L.orc_combine_resid.restype = None
            L.orc_standin.argtypes = [P, i32, P, P, P]
            L.orc_standin.restype = None
            L.orc_moe_stack.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P, P, P, P, i32, i32, P]
            L.orc_moe_stack.restype = i32
            _lib = L
    return _lib


@dataclass(frozen=True)
class Config:
    """Shape of one MoE layer (the oracle's own copy; no code shared with the library)."""
    hidden: int
    inter: int
    num_experts: int
    num_shared: int
    top_k: int
    gate: int = GATE_SOFTMAX
    renormalize: int = 1
    n_group: int = 1
    topk_group: int = 1
    routed_scale: float = 1.0
    dtype: int = BF16

    def c(self) -> _Cfg:
        return _Cfg(self.hidden, self.inter, self.num_experts, self.num_shared, self.top_k,
                    self.gate, self.renormalize, self.n_group, self.topk_group,
                    float(self.routed_scale), self.dtype)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _u8(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint8)


# ---- number formats -------------------------------------------------------
def bf16_round(x: float) -> float:
    return lib().orc_bf16_round(float(x))


def e4m3_decode(c: int) -> float:
    return lib().orc_e4m3_decode(int(c))


def e4m3_encode(v: float) -> int:
    return lib().orc_e4m3_encode(float(v))


def fp8_scale_exp(amax: float) -> int:
    return lib().orc_fp8_scale_exp(float(amax))


def spec_exp(x: float) -> float:
    return lib().orc_spec_exp(float(x))


def spec_sigmoid(x: float) -> float:
    return lib().orc_spec_sigmoid(float(x))


def spec_log1p(y: float) -> float:
    return lib().orc_spec_log1p(float(y))


def spec_sqrt_softplus(x: float) -> float:
    return lib().orc_spec_sqrt_softplus(float(x))


def quant_row_fp8(v):
    v = _f32(v)
    n = v.shape[-1]
    q = np.zeros(n, np.uint8)
    s = np.zeros(n // QG, np.float32)
    lib().orc_quant_row_fp8(n, _p(v), _p(q), _p(s))
    return q, s


# ---- the layer's steps ------------------------------------------------------
def route(cfg: Config, logits, bias=None):
    logits = _f32(logits)
    T = logits.shape[0]
    ids = np.zeros((T, cfg.top_k), np.int32)
    w = np.zeros((T, cfg.top_k), np.float64)
    bias = _f32(bias)
    c = cfg.c()
    lib().orc_route(ctypes.byref(c), T, _p(logits), _p(bias), _p(ids), _p(w))
    return ids, w


def route_hash(cfg: Config, logits, token_ids, table):
    """Hash routing: the experts of token t are table[token_ids[t]] (see moe_oracle.c)."""
    logits = _f32(logits)
    token_ids = _i32(token_ids)
    table = _i32(table)
    T = logits.shape[0]
    ids = np.zeros((T, cfg.top_k), np.int32)
    w = np.zeros((T, cfg.top_k), np.float64)
    c = cfg.c()
    lib().orc_route_hash(ctypes.byref(c), T, _p(logits), _p(token_ids), _p(table), table.shape[0], _p(ids), _p(w))
    return ids, w


def max_rows(cfg: Config, T: int, capacity: int = 0, align: int = 1) -> int:
    c = cfg.c()
    return int(lib().orc_max_rows(ctypes.byref(c), T, capacity, align))


def plan(cfg: Config, ids, capacity: int = 0, align: int = 1):
    ids = _i32(ids)
    T = ids.shape[0]
    E, S, k = cfg.num_experts, cfg.num_shared, cfg.top_k
    rows = max_rows(cfg, T, capacity, align)
    counts = np.zeros(E + S, np.int32)
    offsets = np.zeros(E + S + 1, np.int32)
    slot_of = np.zeros((T, k + S), np.int32)
    token_of = np.full(max(rows, 1), -7, np.int32)
    st = lib().orc_plan(T, k, E, S, _p(ids), capacity, align, _p(counts), _p(offsets),
                        _p(slot_of), _p(token_of))
    return dict(status=int(st), counts=counts, offsets=offsets, slot_of=slot_of,
                token_of=token_of[: offsets[-1]], rows=int(offsets[-1]))


def dispatch(cfg: Config, x, slot_of, rows: int):
    x = _f32(x)
    slot_of = _i32(slot_of)
    T, H = x.shape
    c = cfg.c()
    if cfg.dtype == FP8:
        xe_q = np.zeros((rows, H), np.uint8)
        xe_s = np.zeros((rows, H // QG), np.float32)
        lib().orc_dispatch(ctypes.byref(c), T, _p(x), _p(slot_of), None, _p(xe_q), _p(xe_s))
        return dict(xe_q=xe_q, xe_s=xe_s)
    xe = np.zeros((rows, H), np.float32)
    lib().orc_dispatch(ctypes.byref(c), T, _p(x), _p(slot_of), _p(xe), None, None)
    return dict(xe=xe)


def expert_ffn(cfg: Config, counts, offsets, xe=None, xe_q=None, xe_s=None, weights=None):
    """weights: dict with w13/w2 (float values) or w13_q/w13_s/w2_q/w2_s (fp8)."""
    W = weights
    rows = int(offsets[-1])
    H = cfg.hidden
    ye = np.zeros((max(rows, 1), H), np.float32)
    c = cfg.c()
    counts = _i32(counts)
    offsets = _i32(offsets)
    args = [_f32(xe), _u8(xe_q), _f32(xe_s), _f32(W.get("w13")), _u8(W.get("w13_q")),
            _f32(W.get("w13_s")), _f32(W.get("w2")), _u8(W.get("w2_q")), _f32(W.get("w2_s"))]
    lib().orc_expert_ffn(ctypes.byref(c), _p(counts), _p(offsets),
                         *[_p(a) for a in args], _p(ye))
    return ye[:rows]


def combine(cfg: Config, ye, w, slot_of):
    ye = _f32(ye)
    w = _f64(w)
    slot_of = _i32(slot_of)
    T = slot_of.shape[0]
    y = np.zeros((T, cfg.hidden), np.float32)
    c = cfg.c()
    lib().orc_combine(ctypes.byref(c), T, _p(ye), _p(w), _p(slot_of), _p(y))
    return y


def token_output(cfg: Config, x_t, ids_t, w_t, weights):
    W = weights
    y = np.zeros(cfg.hidden, np.float32)
    c = cfg.c()
    args = [_f32(W.get("w13")), _u8(W.get("w13_q")), _f32(W.get("w13_s")), _f32(W.get("w2")),
            _u8(W.get("w2_q")), _f32(W.get("w2_s"))]
    x_t = _f32(x_t)
    ids_t = _i32(ids_t)
    w_t = _f64(w_t)
    lib().orc_token_output(ctypes.byref(c), _p(x_t), _p(ids_t), _p(w_t), *[_p(a) for a in args], _p(y))
    return y


def moe_layer(cfg: Config, logits, x, weights, bias=None, split: int = 0, capacity: int = 0,
              align: int = 1):
    logits = _f32(logits)
    x = _f32(x)
    T = logits.shape[0]
    W = weights
    ids = np.zeros((T, cfg.top_k), np.int32)
    w = np.zeros((T, cfg.top_k), np.float64)
    y = np.zeros((T, cfg.hidden), np.float32)
    c = cfg.c()
    bias = _f32(bias)
    args = [_f32(W.get("w13")), _u8(W.get("w13_q")), _f32(W.get("w13_s")), _f32(W.get("w2")),
            _u8(W.get("w2_q")), _f32(W.get("w2_s"))]
    st = lib().orc_moe_layer(ctypes.byref(c), T, split, _p(logits), _p(bias), _p(x),
                             *[_p(a) for a in args], capacity, align, _p(ids), _p(w), _p(y))
    return dict(status=int(st), ids=ids, w=w, y=y)


def combine_resid(cfg: Config, ye, w, slot_of, resid):
    """combine with a residual added before the single rounding."""
    ye = _f32(ye)
    w = _f64(w)
    slot_of = _i32(slot_of)
    resid = _f32(resid)
    T = slot_of.shape[0]
    y = np.zeros((T, cfg.hidden), np.float32)
    c = cfg.c()
    lib().orc_combine_resid(ctypes.byref(c), T, _p(ye), _p(w), _p(slot_of), _p(resid), _p(y))
    return y


def standin(cfg: Config, x, wa):
    """a = x + x . Wa^T, rounded once (the stand-in for a layer's non-MoE compute)."""
    x = _f32(x)
    wa = _f32(wa)
    a = np.zeros_like(x)
    c = cfg.c()
    lib().orc_standin(ctypes.byref(c), x.shape[0], _p(x), _p(wa), _p(a))
    return a


def moe_stack(cfg: Config, x0, layers, bias=None, split: int = 0, capacity: int = 0, align: int = 1):
    """L layers; layers[l] = dict(wa=..., logits=..., and the weights as for moe_layer)."""
    x0 = _f32(x0)
    T = x0.shape[0]
    L = len(layers)
    keep = []

    def arr(key, conv):
        vals = [conv(ly.get(key)) for ly in layers]
        keep.append(vals)
        if all(v is None for v in vals):
            return None
        a = (ctypes.c_void_p * L)(*[None if v is None else v.ctypes.data for v in vals])
        keep.append(a)
        return a

    wa = arr("wa", _f32)
    lg = arr("logits", _f32)
    ptrs = [arr("w13", _f32), arr("w13_q", _u8), arr("w13_s", _f32), arr("w2", _f32), arr("w2_q", _u8),
            arr("w2_s", _f32)]
    bias = _f32(bias)
    out = np.zeros_like(x0)
    c = cfg.c()
    st = lib().orc_moe_stack(ctypes.byref(c), L, T, split, _p(x0), wa, lg, _p(bias), *ptrs, capacity, align,
                             _p(out))
    return dict(status=int(st), y=out)
