"""Shared test plumbing: workload -> oracle config, tensor conversions, tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_expert_dispatch_route_gb300 import synth, workloads

# Tolerances on the layer output y (and on ye).  bf16 and fp8: the stated contract
# (max-abs 2e-2 and relative L2 1e-2; fp8 relative L2 3e-2).  fp32: the kernel
# accumulates in fp32 over K <= 2048 terms; typical relative error sqrt(K) * 2^-24
# ~ 3e-6, so relative L2 1e-5 (and max-abs 1e-5 of the largest output).
TOL = {"bf16": dict(max_abs=2e-2, rel_l2=1e-2), "fp8": dict(max_abs=None, rel_l2=3e-2),
       "f32": dict(max_abs_rel=1e-5, rel_l2=1e-5)}


def ocfg(wl: workloads.Workload) -> oracle.Config:
    return oracle.Config(hidden=wl.hidden, inter=wl.inter, num_experts=wl.num_experts,
                         num_shared=wl.num_shared, top_k=wl.top_k,
                         gate={"softmax": oracle.GATE_SOFTMAX, "sigmoid_grouped": oracle.GATE_SIGMOID_GROUPED,
                               "sqrt_softplus": oracle.GATE_SQRT_SOFTPLUS}[wl.gate],
                         renormalize=int(wl.renormalize), n_group=wl.n_group, topk_group=wl.topk_group,
                         routed_scale=wl.routed_scale,
                         dtype={"f32": oracle.F32, "bf16": oracle.BF16, "fp8": oracle.FP8}[wl.dtype])


def np_f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float32).numpy()


def np_weights(W: dict, experts=None) -> dict:
    """Host numpy copies of the weights (optionally only some experts, zeros elsewhere)."""
    out = {}
    for k, v in W.items():
        if experts is None:
            src = v.detach().cpu()
        else:
            src = torch.zeros(v.shape, dtype=v.dtype)
            idx = torch.as_tensor(sorted(experts), dtype=torch.long)
            src[idx] = v[idx.to(v.device)].cpu()
        out[k] = src.float().numpy() if src.dtype == torch.bfloat16 else src.numpy()
    return out


# The stack's output is a residual stream of magnitude O(1..10), where one bf16 step
# exceeds the layer's absolute bound: relative L2 1e-2 and max-abs 2^-6 of the largest
# value (two bf16 steps there).
TOL_STACK = dict(max_abs=None, max_abs_rel=2.0 ** -6, rel_l2=1e-2)


def check_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = "", tol=None):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got - ref
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-30))
    tol = tol or TOL[dtype]
    assert rel <= tol["rel_l2"], f"{what}: relative L2 {rel:.3e} > {tol['rel_l2']}"
    if tol.get("max_abs") is not None:
        mx = float(np.max(np.abs(diff))) if diff.size else 0.0
        assert mx <= tol["max_abs"], f"{what}: max abs {mx:.3e} > {tol['max_abs']}"
    if tol.get("max_abs_rel") is not None and diff.size:
        mx = float(np.max(np.abs(diff)))
        assert mx <= tol["max_abs_rel"] * float(np.max(np.abs(ref))) + 1e-30, f"{what}: max abs {mx:.3e}"
    return rel
