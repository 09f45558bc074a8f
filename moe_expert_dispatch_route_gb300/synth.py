"""Seeded synthetic inputs for the MoE layer (shared by the tests, the smoke check
and the benchmark).  This module draws random numbers and casts them to storage
types; it holds none of the layer's arithmetic.

Recipe (per workload, seed = the workload's seed):

* router logits ``[T, E]`` fp32:
  - ``uniform``: iid N(0, 1) -- the uniform-random routing simulation the Dual-Batch
    Overlap benchmarks use;
  - ``zipf``: ``ln p_e + Gumbel(0, 1)`` with ``p_e ~ (pi(e) + 1)^-1.2`` over a seeded
    permutation ``pi`` of the experts (Gumbel-top-k == sampling k experts without
    replacement with probability ~ p, so expert load follows Zipf(1.2)).
* hidden states ``x [T, H]``: N(0, x_std) rounded to bf16 (fp32 for fp32 layers).
* weights ``W13 [E+S, 2I, H]`` (gate rows, then up rows) and ``W2 [E+S, H, I]``:
  - fp32 / bf16 layers: N(0, w_std) cast to the storage type;
  - fp8 layers: e4m3 codes of ``clamp(N(0,1) * 64, +-448)`` with one power-of-two scale
    per 128x128 block, ``2^(-12 + u)``, u uniform in {-1, 0, 1} -- effective weights of
    standard deviation ~0.016 with block-to-block scale variation.
Large weight sets are drawn on the device they will live on, expert by expert.
"""
from __future__ import annotations

import torch

QG = 128


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def logits(T: int, E: int, routing: str = "uniform", seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(device, seed * 1000 + 1)
    if routing == "uniform":
        return torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if routing == "zipf":
        perm = torch.randperm(E, generator=g, device=device)
        p = (perm.to(torch.float64) + 1.0) ** -1.2
        p = p / p.sum()
        u = torch.rand(T, E, generator=g, device=device, dtype=torch.float64).clamp_(1e-12, 1 - 1e-12)
        gumbel = -torch.log(-torch.log(u))
        return (torch.log(p)[None, :] + gumbel).to(torch.float32)
    raise ValueError(f"unknown routing {routing!r}")


def hidden(T: int, H: int, dtype: str, std: float = 1.0, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(device, seed * 1000 + 2)
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32) * std
    return x if dtype == "f32" else x.to(torch.bfloat16)


def bias(E: int, std: float, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(device, seed * 1000 + 3)
    return torch.randn(E, generator=g, device=device, dtype=torch.float32) * std


def _fp8_block(rows: int, cols: int, g, device):
    codes = (torch.randn(rows, cols, generator=g, device=device, dtype=torch.float32) * 64.0)
    codes = codes.clamp_(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    u = torch.randint(-1, 2, (rows // QG, cols // QG), generator=g, device=device)
    scales = torch.pow(2.0, (u - 12).to(torch.float32))
    return codes, scales


def weights(NE: int, H: int, I: int, dtype: str, std: float = 0.02, seed: int = 0,
            device="cpu") -> dict:
    """Returns {"w13", "w2"} (fp32/bf16 tensors) or {"w13_q", "w13_s", "w2_q", "w2_s"} (fp8)."""
    g = _gen(device, seed * 1000 + 4)
    if dtype == "fp8":
        w13_q = torch.empty(NE, 2 * I, H, dtype=torch.uint8, device=device)
        w13_s = torch.empty(NE, 2 * I // QG, H // QG, dtype=torch.float32, device=device)
        w2_q = torch.empty(NE, H, I, dtype=torch.uint8, device=device)
        w2_s = torch.empty(NE, H // QG, I // QG, dtype=torch.float32, device=device)
        for e in range(NE):
            w13_q[e], w13_s[e] = _fp8_block(2 * I, H, g, device)
            w2_q[e], w2_s[e] = _fp8_block(H, I, g, device)
        return dict(w13_q=w13_q, w13_s=w13_s, w2_q=w2_q, w2_s=w2_s)
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    w13 = torch.empty(NE, 2 * I, H, dtype=tdt, device=device)
    w2 = torch.empty(NE, H, I, dtype=tdt, device=device)
    for e in range(NE):
        w13[e] = (torch.randn(2 * I, H, generator=g, device=device) * std).to(tdt)
        w2[e] = (torch.randn(H, I, generator=g, device=device) * std).to(tdt)
    return dict(w13=w13, w2=w2)


def workload_inputs(wl, device="cpu", T: int | None = None, with_weights: bool = True) -> dict:
    """All inputs of one workload: logits, x, weights (and bias = None)."""
    T = wl.T if T is None else T
    NE = wl.num_experts + wl.num_shared
    out = dict(
        logits=logits(T, wl.num_experts, wl.routing, wl.seed, device),
        x=hidden(T, wl.hidden, wl.dtype, wl.x_std, wl.seed, device),
        bias=None,
    )
    if with_weights:
        out.update(weights(NE, wl.hidden, wl.inter, wl.dtype, wl.w_std, wl.seed, device))
    return out


def to_numpy_f32(t: torch.Tensor):
    """Host float32 copy of a tensor (exact for bf16 / fp32 values)."""
    return t.detach().to("cpu", torch.float32).numpy()


def to_numpy(t: torch.Tensor):
    return t.detach().cpu().numpy()
