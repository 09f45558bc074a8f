"""The five MoE-layer workloads the library is measured and checked on.

Shapes only -- no arithmetic.  Each names the model family it is shaped like:

* ``tiny``            -- T=64, hidden 256, 8 experts, top-2 softmax (renormalised),
                         intermediate 512, fp32; two micro-batches of 32.
* ``qwen3_decode``    -- Qwen3-30B-A3B shaped decode layer: T=256 split 128/128,
                         hidden 2048, 128 experts, top-8 softmax renormalised,
                         intermediate 768, bf16.
* ``dsv2lite``        -- DeepSeek-V2-Lite shaped: hidden 2048, 64 routed + 2 shared
                         experts, top-6 softmax (not renormalised), intermediate
                         1408, bf16, T in {64, 512, 4096}, capacity or exact layout.
* ``qwen3_prefill``   -- Qwen3-30B-A3B shaped prefill chunk: one 8192-token prompt
                         split 4096/4096, hidden 2048, 128 experts top-8,
                         intermediate 768, fp8 e4m3 with 128-block scales.
* ``dsv3``            -- DeepSeek-V3 shaped: hidden 7168, 256 routed + 1 shared,
                         grouped sigmoid gate (8 groups, top-4 groups, top-8
                         experts), intermediate 2048, fp8 e4m3 with 128-block
                         scales, T in {128, 16384}.

The Dual-Batch Overlap pages measure prefill throughput on random data with
uniform-random routing simulation and dummy weights ("[Perf] Fix DBO overlap:
capture DeepEP event before yield", Test Result); these synthetic workloads stand in
for those serving benchmarks.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

F32, BF16, FP8 = "f32", "bf16", "fp8"


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    hidden: int
    inter: int
    num_experts: int
    num_shared: int
    top_k: int
    gate: str = "softmax"          # "softmax" | "sigmoid_grouped" | "sqrt_softplus"
    renormalize: bool = True
    n_group: int = 1
    topk_group: int = 1
    routed_scale: float = 1.0
    dtype: str = BF16
    routing: str = "uniform"       # "uniform" | "zipf"
    capacity: int = 0              # 0 = exact layout; >0 = rows per expert per micro-batch
    align: int = 128
    x_std: float = 1.0
    w_std: float = 0.02
    seed: int = 0

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def split(self) -> int:
        return (self.T + 1) // 2

    def describe(self) -> str:
        return (f"{self.name}: T={self.T} H={self.hidden} I={self.inter} E={self.num_experts}"
                f"+{self.num_shared} k={self.top_k} {self.gate} {self.dtype} {self.routing}"
                f"{' capacity' if self.capacity else ''}")


TINY = Workload("tiny", T=64, hidden=256, inter=512, num_experts=8, num_shared=0, top_k=2,
                dtype=F32, x_std=0.02, w_std=0.02, seed=0)
QWEN3_DECODE = Workload("qwen3_decode", T=256, hidden=2048, inter=768, num_experts=128,
                        num_shared=0, top_k=8, dtype=BF16, seed=1)
DSV2LITE = Workload("dsv2lite", T=512, hidden=2048, inter=1408, num_experts=64, num_shared=2,
                    top_k=6, renormalize=False, dtype=BF16, seed=2)
QWEN3_PREFILL = Workload("qwen3_prefill", T=8192, hidden=2048, inter=768, num_experts=128,
                         num_shared=0, top_k=8, dtype=FP8, seed=3)
DSV3 = Workload("dsv3", T=128, hidden=7168, inter=2048, num_experts=256, num_shared=1, top_k=8,
                gate="sigmoid_grouped", renormalize=True, n_group=8, topk_group=4,
                routed_scale=1.0, dtype=FP8, seed=4)

ALL = {w.name: w for w in (TINY, QWEN3_DECODE, DSV2LITE, QWEN3_PREFILL, DSV3)}
