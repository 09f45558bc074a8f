"""Host-side logic of bench.py, on the CPU: the default SM budget, the layer roofline's
weight accounting, the launch count it reports, and the DRAM-traffic lookup that must
ignore a profile once the FFN sources have changed."""
import math

import numpy as np
import pytest

import bench
from moe_expert_dispatch_route_gb300 import workloads as W


@pytest.mark.parametrize("wl,expected", [
    (W.QWEN3_DECODE, 16),                  # ubatches of 128 tokens
    (W.DSV2LITE.with_(T=512), 16),         # 256
    (W.DSV3.with_(T=128), 16),             # 64
    (W.TINY, 16),
    (W.DSV2LITE.with_(T=4096), 0),         # 2048: prefill, no split of the GPU
    (W.QWEN3_PREFILL, 0),                  # 4096
    (W.DSV3.with_(T=16384), 0),            # 8192
])
def test_default_comm_sms_by_ubatch_size(wl, expected):
    assert bench.default_comm_sms(wl) == expected


def test_expert_weight_bytes_include_fp8_block_scales():
    wl = W.DSV3
    H, I = wl.hidden, wl.inter
    scales = ((2 * I // 128) * (H // 128) + (H // 128) * (I // 128)) * 4
    assert bench.expert_weight_bytes(wl) == 3 * H * I + scales == 44_050_944
    assert bench.expert_weight_bytes(W.DSV2LITE) == 3 * 2048 * 1408 * 2


def test_layer_roofline_counts_weights_per_ubatch_and_once():
    wl = W.DSV2LITE.with_(T=8)  # split 4 / 4, 2 shared experts
    assert wl.split == 4
    k = wl.top_k
    ids = np.zeros((8, k), dtype=np.int32)
    ids[:4] = np.arange(k)          # ubatch 0 touches experts 0..5
    ids[4:] = np.arange(k) + 3      # ubatch 1 touches experts 3..8
    ms = 0.05
    r = bench.layer_roofline(wl, ids, ms, two=True)
    S = wl.num_shared
    assert r["experts_touched_per_ubatch"] == (k + S) + (k + S)
    assert r["experts_touched_once"] == 9 + S
    wb = bench.expert_weight_bytes(wl)
    assert r["bytes_weights_per_ubatch"] - r["bytes_weights_once"] == (2 * (k + S) - (9 + S)) * wb
    pk, _ = bench.peaks()
    tf = pk.get("bf16_tflops_sustained", pk["bf16_tflops"]) * 1e12
    bw = pk["hbm_gbs"] * 1e9
    t_min = max(r["flops"] / tf, r["bytes_weights_per_ubatch"] / bw)
    assert r["frac"] == pytest.approx(t_min / (ms / 1e3), abs=1e-4)  # reported to 4 decimals
    assert r["bound"] == ("tensor" if r["flops"] / tf > r["bytes_weights_per_ubatch"] / bw else "hbm")
    # unsplit: the two bounds coincide
    r1 = bench.layer_roofline(wl, ids, ms, two=False)
    assert r1["bytes_weights_per_ubatch"] == r1["bytes_weights_once"] == r["bytes_weights_once"]


def test_launches_per_step():
    # decode: ubatch 0 runs alone and takes the clustered head (1 launch), ubatch 1 the
    # fused plan + dispatch (route + 1); two FFN kernels and a combine each
    assert bench.launches_per_step(W.QWEN3_DECODE, True) == (1 + 3) + (2 + 3)
    # DeepSeek-V3 prefill: 8192-token ubatches are planned in chunks (count + assign)
    wl = W.DSV3.with_(T=16384)
    kk = wl.top_k + wl.num_shared
    assert math.ceil(wl.split / (4096 // kk)) > 1
    assert bench.launches_per_step(wl, True) == 2 * (1 + 3 + 3)
    # both fused options: route, count + assign, per-token quantisation, two FFN kernels
    assert bench.launches_per_step(wl, True, "both") == 2 * (1 + 2 + 1 + 2)
    assert bench.launches_per_step(wl, True, "gather") == 2 * (1 + 2 + 1 + 3)


def test_code_only_ignores_comments_and_whitespace():
    src = "int a; /* block\n comment */ int  b;  // line comment\n\tint c;"
    assert bench.code_only(src) == "int a; int b; int c;"


def test_profiled_traffic_needs_the_current_ffn_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "moe_expert_dispatch_route_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "ffn_x.cu").write_text("__global__ void k() {} // v1\n")
    (csrc / "route.cu").write_text("not part of the hash\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    wl = W.DSV3.with_(T=16384)
    assert bench.profiled_traffic("ffn", wl) is None  # no profile
    h = bench.ffn_source_hash()
    prof = tmp_path / "profiles" / f"ffn_{wl.name}_T{wl.T}.txt"
    prof.write_text(f"# comment: ignored\nworkload: dsv3\ndram_bytes_per_launch: 12345\nffn_source_hash: {h}\n")
    assert bench.profiled_traffic("ffn", wl) == 12345.0
    # a comment-only edit, or an edit outside the FFN sources, keeps the hash; a code edit does not
    (csrc / "ffn_x.cu").write_text("__global__ void k() {} // v2, comment only\n")
    (csrc / "route.cu").write_text("changed, still not hashed\n")
    assert bench.ffn_source_hash() == h and bench.profiled_traffic("ffn", wl) == 12345.0
    (csrc / "ffn_x.cu").write_text("__global__ void k() { int i = 0; }\n")
    assert bench.profiled_traffic("ffn", wl) is None
