"""Pins for the oracle's number formats and the specified exp / sigmoid.

Each is checked against something other than the oracle: library casts (torch's
bfloat16 and float8_e4m3fn conversions), the OCP FP8 specification's code points,
the defining inequality of the power-of-two scale, and double-precision exp.
"""
import math
import os
import struct

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32(x):
    return struct.unpack("f", struct.pack("f", x))[0]


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(0)
    vals = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * 10.0,
        rng.standard_normal(1000).astype(np.float32) * 1e-30,
        # exact ties between two bf16 neighbours (low 16 bits == 0x8000)
        np.array([struct.unpack("f", struct.pack("I", (b << 16) | 0x8000))[0]
                  for b in range(0x3f00, 0x3f40)], np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 65504.0, 3.0e38], np.float32),
    ])
    ref = torch.from_numpy(vals).to(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_round(float(v)) for v in vals], np.float32)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got), c
        else:
            assert got == float(ref[c]), (c, got, ref[c])


def test_e4m3_ocp_code_points():
    with open(os.path.join(GOLDEN, "e4m3_ocp_points.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 10
    for code_s, val_s in rows:
        code = int(code_s, 16)
        got = oracle.e4m3_decode(code)
        if val_s == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val_s), (code_s, got)
            assert oracle.e4m3_encode(float(val_s)) == code or float(val_s) == 0.0


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(1)
    vals = list(rng.uniform(-448, 448, 3000)) + list(rng.standard_normal(3000) * 0.01)
    # midpoints between neighbouring codes: ties must go to the even code
    dec = [oracle.e4m3_decode(c) for c in range(0x7e)]
    vals += [(dec[i] + dec[i + 1]) / 2 for i in range(len(dec) - 1)]
    vals += [-(dec[i] + dec[i + 1]) / 2 for i in range(len(dec) - 1)]
    v32 = np.array(vals, np.float32)
    ref = torch.from_numpy(v32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(v)) for v in v32], np.uint8)
    assert np.array_equal(got, ref)


def test_e4m3_encode_roundtrip_and_saturation():
    for c in range(256):
        if (c & 0x7f) == 0x7f:
            continue
        assert oracle.e4m3_encode(oracle.e4m3_decode(c)) == c
    assert oracle.e4m3_encode(1e9) == 0x7e
    assert oracle.e4m3_encode(-460.0) == 0xfe


def test_fp8_scale_exp_is_smallest_power_of_two():
    rng = np.random.default_rng(2)
    amaxes = np.concatenate([np.abs(rng.standard_normal(2000)) * 10.0 ** rng.integers(-8, 8, 2000),
                             [448.0, 449.0, 896.0, 1.0, 0.875, 224.0, 3.5]]).astype(np.float32)
    for a in amaxes:
        s = oracle.fp8_scale_exp(float(a))
        assert float(a) <= 448.0 * 2.0 ** s
        assert float(a) > 448.0 * 2.0 ** (s - 1)
    assert oracle.fp8_scale_exp(0.0) == 0


def test_quant_row_fp8_bounds_and_exactness():
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(512) * 3.0).astype(np.float32)
    q, s = oracle.quant_row_fp8(v)
    for g in range(4):
        grp = v[g * 128:(g + 1) * 128]
        sc = float(s[g])
        assert sc == 2.0 ** round(math.log2(sc))
        assert np.max(np.abs(grp)) / sc <= 448.0
        deq = np.array([oracle.e4m3_decode(int(c)) for c in q[g * 128:(g + 1) * 128]]) * sc
        # round-to-nearest: error at most half a code step (<= 2^-4 relative for normals)
        assert np.all(np.abs(deq - grp) <= np.maximum(np.abs(grp) * 2.0 ** -4, sc * 2.0 ** -10))
    ref = torch.from_numpy(v.reshape(4, 128) / s[:, None]).to(torch.float8_e4m3fn)
    assert np.array_equal(ref.view(torch.uint8).numpy().reshape(-1), q)


def test_spec_exp_within_two_ulp_of_exp():
    xs = np.concatenate([np.linspace(-87.0, 87.0, 20001), np.linspace(-1, 1, 2001)]).astype(np.float32)
    worst = 0.0
    for x in xs:
        got = oracle.spec_exp(float(x))
        ref = math.exp(float(x))
        ulp = math.ulp(_f32(ref)) if ref > 0 else 1e-45
        # float ulp at ref: spacing of binary32 numbers near ref
        m, e = math.frexp(ref)
        ulp32 = 2.0 ** (e - 24)
        worst = max(worst, abs(got - ref) / ulp32)
    assert worst < 2.0, worst


def test_spec_sigmoid_matches_double_and_saturates():
    xs = np.linspace(-30.0, 30.0, 6001).astype(np.float32)
    for x in xs:
        ref = 1.0 / (1.0 + math.exp(-float(x)))
        got = oracle.spec_sigmoid(float(x))
        assert abs(got - ref) <= 4 * 2.0 ** -24 * max(ref, 2.0 ** -30) + 1e-45, (x, got, ref)
    assert oracle.spec_sigmoid(1000.0) == 1.0
    assert 0.0 < oracle.spec_sigmoid(-1000.0) < 1e-30
    assert oracle.spec_sigmoid(0.0) == 0.5
