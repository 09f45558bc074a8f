"""Pins for the oracle's gates: brute force selection, closed-form weights,
hand-worked examples, and reductions to the plain case."""
import itertools
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cfg(E, k, renorm=1, gate=oracle.GATE_SOFTMAX, n_group=1, topk_group=1, scale=1.0):
    return oracle.Config(hidden=128, inter=128, num_experts=E, num_shared=0, top_k=k, gate=gate,
                         renormalize=renorm, n_group=n_group, topk_group=topk_group,
                         routed_scale=scale, dtype=oracle.BF16)


@pytest.mark.parametrize("E,k,renorm", [(8, 2, 1), (16, 4, 0), (64, 6, 0), (128, 8, 1)])
def test_softmax_selection_brute_force_and_weights_closed_form(E, k, renorm):
    rng = np.random.default_rng(E * 10 + k)
    T = 40
    logits = rng.standard_normal((T, E)).astype(np.float32)
    # inject exact ties
    logits[::5, 3] = logits[::5, 1]
    ids, w = oracle.route(_cfg(E, k, renorm), logits)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        assert list(ids[t]) == order[:k]
        l64 = logits[t].astype(np.float64)
        p = np.exp(l64 - l64.max())
        if renorm:
            ref = p[order[:k]] / p[order[:k]].sum()
            assert abs(w[t].sum() - 1.0) < 1e-12
        else:
            ref = p[order[:k]] / p.sum()
        np.testing.assert_allclose(w[t], ref, rtol=1e-12, atol=0)


def test_renormalised_softmax_equals_softmax_over_chosen_logits():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((10, 32)).astype(np.float32) * 3
    ids, w = oracle.route(_cfg(32, 4, 1), logits)
    for t in range(10):
        sub = logits[t, ids[t]].astype(np.float64)
        ref = np.exp(sub) / np.exp(sub).sum()
        np.testing.assert_allclose(w[t], ref, rtol=1e-12)


def _brute_grouped(logits, bias, E, k, n_group, topk_group, renorm, scale):
    gsz = E // n_group
    s = np.array([oracle.spec_sigmoid(float(v)) for v in logits], np.float32)
    c = (s + (bias if bias is not None else np.zeros(E, np.float32))).astype(np.float32)
    gscore = []
    for g in range(n_group):
        vals = sorted(c[g * gsz:(g + 1) * gsz].tolist(), reverse=True)
        gscore.append(np.float32(vals[0]) + np.float32(vals[1]))
    # every subset of topk_group groups; the kept set is the best by (scores desc, id asc)
    best = None
    for sub in itertools.combinations(range(n_group), topk_group):
        key = sorted(((-float(gscore[g]), g) for g in sub))
        if best is None or key < best[0]:
            best = (key, sub)
    kept = set(best[1])
    cand = [e for e in range(E) if e // gsz in kept]
    order = sorted(cand, key=lambda e: (-float(c[e]), e))[:k]
    sd = np.array([1.0 / (1.0 + math.exp(-float(logits[e]))) for e in order])
    w = (sd / sd.sum() if renorm else sd) * scale
    return order, w


@pytest.mark.parametrize("E,k,G,TG,renorm,scale,use_bias", [
    (256, 8, 8, 4, 1, 1.0, False), (256, 8, 8, 4, 1, 2.5, True), (64, 6, 8, 3, 0, 1.0, True),
    (32, 4, 4, 2, 1, 1.0, False)])
def test_grouped_sigmoid_brute_force_over_group_subsets(E, k, G, TG, renorm, scale, use_bias):
    rng = np.random.default_rng(E + k + G)
    T = 12
    logits = rng.standard_normal((T, E)).astype(np.float32) * 2
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32) if use_bias else None
    cfg = _cfg(E, k, renorm, oracle.GATE_SIGMOID_GROUPED, G, TG, scale)
    ids, w = oracle.route(cfg, logits, bias)
    for t in range(T):
        order, wref = _brute_grouped(logits[t], bias, E, k, G, TG, renorm, scale)
        assert list(ids[t]) == order
        np.testing.assert_allclose(w[t], wref, rtol=1e-12)


def test_grouped_sigmoid_one_group_is_plain_sigmoid_topk():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((20, 16)).astype(np.float32)
    ids, w = oracle.route(_cfg(16, 3, 1, oracle.GATE_SIGMOID_GROUPED, 1, 1), logits)
    for t in range(20):
        order = sorted(range(16), key=lambda e: (-float(logits[t, e]), e))[:3]
        assert list(ids[t]) == order


def test_worked_examples():
    with open(os.path.join(GOLDEN, "route_worked.txt")) as f:
        cases = [ln for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(cases) == 2
    for ln in cases:
        head, lg, want_ids, want_w = [p.split() for p in ln.split("|")]
        name = head[0]
        logits = np.array([[float(v) for v in lg]], np.float32)
        if name == "softmax_tie":
            E, k = int(head[1]), int(head[2])
            cfg = _cfg(E, k, 1)
        else:
            E, k, G, TG = (int(v) for v in head[1:5])
            cfg = _cfg(E, k, 1, oracle.GATE_SIGMOID_GROUPED, G, TG)
        ids, w = oracle.route(cfg, logits)
        assert list(ids[0]) == [int(v) for v in want_ids], name
        np.testing.assert_allclose(w[0], [float(v) for v in want_w], rtol=1e-12)
