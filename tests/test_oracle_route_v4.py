"""Pins for the oracle's DeepSeek-V4-shaped gate (reading: the group-limited gate of
the DeepSeek-V3 shape with the score sqrt(softplus(l)) in place of sigma) and its hash
routing (the experts of a token are a fixed table's row for its token id).

The specified log1p and sqrt-softplus are pinned against double-precision library
routines and monotonicity; the selection against brute force over group subsets and,
with one group and no bias, against a plain sort of the logits (the score is
increasing); the weights against their closed form; hash routing against numpy
indexing."""
import itertools
import math

import numpy as np
import pytest

import oracle


def _cfg(E, k, renorm=1, n_group=1, topk_group=1, scale=1.0):
    return oracle.Config(hidden=128, inter=128, num_experts=E, num_shared=0, top_k=k, gate=oracle.GATE_SQRT_SOFTPLUS,
                         renormalize=renorm, n_group=n_group, topk_group=topk_group, routed_scale=scale,
                         dtype=oracle.BF16)


def _ulps(got: float, ref: float) -> float:
    return abs(got - ref) / np.spacing(np.float32(abs(ref)))


def _sqrt_softplus_d(x: float) -> float:
    return math.sqrt(x + math.log1p(math.exp(-x)) if x > 30 else math.log1p(math.exp(x)))


def test_spec_log1p_within_3_ulp_on_unit_interval():
    # rounding budget of the stated operations: z = y / (2 + y) (two roundings), the
    # Horner sum (< 1 ulp on a value near 1), the final product: below 3 ulp
    ys = np.concatenate([np.linspace(0.0, 1.0, 20001, dtype=np.float32),
                         np.float32(2.0) ** -np.arange(1, 60, dtype=np.float32)])
    worst = 0.0
    for y in ys:
        got = oracle.spec_log1p(float(y))
        ref = math.log1p(float(y))
        if ref == 0.0:
            assert got == 0.0
            continue
        worst = max(worst, _ulps(got, ref))
    assert worst <= 3.0, worst


def test_spec_sqrt_softplus_within_3_ulp_monotone_and_saturating():
    xs = np.linspace(-80.0, 80.0, 40001, dtype=np.float32)
    prev = -1.0
    worst = 0.0
    for x in xs:
        got = oracle.spec_sqrt_softplus(float(x))
        worst = max(worst, _ulps(got, _sqrt_softplus_d(float(x))))
        assert got >= prev
        prev = got
    assert worst <= 3.0, worst
    assert oracle.spec_sqrt_softplus(200.0) == oracle.spec_sqrt_softplus(80.0)
    assert oracle.spec_sqrt_softplus(-200.0) == oracle.spec_sqrt_softplus(-80.0)
    assert oracle.spec_sqrt_softplus(0.0) == np.float32(math.sqrt(math.log(2.0)))


def _brute(logits, bias, E, k, G, TG, renorm, scale):
    gsz = E // G
    s = np.array([oracle.spec_sqrt_softplus(float(v)) for v in logits], np.float32)
    c = (s + (bias if bias is not None else np.zeros(E, np.float32))).astype(np.float32)
    gscore = []
    for g in range(G):
        vals = sorted(c[g * gsz:(g + 1) * gsz].tolist(), reverse=True)
        gscore.append(np.float32(vals[0]) + np.float32(vals[1]) if gsz >= 2 else np.float32(vals[0]))
    best = None
    for sub in itertools.combinations(range(G), TG):
        key = sorted((-float(gscore[g]), g) for g in sub)
        if best is None or key < best[0]:
            best = (key, sub)
    cand = [e for e in range(E) if e // gsz in set(best[1])]
    order = sorted(cand, key=lambda e: (-float(c[e]), e))[:k]
    sd = np.array([_sqrt_softplus_d(float(logits[e])) for e in order])
    return order, (sd / sd.sum() if renorm else sd) * scale


@pytest.mark.parametrize("E,k,G,TG,renorm,scale,use_bias", [
    (256, 8, 8, 4, 1, 1.0, False), (256, 8, 8, 4, 1, 2.5, True), (64, 6, 4, 2, 0, 1.0, True),
    (128, 6, 1, 1, 1, 1.0, True)])
def test_sqrt_softplus_gate_brute_force_over_group_subsets(E, k, G, TG, renorm, scale, use_bias):
    rng = np.random.default_rng(E + 3 * k + G)
    T = 12
    logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32) if use_bias else None
    ids, w = oracle.route(_cfg(E, k, renorm, G, TG, scale), logits, bias)
    for t in range(T):
        order, wref = _brute(logits[t], bias, E, k, G, TG, renorm, scale)
        assert list(ids[t]) == order
        np.testing.assert_allclose(w[t], wref, rtol=1e-12)


def test_one_group_without_bias_is_the_top_k_of_the_logits():
    rng = np.random.default_rng(21)
    E, k, T = 64, 6, 40
    logits = (rng.standard_normal((T, E)) * 3).astype(np.float32)
    ids, w = oracle.route(_cfg(E, k, 1), logits)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        assert list(ids[t]) == order
        sd = np.array([_sqrt_softplus_d(float(logits[t, e])) for e in order])
        np.testing.assert_allclose(w[t], sd / sd.sum(), rtol=1e-12)
        assert abs(w[t].sum() - 1.0) < 1e-12


def test_hash_routing_is_a_table_lookup_with_gate_weights():
    rng = np.random.default_rng(5)
    E, k, T, V = 32, 4, 50, 100
    logits = rng.standard_normal((T, E)).astype(np.float32)
    table = np.stack([rng.permutation(E)[:k] for _ in range(V)]).astype(np.int32)
    table[7, 2] = E + 3  # an entry outside [0, E): passed on, weight 0
    tids = rng.integers(0, V, T).astype(np.int32)
    tids[4] = 7
    tids[9] = -1  # outside [0, vocab)
    tids[10] = V
    for renorm, scale in ((1, 1.0), (0, 2.0)):
        ids, w = oracle.route_hash(_cfg(E, k, renorm, scale=scale), logits, tids, table)
        for t in range(T):
            if not 0 <= tids[t] < V:
                assert list(ids[t]) == [-1] * k and not w[t].any()
                continue
            assert list(ids[t]) == table[tids[t]].tolist()
            sd = np.array([_sqrt_softplus_d(float(logits[t, e])) if 0 <= e < E else 0.0 for e in ids[t]])
            ref = (sd / sd.sum() if renorm else sd) * scale
            np.testing.assert_allclose(w[t], ref, rtol=1e-12)
        assert w[4, 2] == 0.0 and ids[4, 2] == E + 3
