"""Pins for the oracle's plan (counting sort of (token, choice) pairs by expert):
brute-force stable sort, the plan invariants, capacity and bad-index reporting."""
import numpy as np
import pytest

import oracle


def _cfg(E, S, k):
    return oracle.Config(hidden=128, inter=128, num_experts=E, num_shared=S, top_k=k)


def _rand_ids(rng, T, E, k):
    return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,S,k,align", [(1, 4, 0, 2, 1), (37, 8, 0, 2, 1), (64, 16, 2, 4, 8),
                                           (200, 64, 2, 6, 128), (300, 128, 0, 8, 16)])
def test_plan_exact_mode_brute_force(T, E, S, k, align):
    rng = np.random.default_rng(T + E)
    ids = _rand_ids(rng, T, E, k)
    p = oracle.plan(_cfg(E, S, k), ids, capacity=0, align=align)
    assert p["status"] == oracle.OK
    kk = k + S
    ent_e = np.concatenate([ids, np.tile(np.arange(E, E + S, dtype=np.int32), (T, 1))], axis=1)
    flat = ent_e.reshape(-1)
    # counts
    ref_counts = np.bincount(flat, minlength=E + S)
    assert np.array_equal(p["counts"], ref_counts)
    assert p["counts"].sum() == T * k + T * S
    # offsets = exclusive scan of counts rounded up to `align`
    padded = (ref_counts + align - 1) // align * align
    assert np.array_equal(p["offsets"], np.concatenate([[0], np.cumsum(padded)]))
    # slots: stable sort by expert of the (t, j)-ordered entries
    order = np.argsort(flat, kind="stable")
    rank = np.empty_like(order)
    for e in range(E + S):
        idx = order[flat[order] == e]
        rank[idx] = np.arange(len(idx))
    ref_slot = p["offsets"][flat] + rank
    assert np.array_equal(p["slot_of"].reshape(-1), ref_slot)
    # token_of is the inverse map; everything else is padding (-1)
    tok = np.full(p["rows"], -1, np.int32)
    tok[ref_slot] = np.repeat(np.arange(T, dtype=np.int32), kk)
    assert np.array_equal(p["token_of"], tok)
    assert len(np.unique(ref_slot)) == T * kk


def test_plan_capacity_mode_and_overflow():
    rng = np.random.default_rng(5)
    T, E, S, k = 50, 8, 1, 2
    ids = _rand_ids(rng, T, E, k)
    p = oracle.plan(_cfg(E, S, k), ids, capacity=T)
    assert p["status"] == oracle.OK
    assert np.array_equal(p["offsets"], np.arange(E + S + 1) * T)
    exact = oracle.plan(_cfg(E, S, k), ids, capacity=0, align=1)
    assert np.array_equal(p["counts"], exact["counts"])
    # slot = e*C + the same within-expert rank as exact mode
    flat_e = np.concatenate([ids, np.full((T, 1), E, np.int32)], 1).reshape(-1)
    rank_exact = exact["slot_of"].reshape(-1) - exact["offsets"][flat_e]
    assert np.array_equal(p["slot_of"].reshape(-1), flat_e * T + rank_exact)
    # too small a capacity: entries past it get -1 and the call reports it
    C = 6
    q = oracle.plan(_cfg(E, S, k), ids, capacity=C)
    assert q["status"] == oracle.CAPACITY
    assert np.all(q["counts"] <= C)
    so = q["slot_of"].reshape(-1)
    assert np.all((so == -1) == (rank_exact >= C))
    assert np.array_equal(so[so >= 0], (flat_e * C + rank_exact)[so >= 0])


def test_plan_bad_index_reported_not_placed():
    ids = np.array([[0, 1], [2, 9], [-1, 3]], np.int32)
    p = oracle.plan(_cfg(4, 0, 2), ids, align=1)
    assert p["status"] == oracle.BAD_INDEX
    assert p["slot_of"][1, 1] == -1 and p["slot_of"][2, 0] == -1
    assert p["counts"].sum() == 4


def test_plan_expert_relabelling_permutes_counts():
    rng = np.random.default_rng(9)
    T, E, k = 80, 16, 4
    ids = _rand_ids(rng, T, E, k)
    perm = rng.permutation(E).astype(np.int32)
    a = oracle.plan(_cfg(E, 0, k), ids, align=1)
    b = oracle.plan(_cfg(E, 0, k), perm[ids], align=1)
    assert np.array_equal(b["counts"][perm], a["counts"])


def test_plan_empty_batch():
    p = oracle.plan(_cfg(8, 2, 2), np.zeros((0, 2), np.int32), align=128)
    assert p["status"] == oracle.OK and p["rows"] == 0
    assert np.array_equal(p["counts"], np.zeros(10, np.int32))
