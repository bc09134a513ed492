"""Pins of the oracle's router and schedule against things other than itself:
closed forms, special cases that fix the tie-break, subset enumeration and a
brute-force nested-loop schedule."""
import itertools
import math

import numpy as np
import pytest

from oracle import moe_oracle as O


def test_router_zero_weights_pins_tie_break():
    # all logits equal -> all p equal -> the k lowest expert indices, w = 1/k
    T, H, E, k = 5, 8, 6, 3
    x = np.random.default_rng(0).standard_normal((T, H))
    r = O.router(x, np.zeros((H, E)), None, k)
    assert (r["ids"] == np.arange(k)[None, :]).all()
    np.testing.assert_allclose(r["w"], 1.0 / k, rtol=0, atol=1e-15)
    np.testing.assert_allclose(r["probs"], 1.0 / E, rtol=0, atol=1e-15)


def test_router_bias_only_closed_form():
    # zero weights + bias: every token picks the k largest biases, ties to lower index
    E, k = 6, 3
    bias = np.array([0.0, math.log(3.0), 0.0, math.log(3.0), -1.0, 0.0])
    x = np.ones((4, 2))
    r = O.router(x, np.zeros((2, E)), bias, k)
    # p ∝ (1, 3, 1, 3, e^-1, 1); top: experts 1 and 3 (p=3/Z), then expert 0 (lowest of the tied 1s)
    assert (r["ids"] == np.array([1, 3, 0])[None, :]).all()
    np.testing.assert_allclose(r["w"], np.array([[3 / 7, 3 / 7, 1 / 7]] * 4), rtol=1e-14)
    Z = 1 + 3 + 1 + 3 + math.exp(-1) + 1
    np.testing.assert_allclose(r["probs"][0], np.array([1, 3, 1, 3, math.exp(-1), 1]) / Z, rtol=1e-14)


def test_router_two_expert_closed_form():
    # logits (0, ln 3) -> p = (1/4, 3/4)
    x = np.array([[1.0]])
    Wr = np.array([[0.0, math.log(3.0)]])
    r = O.router(x, Wr, None, 1)
    np.testing.assert_allclose(r["probs"], [[0.25, 0.75]], rtol=1e-15)
    assert r["ids"].tolist() == [[1]]
    assert r["w"].tolist() == [[1.0]]


def test_router_k_equals_E_weights_are_probs():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 16)); Wr = rng.standard_normal((16, 5))
    r = O.router(x, Wr, None, 5)
    for t in range(7):
        np.testing.assert_allclose(r["w"][t], r["probs"][t][r["ids"][t]], rtol=1e-14)
        assert sorted(r["ids"][t].tolist()) == list(range(5))
        assert np.all(np.diff(r["w"][t]) <= 0)       # descending order


def test_router_topk_is_max_subset_by_enumeration():
    rng = np.random.default_rng(2)
    T, H, E, k = 20, 6, 6, 3
    x = rng.standard_normal((T, H)); Wr = rng.standard_normal((H, E))
    r = O.router(x, Wr, None, k)
    logits = x @ Wr
    for t in range(T):
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(logits[t, list(c)]))
        assert set(r["ids"][t].tolist()) == set(best)
        # slot order: descending logit
        assert all(logits[t, r["ids"][t][i]] >= logits[t, r["ids"][t][i + 1]] for i in range(k - 1))
        np.testing.assert_allclose(r["w"][t].sum(), 1.0, rtol=1e-14)


def test_router_shift_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((6, 4)); Wr = rng.standard_normal((4, 5))
    a = O.router(x, Wr, None, 2)
    b = O.router(x, Wr, np.full(5, 123.0), 2)
    np.testing.assert_allclose(a["probs"], b["probs"], rtol=1e-12)
    assert (a["ids"] == b["ids"]).all()


def brute_schedule(ids, E, Mb):
    T, k = ids.shape
    nM = 1 if Mb <= 0 else -(-T // Mb)
    MbE = T if Mb <= 0 else Mb
    order, counts, offsets = [], np.zeros((nM, E), int), np.zeros((nM, E + 1), int)
    for m in range(nM):
        for e in range(E):
            offsets[m, e] = len(order)
            for t in range(m * MbE, min(T, (m + 1) * MbE)):
                for j in range(k):
                    if ids[t, j] == e:
                        order.append(t * k + j)
                        counts[m, e] += 1
        offsets[m, E] = len(order)
    return np.array(order), counts, offsets


def random_ids(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k,Mb", [(1, 1, 1, 0), (37, 5, 2, 0), (64, 8, 3, 10), (50, 4, 4, 7), (33, 16, 1, 0), (30, 6, 2, 100)])
def test_schedule_matches_bruteforce(T, E, k, Mb):
    rng = np.random.default_rng(T * 100 + E)
    ids = random_ids(rng, T, E, k)
    s = O.schedule(ids, E, Mb)
    order, counts, offsets = brute_schedule(ids, E, Mb)
    assert (s["sorted_to_slot"] == order).all()
    assert (s["counts"] == counts).all()
    assert (s["offsets"] == offsets).all()
    R = T * k
    assert s["counts"].sum() == R                                   # sum counts = T*k
    assert (s["slot_to_sorted"][s["sorted_to_slot"]] == np.arange(R)).all()   # round trip
    assert (s["sorted_to_slot"][s["slot_to_sorted"]] == np.arange(R)).all()
    # stability: tokens ascending inside every (m, e) run
    for m in range(s["offsets"].shape[0]):
        for e in range(E):
            run = s["sorted_to_slot"][s["offsets"][m, e]:s["offsets"][m, e + 1]] // k
            assert (np.diff(run) > 0).all()


def test_schedule_empty_experts_and_single_expert():
    ids = np.zeros((9, 1), np.int32)
    s = O.schedule(ids, 4, 0)
    assert s["counts"].tolist() == [[9, 0, 0, 0]]
    assert s["offsets"].tolist() == [[0, 9, 9, 9, 9]]
    assert (s["sorted_to_slot"] == np.arange(9)).all()
