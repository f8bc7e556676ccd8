"""Pins of the oracle's router (A1) and layout (A2) steps (CPU only).

Router: brute force over every k-subset, a library sort, a hand-made tie,
and the closed form "softmax then renormalise over the chosen experts equals
a softmax over the chosen logits".  Layout: the invariants the pages fix
(every token's k choices placed exactly once, one expert's rows contiguous)
plus brute force by a library sort.
"""
import itertools

import numpy as np
import pytest

from oracle import oracle as O


def _brute_topk(scores, k):
    """The chosen set is the k-subset whose members all beat (or tie with a
    higher id than) every non-member; the order is by score, ties to lower id."""
    E = len(scores)
    best = None
    for sub in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in sub]
        ok = all(scores[a] > scores[b] or (scores[a] == scores[b] and a < b)
                 for a in sub for b in rest)
        if ok:
            assert best is None
            best = sub
    return sorted(best, key=lambda e: (-scores[e], e))


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
def test_router_brute_force_small(kind):
    rng = np.random.default_rng(5)
    T, d, E, k = 4, 16, 8, 2
    x = rng.standard_normal((T, d))
    Wr = rng.standard_normal((E, d)) * 0.3
    r = O.router(x, Wr, None, k, kind)
    logits = x @ Wr.T
    assert np.allclose(r["logits"], logits, rtol=1e-13, atol=1e-13)
    for t in range(T):
        assert list(r["ids"][t]) == _brute_topk(r["scores"][t], k)
        assert list(r["ids"][t]) == sorted(range(E), key=lambda e: (-r["scores"][t][e], e))[:k]


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
def test_router_brute_force_k3_e6(kind):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 8))
    Wr = rng.standard_normal((6, 8))
    b = rng.standard_normal(6)
    r = O.router(x, Wr, b, 3, kind)
    assert np.allclose(r["logits"], x @ Wr.T + b, rtol=1e-13, atol=1e-13)
    for t in range(16):
        assert list(r["ids"][t]) == _brute_topk(r["scores"][t], 3)


@pytest.mark.parametrize("kind", [O.SOFTMAX, O.SIGMOID])
def test_router_top1_is_argmax_with_unit_gate(kind):
    # k = 1: the expert of largest score (ties to the lower id), and the
    # renormalised gate of a single chosen expert is exactly 1; E = 1 routes
    # every token to expert 0.
    rng = np.random.default_rng(13)
    x = rng.standard_normal((40, 12))
    Wr = rng.standard_normal((5, 12))
    r = O.router(x, Wr, None, 1, kind)
    assert np.array_equal(r["ids"][:, 0], np.argmax(x @ Wr.T, axis=1))
    assert np.all(r["gates"] == 1.0)
    r1 = O.router(x, Wr[:1], None, 1, kind)
    assert np.all(r1["ids"] == 0) and np.all(r1["gates"] == 1.0)


def test_router_tie_goes_to_lower_id():
    # d = 1, x = 1: the logits are the router weights themselves.
    x = np.ones((1, 1))
    Wr = np.array([[0.5], [2.0], [1.0], [2.0], [1.0]])
    r = O.router(x, Wr, None, 3, O.SOFTMAX)
    assert list(r["ids"][0]) == [1, 3, 2]
    r = O.router(x, Wr, None, 3, O.SIGMOID)
    assert list(r["ids"][0]) == [1, 3, 2]


def test_softmax_renormalised_gates_closed_form():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((32, 24))
    Wr = rng.standard_normal((10, 24)) * 0.5
    r = O.router(x, Wr, None, 4, O.SOFTMAX)
    for t in range(32):
        l = r["logits"][t, r["ids"][t]]
        ref = np.exp(l - l.max()) / np.exp(l - l.max()).sum()
        assert np.allclose(r["gates"][t], ref, rtol=1e-14, atol=0)
        assert abs(r["gates"][t].sum() - 1.0) < 4e-16
        assert np.all(np.diff(r["gates"][t]) <= 0)


def test_sigmoid_gates_closed_form():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((32, 24))
    Wr = rng.standard_normal((10, 24)) * 0.5
    r = O.router(x, Wr, None, 4, O.SIGMOID)
    for t in range(32):
        l = r["logits"][t, r["ids"][t]]
        s = 1 / (1 + np.exp(-l))
        assert np.allclose(r["gates"][t], s / s.sum(), rtol=1e-14, atol=0)


def _check_layout(ids, E, lay):
    T, k = ids.shape
    S = T * k
    counts, off = lay["counts"], lay["offsets"]
    assert counts.sum() == S
    assert np.array_equal(counts, np.bincount(ids.reshape(-1), minlength=E))
    assert off[0] == 0 and off[-1] == S
    assert np.array_equal(np.diff(off), counts)
    seen = np.zeros(S, dtype=int)
    for t in range(T):
        for j in range(k):
            p = lay["slot_pos"][t, j]
            e = ids[t, j]
            assert off[e] <= p < off[e + 1]
            assert lay["row_tok"][p] == t and lay["row_j"][p] == j
            seen[p] += 1
    assert np.all(seen == 1)
    # brute force: rows in (expert, flat slot index) order
    order = sorted(range(S), key=lambda i: (ids.reshape(-1)[i], i))
    assert np.array_equal(lay["row_tok"], np.array(order) // k)
    assert np.array_equal(lay["row_j"], np.array(order) % k)


@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (7, 2, 8), (128, 2, 8), (300, 8, 256), (64, 4, 5)])
def test_layout_invariants_and_brute_force(T, k, E):
    rng = np.random.default_rng(T * 31 + k)
    ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    lay = O.layout(ids, E)
    _check_layout(ids, E, lay)


def test_layout_degenerate_one_expert_and_empty_experts():
    T, k, E = 50, 1, 16
    ids = np.full((T, k), 7, dtype=np.int32)
    lay = O.layout(ids, E)
    _check_layout(ids, E, lay)
    assert lay["counts"][7] == T and lay["counts"].sum() == T
    assert np.array_equal(lay["row_tok"], np.arange(T))
