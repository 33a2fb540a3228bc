"""Pins of the MoE FFN oracle against closed forms, special cases that reduce
to the dense FFN, and brute force (no GPU)."""

import numpy as np
import pytest

from oracle import model as om
from oracle import moe


def _weights(rng, E, F, d):
    return (rng.standard_normal((E, 2 * F, d)) * 0.1, rng.standard_normal((E, d, F)) * 0.1,
            rng.standard_normal((E, d)))


def test_route_hand_worked():
    # logits (2, 0, 1, 2): probabilities e^z / sum; top-2 = experts 0 and 3
    # (tie at 2, lower index ranked first), weights 1/2 each
    h = np.array([[1.0]])
    wr = np.array([[2.0], [0.0], [1.0], [2.0]])
    ids, w, z = moe.route(h, wr, 2)
    assert ids.tolist() == [[0, 3]] and np.allclose(w, [[0.5, 0.5]])
    # top-3 adds expert 2 with weight e^1 / (2 e^2 + e^1)
    ids, w, _ = moe.route(h, wr, 3)
    assert ids.tolist() == [[0, 3, 2]]
    s = 2 * np.e ** 2 + np.e
    assert np.allclose(w, [[np.e ** 2 / s, np.e ** 2 / s, np.e / s]], rtol=1e-14)


def test_single_expert_is_the_dense_ffn():
    rng = np.random.default_rng(1)
    d, F, n = 16, 24, 7
    w13, w2, wr = _weights(rng, 1, F, d)
    h = rng.standard_normal((n, d))
    y, ids, w = moe.moe_ffn(h, wr, w13, w2, 1)
    assert (ids == 0).all() and np.allclose(w, 1.0)
    ref = (om.silu(h @ w13[0, :F].T) * (h @ w13[0, F:].T)) @ w2[0].T
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_all_experts_chosen_weights_are_the_softmax():
    rng = np.random.default_rng(2)
    d, F, n, E = 8, 8, 5, 6
    w13, w2, wr = _weights(rng, E, F, d)
    h = rng.standard_normal((n, d))
    ids, w, z = moe.route(h, wr, E)
    p = np.exp(z) / np.exp(z).sum(axis=1, keepdims=True)
    np.testing.assert_allclose(np.take_along_axis(p, ids, axis=1), w, rtol=1e-13)
    assert (np.diff(np.take_along_axis(p, ids, axis=1), axis=1) <= 0).all()   # highest first


def test_zero_router_picks_the_lowest_indices_evenly():
    rng = np.random.default_rng(3)
    d, F, n, E, k = 8, 8, 4, 10, 3
    w13, w2, _ = _weights(rng, E, F, d)
    h = rng.standard_normal((n, d))
    y, ids, w = moe.moe_ffn(h, np.zeros((E, d)), w13, w2, k)
    assert (ids == np.arange(k)).all() and np.allclose(w, 1.0 / k)
    ref = sum(moe.expert(h, w13[e], w2[e], F) for e in range(k)) / k
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


def test_matches_brute_force_loops():
    rng = np.random.default_rng(4)
    d, F, n, E, k = 6, 5, 9, 7, 3
    w13, w2, wr = _weights(rng, E, F, d)
    h = rng.standard_normal((n, d))
    y, ids, w = moe.moe_ffn(h, wr, w13, w2, k)
    for t in range(n):
        z = [sum(h[t, c] * wr[e, c] for c in range(d)) for e in range(E)]
        m = max(z)
        p = [np.exp(v - m) for v in z]
        p = [v / sum(p) for v in p]
        chosen = sorted(range(E), key=lambda e: (-p[e], e))[:k]
        assert ids[t].tolist() == chosen
        tot = sum(p[e] for e in chosen)
        acc = np.zeros(d)
        for e in chosen:
            for c in range(d):
                s = 0.0
                for f in range(F):
                    g = sum(h[t, i] * w13[e, f, i] for i in range(d))
                    u = sum(h[t, i] * w13[e, F + f, i] for i in range(d))
                    s += g / (1 + np.exp(-g)) * u * w2[e, c, f]
                acc[c] += p[e] / tot * s
        np.testing.assert_allclose(y[t], acc, rtol=1e-11, atol=1e-12)


def test_tokens_are_independent_and_given_routing_is_used():
    rng = np.random.default_rng(5)
    d, F, n, E, k = 8, 8, 6, 5, 2
    w13, w2, wr = _weights(rng, E, F, d)
    h = rng.standard_normal((n, d))
    y, ids, w = moe.moe_ffn(h, wr, w13, w2, k)
    perm = rng.permutation(n)
    y2, _, _ = moe.moe_ffn(h[perm], wr, w13, w2, k)
    np.testing.assert_allclose(y2, y[perm], rtol=1e-13)
    # forcing other experts changes the result; forcing the router's own does not
    y3, _, _ = moe.moe_ffn(h, wr, w13, w2, k, ids=ids, weights=w)
    np.testing.assert_array_equal(y3, y)
    y4, _, _ = moe.moe_ffn(h, wr, w13, w2, k, ids=(ids + 1) % E, weights=w)
    assert np.abs(y4 - y).max() > 1e-3


@pytest.mark.parametrize("k", [1, 4])
def test_topk_gap(k):
    z = np.array([[3.0, 1.0, 2.0, 0.5, 2.5]])
    gap, sc = moe.topk_gap(z, k)
    expect = {1: 3.0 - 2.5, 4: 1.0 - 0.5}[k]
    assert gap[0] == pytest.approx(expect) and sc[0] == 3.0
