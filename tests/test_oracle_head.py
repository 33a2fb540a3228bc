"""Pins for the oracle's LM head, softmax statistics and P.E (CPU only)."""

import math

import numpy as np
import scipy.special
import torch

from oracle import expected_embedding, head_confidence, vocab_softmax_stats


def test_handworked(golden):
    g = golden("head_handworked.json")
    r = head_confidence(np.array(g["hidden"], float), np.array(g["w_head"], float),
                        np.array(g["emb"], float))
    np.testing.assert_allclose(r["z"], g["logits"], atol=0)
    assert list(r["argmax"]) == g["argmax"]
    np.testing.assert_allclose(r["conf"], g["conf"], atol=g["abs_tol"])
    np.testing.assert_allclose(r["pe"], g["pe"], atol=g["abs_tol"])
    # closed form of the same example
    e2, e1 = math.exp(2.0), math.exp(1.0)
    tot = e2 + 1.0 + e1
    assert abs(r["conf"][0] - e2 / tot) < 1e-15
    assert abs(r["pe"][0, 0] - (e2 + e1) / tot) < 1e-15
    assert abs(r["pe"][0, 1] - (1.0 + e1) / tot) < 1e-15


def test_explicit_softmax_and_logsumexp():
    rng = np.random.default_rng(5)
    z = rng.standard_normal((4, 37)) * 3.0
    m, a, l, conf = vocab_softmax_stats(z)
    for r in range(4):
        ex = [math.exp(x) for x in z[r]]
        tot = math.fsum(ex)
        probs = [x / tot for x in ex]
        assert abs(math.fsum(probs) - 1.0) < 1e-14
        assert abs(conf[r] - max(probs)) < 1e-14
        assert a[r] == int(np.flatnonzero(z[r] == z[r].max())[0])
    np.testing.assert_allclose(np.log(conf), m - scipy.special.logsumexp(z, axis=1), rtol=1e-12)
    np.testing.assert_allclose(np.log(conf), (torch.from_numpy(z).max(1).values
                                              - torch.logsumexp(torch.from_numpy(z), 1)).numpy(),
                               rtol=1e-12)


def test_uniform_logits_and_ties():
    V = 64
    z = np.zeros((2, V))
    z[1, [5, 9, 40]] = 2.0
    m, a, l, conf = vocab_softmax_stats(z)
    assert abs(conf[0] - 1.0 / V) < 1e-15
    assert a[0] == 0 and a[1] == 5          # lowest index wins a tie
    r = head_confidence(np.ones((1, 3)), np.ones((V, 3)), np.arange(V * 2, dtype=float).reshape(V, 2))
    assert abs(r["conf"][0] - 1.0 / V) < 1e-15
    np.testing.assert_allclose(r["pe"][0], np.arange(V * 2, dtype=float).reshape(V, 2).mean(0), rtol=1e-13)


def test_one_hot_probability_gives_row():
    rng = np.random.default_rng(6)
    V, d = 50, 8
    emb = rng.standard_normal((V, d))
    z = rng.standard_normal((1, V))
    z[0, 17] = 100.0
    m, a, l, conf = vocab_softmax_stats(z)
    assert a[0] == 17 and conf[0] == 1.0
    np.testing.assert_allclose(expected_embedding(z, m, l, emb)[0], emb[17], rtol=1e-15, atol=1e-40)


def test_pe_brute_force():
    rng = np.random.default_rng(7)
    V, d = 30, 5
    z = rng.standard_normal((3, V))
    emb = rng.standard_normal((V, d))
    m, a, l, conf = vocab_softmax_stats(z)
    pe = expected_embedding(z, m, l, emb)
    for r in range(3):
        tot = math.fsum(math.exp(x) for x in z[r])
        for c in range(d):
            ref = math.fsum(math.exp(z[r, v]) / tot * emb[v, c] for v in range(V))
            assert abs(pe[r, c] - ref) < 1e-13
