"""Pins for the oracle's parallel-decode commit (CPU only).

Hand-worked 3-position cases, the invariants the dInfer article's decoding
strategies imply, special cases that reduce to plain threshold decoding, and
the logarithmic fill of hierarchical decoding.
"""

import math

import numpy as np
import pytest

from oracle import commit, masked_spans

BASE = dict(tau=0.9, lam=0.7, kappa=1.5, hierarchical=1, hier_levels=1,
            smoothing=0, alpha=1.0, mask_id=9)


def _run(prev, credit, argmax, p, mode, extra=None, mask=None, emb=None, pe=None, **prm):
    n = len(p)
    params = dict(BASE, **prm)
    if mode == "off":
        params["hierarchical"] = 0
    elif mode == "levels1":
        params.update(hierarchical=1, hier_levels=1)
    elif mode == "levels2":
        params.update(hierarchical=1, hier_levels=2)
    elif mode == "inf":
        params.update(hierarchical=1, hier_levels=10 ** 6)
    mask = np.ones((1, n), np.uint8) if mask is None else np.asarray(mask, np.uint8)[None]
    rows = [j for j in range(n) if mask[0, j]]
    emb = np.eye(12, 4) if emb is None else emb
    return commit(np.asarray(argmax)[rows], np.asarray(p, np.float32)[rows],
                  None if pe is None else pe[rows],
                  np.zeros(len(rows), np.int32), np.asarray(rows, np.int32),
                  mask, np.full((1, n), params["mask_id"], np.int32),
                  np.asarray(credit, np.float32)[None], np.asarray(prev, np.int32)[None],
                  emb, params)


def test_handworked(golden):
    g = golden("commit_handworked.json")
    for case in g["cases"]:
        for mode, want in case["selected"].items():
            r = _run(case["prev"], case["credit"], case["argmax"], case["p"], mode, **g["params"])
            assert sorted(np.flatnonzero(r["selected"][0])) == want, (case["name"], mode)
            assert sorted(np.flatnonzero(r["cand"][0])) == case["candidates"], case["name"]
            # credit after the update is observable on the positions left masked
            for j in range(3):
                if not r["selected"][0, j]:
                    assert abs(float(r["credit"][0, j]) - case["credit_after"][j]) < g["abs_tol"]
                else:
                    assert r["credit"][0, j] == 0 and r["prev"][0, j] == -1
            assert r["n_commit"][0] == len(want)


def _random_state(rng, n, V=12):
    mask = (rng.random(n) < 0.7).astype(np.uint8)
    if not mask.any():
        mask[rng.integers(n)] = 1
    prev = np.where(rng.random(n) < 0.5, rng.integers(0, V, n), -1)
    credit = rng.uniform(0, 1.5, n).astype(np.float32)
    argmax = rng.integers(0, V, n)
    argmax = np.where(rng.random(n) < 0.5, np.maximum(prev, 0), argmax)
    p = rng.uniform(0.3, 1.0, n).astype(np.float32)
    return mask, prev, credit, argmax, p


@pytest.mark.parametrize("mode", ["off", "levels1", "levels2", "inf"])
def test_invariants_random(mode):
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(1, 20))
        mask, prev, credit, argmax, p = _random_state(rng, n)
        r = _run(prev, credit, argmax, p, mode, mask=mask)
        sel, cand = r["selected"][0], r["cand"][0]
        # committed positions were masked, are now unmasked, and are the only changes
        assert not (sel & ~mask.astype(bool)).any()
        assert np.array_equal(r["mask"][0], mask & ~sel)
        assert r["n_commit"][0] == sel.sum() >= 1
        if not r["fallback"][0]:
            assert not (sel & ~cand).any()        # S subset of C
        else:
            assert sel.sum() == 1 and not cand.any()
        for (l, rr) in masked_spans(mask.astype(bool)):
            cs = [s for s in range(l, rr) if cand[s]]
            if not cs or r["fallback"][0]:
                continue
            c = l + (rr - l - 1) // 2
            got = [s for s in range(l, rr) if sel[s]]
            if mode == "levels1":
                assert len(got) == 1               # exactly one per span
                dist = np.array([abs(s - c) for s in cs])
                near = [s for s, dd in zip(cs, dist) if dd == dist.min()]
                best = max(float(p[s]) for s in near)
                assert got[0] == min(s for s in near if float(p[s]) == best)
            if c in cs:
                assert sel[c]                       # the centre first
        if mode in ("off", "inf") and not r["fallback"][0]:
            assert np.array_equal(sel, cand)        # unlimited levels = threshold set


def test_kappa_infinite_is_pure_threshold_and_lambda_zero_is_p():
    rng = np.random.default_rng(12)
    for _ in range(100):
        n = int(rng.integers(2, 16))
        mask, prev, credit, argmax, p = _random_state(rng, n)
        r = _run(prev, credit, argmax, p, "off", mask=mask, kappa=math.inf)
        want = mask.astype(bool) & (p >= np.float32(0.9))
        if want.any():
            assert np.array_equal(r["selected"][0], want)
        r = _run(prev, credit, argmax, p, "off", mask=mask, lam=0.0)
        kept = mask.astype(bool) & ~r["selected"][0]
        np.testing.assert_array_equal(r["credit"][0][kept], p[kept])


def test_credit_reaches_kappa_over_steps():
    # position 0: p = 0.5, argmax unchanged, so credit_n = 0.5 (1 - 0.7^n) / 0.3,
    # which first reaches kappa = 1.5 at n = 7 (1.4706 at n = 6, 1.5294 at n = 7).
    # positions 1..7: p = 0.6 with an argmax that changes every step, so they
    # never qualify and absorb the one-per-step fallback commits meanwhile.
    n = 8
    mask = np.ones(n, np.uint8)
    prev, credit = [-1] * n, [0.0] * n
    for step in range(1, 8):
        argmax = [3] + [step] * 7
        p = [0.5] + [0.6] * 7
        r = _run(prev, credit, argmax, p, "off", mask=mask)
        if step < 7:
            assert r["fallback"][0] and r["selected"][0, step] and not r["selected"][0, 0]
        else:
            assert not r["fallback"][0] and r["selected"][0, 0]
            assert list(np.flatnonzero(r["selected"][0])) == [0]
        mask = r["mask"][0].copy()
        prev, credit = list(r["prev"][0]), list(r["credit"][0])


@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 31, 32, 64])
def test_hierarchical_fills_in_log_steps(n):
    mask = np.ones(n, np.uint8)
    prev, credit = [-1] * n, [0.0] * n
    steps, order = 0, []
    while mask.any():
        steps += 1
        r = _run(prev, credit, [1] * n, [0.99] * n, "levels1", mask=mask)
        order.append(sorted(np.flatnonzero(r["selected"][0])))
        mask = r["mask"][0].copy()
        prev, credit = list(r["prev"][0]), list(r["credit"][0])
    assert steps == math.ceil(math.log2(n + 1))
    assert order[0] == [(n - 1) // 2]


def test_next_embedding_rows():
    emb = np.arange(12 * 4, dtype=float).reshape(12, 4)
    pe = np.full((3, 4), 0.5)
    r = _run([-1, -1, -1], [0, 0, 0], [3, 4, 5], [0.95, 0.2, 0.3], "off",
             emb=emb, pe=pe, smoothing=1, alpha=2.0, mask=[1, 1, 0])
    ne = r["next_emb"][0]
    np.testing.assert_array_equal(ne[0], emb[3])               # committed now
    np.testing.assert_array_equal(ne[1], emb[9] + 2.0 * 0.5)    # smoothed mask row
    np.testing.assert_array_equal(ne[2], emb[9])                # committed earlier (token = mask_id here)
