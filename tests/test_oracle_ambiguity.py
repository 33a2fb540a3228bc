"""Pins for the oracle's ambiguity record and top-2 gap (CPU only).

The parity protocol compares committed sets and argmax ids bit-exactly except
where the two sides may decide differently for rounding reasons alone: a
confidence or credit within 1e-3 of tau or kappa, an argmax whose top-2
logits nearly tie, and (readings of the same rule) a close tie of two
equidistant candidates in the hierarchical selection or of the two best
confidences in the fallback. For each request the record lists every
selection the commit can reach with those decisions taken either way; the
device must commit one of them (exactly the oracle's own when there is only
one). Every case below is built by hand so that the flagged positions and
the allowed selections are known by construction; a rule that allows too
much or too little fails one of them.
"""

import math

import numpy as np
import pytest

import oracle
from oracle.step import (ARGMAX_GAP_REL, FALLBACK_GAP_REL, MAX_FLIPS, THRESH_BAND, ambiguity,
                         hierarchical_choices, hierarchical_close_tie, top2_gap)

F32 = np.float32
V = 6
PARAMS = dict(tau=0.9, lam=0.7, kappa=1.5, hierarchical=1, hier_levels=1,
              smoothing=0, alpha=1.0, mask_id=V - 1)


def _row_with_conf(p, a):
    """Logits over V entries whose softmax max is p, at token a (V - 1 zeros)."""
    z = np.zeros(V)
    z[a] = math.log(p * (V - 1) / (1.0 - p))
    return z


def _row_with_gap(m, g, a, b):
    """Logits with the largest m at a and the second m - g at b."""
    z = np.full(V, m - 30.0)
    z[a] = m
    z[b] = m - g
    return z


def _run(zrows, mask, prev=None, credit=None, **prm):
    """One request: head rows for the masked positions (in position order)."""
    mask = np.asarray(mask, np.uint8)[None]
    blk = mask.shape[1]
    pos = np.flatnonzero(mask[0])
    assert len(pos) == len(zrows)
    params = dict(PARAMS, **prm)
    z = np.asarray(zrows, np.float64).reshape(-1, V)
    m, a, l, conf = oracle.vocab_softmax_stats(z)
    head = dict(z=z, m=m, l=l, argmax=a, conf=conf, pe=None)
    prev = np.full((1, blk), -1, np.int32) if prev is None else np.asarray(prev, np.int32)[None]
    credit = np.zeros((1, blk), F32) if credit is None else np.asarray(credit, F32)[None]
    inp = dict(params=params, mask=mask, row_req=np.zeros(len(pos), np.int32),
               row_pos=pos.astype(np.int32), credit=credit, prev=prev,
               tokens=np.full((1, blk), V - 1, np.int32))
    com = oracle.commit(a, conf, None, inp["row_req"], inp["row_pos"], mask, inp["tokens"],
                        credit, prev, np.eye(V, 4), params)
    return ambiguity(inp, head, com), com


# --------------------------------------------------------------------------
# top-2 gap
# --------------------------------------------------------------------------

def test_top2_gap_special_cases():
    gap, sc = top2_gap(np.array([[2.5]]))            # V = 1: no second logit
    assert gap[0] == np.inf and sc[0] == 2.5
    gap, sc = top2_gap(np.array([[3.0, 1.0], [0.25, 0.5]]))   # V = 2
    assert gap.tolist() == [2.0, 0.25] and sc.tolist() == [3.0, 1.0]
    gap, sc = top2_gap(np.array([[2.0, 0.0, 2.0]]))   # exact tie
    assert gap[0] == 0.0 and sc[0] == 2.0
    gap, sc = top2_gap(np.array([[-50.0, -50.5, -70.0]]))   # negative maximum: |m| scales
    assert gap[0] == 0.5 and sc[0] == 50.0


@pytest.mark.parametrize("m", [0.5, 20.0, -20.0])
def test_argmax_gap_band_is_relative_to_max_one(m):
    band = ARGMAX_GAP_REL * max(1.0, abs(m))
    zrows = [_row_with_gap(m, 0.99 * band, 1, 2), _row_with_gap(m, 1.01 * band, 3, 0),
             _row_with_conf(0.5, 4)]
    amb, _ = _run(zrows, [1, 1, 1], hierarchical=0)
    assert amb["argmax_row"].tolist() == [True, False, False]
    assert amb["argmax_pos"][0].tolist() == [True, False, False]
    assert amb["position"][0].tolist() == [True, False, False]
    assert amb["counts"]["argmax_rows"] == 1


# --------------------------------------------------------------------------
# confidence and credit bands
# --------------------------------------------------------------------------

def test_threshold_band_on_p():
    tau = PARAMS["tau"]
    ps = [tau - 2e-3, tau - 0.5e-3, tau + 0.5e-3, tau + 2e-3]
    amb, com = _run([_row_with_conf(p, 1) for p in ps], [1, 1, 1, 1], hierarchical=0)
    assert amb["position"][0].tolist() == [False, True, True, False]
    assert amb["argmax_pos"][0].tolist() == [False] * 4
    assert amb["counts"]["near_threshold"] == 2
    # hierarchy off (S = C): positions 1 and 2 may each go either way
    assert com["cand"][0].tolist() == [False, False, True, True]
    assert _choices(amb) == {(3,), (2, 3), (1, 3), (1, 2, 3)}
    assert not amb["selection"].any() and not amb["request"][0]


@pytest.mark.parametrize("changed", [False, True])
def test_credit_band_after_update(changed):
    """credit' = lam*credit + p while the argmax holds, p after a change."""
    kappa, lam = PARAMS["kappa"], PARAMS["lam"]
    p = 0.5
    targets = [kappa - 2e-3, kappa - 0.5e-3, kappa + 0.5e-3, kappa + 2e-3]
    credit = [F32((t - p) / lam) for t in targets]
    prev = [7, 7, 7, 7] if changed else [1, 1, 1, 1]
    amb, com = _run([_row_with_conf(p, 1)] * 4, [1] * 4, prev=prev, credit=credit, hierarchical=0)
    if changed:
        # the history is dropped: credit' = p, nowhere near kappa
        assert np.allclose(com["credit_upd"][0], p)
        assert amb["position"][0].tolist() == [False] * 4
    else:
        assert amb["position"][0].tolist() == [False, True, True, False]
        assert com["cand"][0].tolist() == [False, False, True, True]


def test_credit_band_is_decided_in_float32():
    """Two (credit, p) pairs whose float32 update lands on the other side of
    the band edge from the float64 value of the same expression: the flag
    follows the float32 value the commit decided with."""
    kappa, lam = PARAMS["kappa"], PARAMS["lam"]
    cases = [(1.6016584634780884, 0.37983909249305725, True),    # float32 inside, float64 outside
             (1.5954933166503906, 0.3821547329425812, False)]    # float32 outside, float64 inside
    for c, p, inside in cases:
        c32, p32 = F32(c), F32(p)
        cr32 = float(F32(F32(F32(lam) * c32) + p32))
        cr64 = lam * float(c32) + float(p32)
        assert (abs(cr32 - kappa) < THRESH_BAND) == inside
        assert (abs(cr64 - kappa) < THRESH_BAND) != inside
        amb, com = _run([_row_with_conf(float(p32), 2)], [1], prev=[2], credit=[c32], hierarchical=0)
        assert float(com["p"][0, 0]) == float(p32)
        assert float(com["credit_upd"][0, 0]) == cr32
        assert bool(amb["position"][0, 0]) == inside


# --------------------------------------------------------------------------
# selection: spans, ties, fallback
# --------------------------------------------------------------------------

def _choices(amb, i=0):
    return {tuple(sorted(c)) for c in amb["choices"][i]}


def test_hierarchical_flip_changes_only_its_own_span():
    # spans [0, 3) and [4, 8); position 1 (the centre of [0, 3)) sits on the
    # tau band; span [4, 8) has a clean candidate at its centre 5
    tau = PARAMS["tau"]
    mask = [1, 1, 1, 0, 1, 1, 1, 1]
    ps = [0.3, tau + 0.5e-3, 0.97, 0.3, 0.97, 0.3, 0.3]
    amb, com = _run([_row_with_conf(p, 1) for p in ps], mask)
    assert com["selected"][0].tolist() == [False, True, False, False, False, True, False, False]
    # 1 a candidate: the centre; not: the other candidate, 2
    assert _choices(amb) == {(1, 5), (2, 5)}
    assert not amb["request"][0] and not amb["selection"].any()
    assert amb["counts"]["requests_with_choices"] == 1


def test_a_flip_that_cannot_change_the_pick_leaves_one_choice():
    tau = PARAMS["tau"]
    # the only candidate is on the band; without it the fallback commits the
    # most confident position, which is that same one
    amb, _ = _run([_row_with_conf(p, 1) for p in [0.3, tau + 0.5e-3, 0.3, 0.3, 0.3, 0.3, 0.3]],
                  [1, 1, 1, 0, 1, 1, 1, 1])
    assert _choices(amb) == {(1,)}
    # a band position farther from the centre than the clean pick
    amb, _ = _run([_row_with_conf(p, 1) for p in [tau + 0.5e-3, 0.97, 0.3]], [1, 1, 1])
    assert _choices(amb) == {(1,)}


def test_hierarchical_close_tie_of_equidistant_candidates():
    # centre 1 of [0, 3) is no candidate; 0 and 2 are equally far from it
    close = [0.95, 0.3, 0.95 * (1 + 0.5 * FALLBACK_GAP_REL)]
    clear = [0.95, 0.3, 0.92]
    amb, com = _run([_row_with_conf(p, 1) for p in close], [1, 1, 1])
    assert com["selected"][0].tolist() == [False, False, True]
    assert _choices(amb) == {(0,), (2,)}
    amb, com = _run([_row_with_conf(p, 1) for p in clear], [1, 1, 1])
    assert com["selected"][0].tolist() == [True, False, False]
    assert _choices(amb) == {(0,)}
    # hierarchy off takes every candidate: no tie to break
    amb, _ = _run([_row_with_conf(p, 1) for p in close], [1, 1, 1], hierarchical=0)
    assert _choices(amb) == {(0, 2)}


def test_close_tie_counts_only_at_the_levels_walked():
    # [0, 7): centre 3 is a candidate; [0, 3) then has a close tie of 0 and 2,
    # which only a second level reaches
    ps = [0.95, 0.3, 0.9504, 0.99, 0.3, 0.3, 0.3]
    amb1, _ = _run([_row_with_conf(p, 1) for p in ps], [1] * 7, hier_levels=1)
    amb2, _ = _run([_row_with_conf(p, 1) for p in ps], [1] * 7, hier_levels=2)
    assert _choices(amb1) == {(3,)}
    assert _choices(amb2) == {(0, 3), (2, 3)}
    cand = np.array([True, False, True, True, False, False, False])
    p = np.array(ps, F32)
    assert not hierarchical_close_tie(cand, p, 0, 7, 1)
    assert hierarchical_close_tie(cand, p, 0, 7, 2)
    # a third level fills [0, 3) completely: both branches reach {0, 2, 3}
    assert {tuple(sorted(c)) for c in hierarchical_choices(cand, p, 0, 7, 3)} == {(0, 2, 3)}


@pytest.mark.parametrize("hier", [0, 1])
def test_fallback_gap(hier):
    close = [0.2, 0.5, 0.5 * (1 - 0.8 * FALLBACK_GAP_REL)]
    clear = [0.2, 0.5, 0.498]
    amb, com = _run([_row_with_conf(p, 1) for p in close], [1, 1, 1], hierarchical=hier)
    assert com["fallback"][0] and com["selected"][0].tolist() == [False, True, False]
    assert _choices(amb) == {(1,), (2,)}
    amb, com = _run([_row_with_conf(p, 1) for p in clear], [1, 1, 1], hierarchical=hier)
    assert com["fallback"][0] and _choices(amb) == {(1,)}


def test_band_position_that_may_lift_the_fallback():
    tau = PARAMS["tau"]
    # 2 is on the band below tau: as a candidate it is the pick nearest the
    # centre, and without it the fallback picks it as the most confident
    amb, com = _run([_row_with_conf(p, 1) for p in [0.2, 0.5, tau - 0.5e-3]], [1, 1, 1])
    assert com["fallback"][0] and _choices(amb) == {(2,)}
    # hierarchy off, the band candidate is the only one, another position is
    # the most confident: a flip moves the commit from {0} to {1}
    amb, com = _run([_row_with_conf(p, 1) for p in [tau + 0.5e-3, 0.3, 0.2]], [1, 1, 1], hierarchical=0)
    assert _choices(amb) == {(0,)}
    ps = [tau + 0.5e-3, 0.3, 0.2]
    cr = [0.0, 0.0, 0.0]
    # credit path: 1 holds its argmax with credit reaching kappa exactly on
    # the band; 0 is a clean candidate by p
    lam, kappa = PARAMS["lam"], PARAMS["kappa"]
    cr[1] = F32((kappa + 0.5e-3 - 0.3) / lam)
    amb, com = _run([_row_with_conf(p, 1) for p in [0.95, 0.3, 0.2]], [1, 1, 1], prev=[-1, 1, -1],
                    credit=cr, hierarchical=0)
    assert com["cand"][0].tolist() == [True, True, False]
    assert _choices(amb) == {(0,), (0, 1)}


def test_no_hierarchy_flip_of_one_of_two_candidates():
    tau = PARAMS["tau"]
    amb, com = _run([_row_with_conf(p, 1) for p in [tau + 0.5e-3, 0.95, 0.2]], [1, 1, 1],
                    hierarchical=0)
    assert _choices(amb) == {(0, 1), (1,)}
    assert not amb["request"][0]


def test_too_many_uncertain_positions_exclude_the_request():
    tau = PARAMS["tau"]
    n = MAX_FLIPS + 1
    amb, _ = _run([_row_with_conf(tau + 0.5e-3, 1)] * n, [1] * n, hierarchical=0)
    assert amb["request"][0] and amb["selection"][0].all() and amb["choices"][0] is None
    assert amb["counts"]["requests"] == 1 and amb["counts"]["selection_positions"] == n


def test_unmasked_positions_and_empty_requests():
    tau = PARAMS["tau"]
    amb, _ = _run([_row_with_conf(tau + 0.5e-3, 1)], [0, 1, 0])
    assert amb["position"][0].tolist() == [False, True, False]
    assert _choices(amb) == {(1,)}
    amb, _ = _run([], [0, 0, 0])
    assert _choices(amb) == {()}


def test_the_oracle_selection_is_always_a_choice():
    """Random requests, thresholds, credit and ties: the oracle's own
    selection is one of the allowed ones, and without any uncertain
    position or close tie it is the only one."""
    rng = np.random.default_rng(3)
    for trial in range(300):
        blk = int(rng.integers(1, 12))
        mask = (rng.random(blk) < 0.8).astype(np.uint8)
        n = int(mask.sum())
        ps = rng.choice([0.3, 0.6, 0.95, 0.9995, 0.9 + 0.4e-3, 0.9 - 0.4e-3], n)
        hier = int(rng.integers(0, 2))
        levels = int(rng.choice([1, 2, 64]))
        amb, com = _run([_row_with_conf(float(p), 1) for p in ps], mask, hierarchical=hier, hier_levels=levels)
        own = tuple(sorted(np.flatnonzero(com["selected"][0]).tolist()))
        assert own in _choices(amb), trial
        if not amb["position"].any() and len(set(np.round(ps, 6))) == len(ps):
            assert _choices(amb) == {own}, trial
