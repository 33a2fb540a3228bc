"""Pins of the scheduler oracle: hand-worked traces of the deficit budget
(Sangam abstract: in-flight decodes first, whole prefills when the
accumulated budget allows, unused budget carried forward) and invariants on
random traces."""

import numpy as np
import pytest

from oracle.sched import Scheduler

BIG = dict(max_step_rows=8192, max_seq=1024)


def test_first_admissions_and_window_costs():
    # T = 128: block 0 at b0 = 64, window [32, 128) = 96 rows, keys [0, 128)
    s = Scheduler(4, 32, 32, quantum=200, budget_cap=400, **BIG)
    assert s.submit(0, 64, 64) and s.submit(1, 64, 64)
    e1 = s.plan()                      # D = 200: r0 (128) in, D = 72; r1 128 > 72
    assert [(e["req"], e["kind"], e["slot"]) for e in e1] == [(0, 1, 0)]
    assert e1[0]["q_rows"] == 128 and e1[0]["kv_rows"] == 128 and e1[0]["b0"] == 64
    assert s.D == 72
    s.complete([31, 0, 0, 0], [0] * 4)
    e2 = s.plan()                      # D = 272 - 96 = 176 >= 128: r1 in, D = 48
    assert [(e["req"], e["kind"], e["slot"]) for e in e2] == [(0, 0, 0), (1, 1, 1)]
    assert (e2[0]["q_pos0"], e2[0]["q_rows"], e2[0]["kv_rows"]) == (32, 96, 128)
    assert s.D == 48


def test_carry_forward_admits_after_exactly_enough_steps():
    """A decode of 96 rows per step under a quantum of 100 nets +4 a step:
    the 128-row prefill behind it waits until the carried budget covers it."""
    s = Scheduler(4, 32, 32, quantum=100, budget_cap=1000, **BIG)
    s.submit(0, 64, 64)
    e = s.plan()                       # 128 > 100, nothing else: work conservation
    assert [x["req"] for x in e] == [0] and s.D == 100 - 128
    s.complete([5, 1, 1, 1], [0] * 4)
    s.submit(1, 64, 64)
    admitted_at = None
    for k in range(2, 80):
        es = s.plan()
        # before the prefill check: D_k = -28 + 100 (k - 1) - 96 (k - 1) = -28 + 4 (k - 1)
        if any(x["kind"] == 1 for x in es):
            admitted_at = k
            break
        assert s.D == -28 + 4 * (k - 1)
        s.complete([5, 1, 1, 1], [0] * 4)
    assert admitted_at == 40          # first k with -28 + 4 (k - 1) >= 128


def test_no_carry_starves_and_prefill_first_does_not():
    for policy, expect in (("no_carry", None), ("prefill_first", 2)):
        s = Scheduler(4, 32, 32, quantum=100, budget_cap=1000, policy=policy, **BIG)
        s.submit(0, 64, 64)
        s.plan()
        s.complete([5, 1, 1, 1], [0] * 4)
        s.submit(1, 64, 64)
        got = None
        for k in range(2, 200):
            if any(x["kind"] == 1 for x in s.plan()):
                got = k
                break
            s.complete([5, 1, 1, 1], [0] * 4)
        assert got == expect, policy


def test_cap_bounds_the_budget():
    s = Scheduler(4, 32, 32, quantum=100, budget_cap=120, **BIG)
    s.submit(0, 64, 64)
    s.plan()
    s.complete([5, 1, 1, 1], [0] * 4)
    s.submit(1, 64, 64)
    for _ in range(100):               # D <= min(120, D + 100) - 96 <= 24 < 128
        assert not any(x["kind"] == 1 for x in s.plan())
        assert s.D <= 24
        s.complete([5, 1, 1, 1], [0] * 4)


def test_strict_fifo_blocks_smaller_prefills_behind():
    s = Scheduler(4, 32, 32, quantum=100, budget_cap=300, **BIG)
    s.submit(0, 64, 64)
    s.plan()                           # r0 in by work conservation
    s.complete([5, 1, 1, 1], [0] * 4)
    s.submit(1, 600, 64)               # 664 rows: never within a cap of 300
    s.submit(2, 0, 32)                 # 32 rows, would fit
    for _ in range(50):
        assert [x["req"] for x in s.plan()] == [0]
        s.complete([5, 1, 1, 1], [0] * 4)
    # r0's second block is queued behind r1 and r2 when its first block ends
    s.plan()
    s.complete([0, 1, 1, 1], [0] * 4)
    assert [r.rid for r in s.queue] == [1, 2, 0]
    es = s.plan()                      # nothing in flight: r1 by work conservation
    assert [(x["req"], x["kind"]) for x in es] == [(1, 1)]


def test_slots_pass_over_new_requests_but_not_resident_ones():
    s = Scheduler(1, 32, 0, quantum=1000, budget_cap=1000, **BIG)
    s.submit(0, 32, 64)                # two blocks
    s.submit(1, 32, 32)
    assert [(x["req"], x["slot"]) for x in s.plan()] == [(0, 0)]   # r1: no slot
    s.complete([0], [0])               # r0 block 0 done -> queue [r1, r0]
    es = s.plan()                      # r1 passed over, r0 (resident) admitted
    assert [(x["req"], x["kind"], x["block"]) for x in es] == [(0, 1, 1)]
    assert es[0]["b0"] == 64
    s.complete([0], [0])               # r0 done, slot freed
    assert s.finished == [0]
    assert [(x["req"], x["slot"]) for x in s.plan()] == [(1, 0)]


def test_eos_evicts_after_the_block():
    s = Scheduler(2, 32, 8, quantum=1000, budget_cap=1000, **BIG)
    s.submit(0, 16, 128)
    s.plan()
    s.complete([0, 0], [1, 0])         # block done with an end token
    assert s.finished == [0] and s.free == [1, 0] and not s.queue


def test_dual_cache_decodes_attend_the_whole_sequence():
    s = Scheduler(2, 32, 16, quantum=10000, budget_cap=10000, dual_cache=1, **BIG)
    s.submit(0, 100, 96)               # T = 196, block 0 window [84, 148)
    s.plan()
    s.complete([3, 1], [0, 0])
    e = s.plan()[0]
    assert (e["kind"], e["q_pos0"], e["q_rows"], e["kv_rows"]) == (0, 84, 64, 196)


def test_submit_rejects_bad_requests():
    s = Scheduler(2, 32, 16, quantum=100, budget_cap=100, **BIG)
    assert not s.submit(0, 10, 40)           # not a whole number of blocks
    assert not s.submit(1, 1000, 64)         # longer than max_seq
    assert s.submit(2, 10, 64) and not s.submit(2, 10, 64)   # duplicate id


@pytest.mark.parametrize("policy", ["deficit", "prefill_first", "no_carry"])
def test_random_traces_keep_the_invariants(policy):
    rng = np.random.default_rng(3)
    s = Scheduler(3, 8, 4, quantum=60, budget_cap=150, max_step_rows=3 * 16 + 256, max_seq=256, policy=policy)
    left = {}
    nxt = 0
    for step in range(3000):
        if nxt < 40 and rng.random() < 0.05:
            P, nb = int(rng.integers(0, 100)), int(rng.integers(1, 5))
            assert s.submit(nxt, P, 8 * nb)
            nxt += 1
        es = s.plan()
        slots = [e["slot"] for e in es]
        assert len(set(slots)) == len(slots)
        assert sum(e["q_rows"] for e in es) <= s.M
        if policy == "deficit":
            assert s.D <= s.cap
        decoding = {i for i, r in enumerate(s.slot_req) if r is not None and r.state == "decoding"}
        assert decoding == set(slots)        # every in-flight decode runs every step
        rem = [1] * s.S
        for e in es:
            key = (e["req"], e["block"])
            left[key] = (8 if e["kind"] == 1 else left[key]) - int(rng.integers(1, 4))
            rem[e["slot"]] = max(0, left[key])
        s.complete(rem, [0] * s.S)
    if policy != "no_carry":
        assert sorted(s.finished) == list(range(nxt)), policy
