"""The native scheduler (C ABI, host code) against the scheduler oracle:
identical plans, budgets and finishing order, step by step (CPU only)."""

import numpy as np
import pytest

from oracle.sched import Scheduler as OracleSched

from block_decoding_gb300.sched import Scheduler, pack


def _pair(**cfg):
    return OracleSched(**cfg), Scheduler(**cfg)


def _same_plan(a, b):
    ea, eb = a.plan(), b.plan()
    assert ea == eb
    assert a.D == b.D
    return ea


@pytest.mark.parametrize("policy", ["deficit", "prefill_first", "no_carry"])
@pytest.mark.parametrize("dual", [0, 1])
def test_random_traces_match_the_oracle(policy, dual):
    cfg = dict(slots=4, blk=8, vic=4, quantum=70, budget_cap=180, max_step_rows=4 * 16 + 300, max_seq=300,
               policy=policy, dual_cache=dual)
    o, n = _pair(**cfg)
    rng = np.random.default_rng(11 + dual)
    left, nxt, eos_p = {}, 0, 0.02
    for step in range(4000):
        if nxt < 60 and rng.random() < 0.06:
            P, nb = int(rng.integers(0, 200)), int(rng.integers(1, 6))
            bad = rng.random() < 0.05
            args = (nxt, P, 8 * nb + (3 if bad else 0))
            assert o.submit(*args) == n.submit(*args) == (not bad)
            nxt += 1
        es = _same_plan(o, n)
        rem = np.ones(cfg["slots"], np.int32)
        eos = np.zeros(cfg["slots"], np.uint8)
        for e in es:
            key = (e["req"], e["block"])
            left[key] = (8 if e["kind"] == 1 else left[key]) - int(rng.integers(1, 4))
            rem[e["slot"]] = max(0, left[key])
            eos[e["slot"]] = rng.random() < eos_p
        o.complete(list(rem), list(eos))
        n.complete(rem, eos)
        assert len(o.queue) == n.queued()
    assert o.finished == n.finished()


def test_hand_trace_carry_forward():
    """The carried-budget trace of the oracle pins, through the C ABI."""
    s = Scheduler(4, 32, 32, quantum=100, budget_cap=1000, max_step_rows=8192, max_seq=1024)
    s.submit(0, 64, 64)
    assert [(e["req"], e["kind"]) for e in s.plan()] == [(0, 1)] and s.D == -28
    s.complete([5, 1, 1, 1])
    s.submit(1, 64, 64)
    for k in range(2, 80):
        if any(e["kind"] == 1 for e in s.plan()):
            break
        s.complete([5, 1, 1, 1])
    assert k == 40


def test_plan_and_complete_must_alternate():
    s = Scheduler(2, 32, 0, quantum=100, budget_cap=100, max_step_rows=1024, max_seq=512)
    s.submit(0, 0, 32)
    s.plan()
    with pytest.raises(Exception):
        s.plan()
    s.complete([0, 0])
    with pytest.raises(Exception):
        s.complete([0, 0])
    assert s.finished() == [0]


def test_create_rejects_bad_configs():
    with pytest.raises(Exception):
        Scheduler(4, 32, 32, quantum=100, budget_cap=50, max_step_rows=8192, max_seq=1024)   # cap < quantum
    with pytest.raises(Exception):
        Scheduler(4, 32, 32, quantum=100, budget_cap=100, max_step_rows=300, max_seq=256)    # < 4 windows
    with pytest.raises(Exception):
        Scheduler(4, 65, 0, quantum=100, budget_cap=100, max_step_rows=8192, max_seq=1024)   # blk > 64


def test_pack_orders_by_slot_and_leaves_absent_slots_empty():
    s = Scheduler(4, 4, 2, quantum=10000, budget_cap=10000, max_step_rows=4096, max_seq=512)
    s.submit(7, 10, 8)       # slot 0
    s.submit(8, 20, 4)       # slot 1
    s.plan()
    s.complete([2, 0, 1, 1])                # 8 finishes -> slot 1 free
    s.submit(9, 5, 4)                       # takes slot 1
    raw, n = s.plan_raw()                   # decode of 7 (slot 0), prefill of 9 (slot 1)
    ents = [(raw[i].slot, raw[i].kind, raw[i].q_rows, raw[i].kv_rows) for i in range(n)]
    assert ents == [(0, 0, 8, 16), (1, 1, 9, 9)]   # window [8, 16) of T = 18; prefill T = 9
    q_off, kv_off, rr, rp = pack(raw, n, 4, 4)
    assert list(q_off) == [0, 8, 17, 17, 17] and list(kv_off) == [0, 16, 25, 25, 25]
    assert list(rr) == [0, 0, 0, 0, 1, 1, 1, 1] and list(rp) == [0, 1, 2, 3] * 2
