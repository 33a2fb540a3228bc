"""Oracle (test infrastructure only): the step-level scheduler of cached
block decoding, written plainly in Python.

What the pages fix (Sangam abstract; serving study, design principles):
  * cached dLLM decoding is a repeated prefill/decode structure: each block
    starts with a refresh of the whole sequence's K/V (an indivisible
    prefill; bidirectional attention rules out chunking it) followed by
    decodes of the block until it is committed;
  * the deficit token-budget scheduler admits the in-flight decodes first,
    admits whole prefills only when the accumulated token budget allows,
    and carries the unused budget into the next cycle;
  * scheduling happens at the granularity of one denoising step, with
    requests admitted and evicted between steps.
Readings (the pages give the policy in one sentence, not its arithmetic):
  * one cycle = one denoising step; every step adds `quantum` tokens to the
    budget, which is then capped at `budget_cap` (the carry ceiling);
  * a step's cost is the number of query rows it runs: a decode of block b
    costs its window [b0 - vic, b0 + blk + vic) clipped to [0, T); a
    prefill costs T (every position of the sequence);
  * every in-flight decode runs every step and is charged, so the budget
    can go negative: the decodes are protected, prefills wait;
  * prefills wait in one FIFO queue (a new request when submitted, a
    resident request when its block is done and another block remains);
    the queue is scanned in order: a request that needs a cache slot when
    none is free is passed over (it keeps its place); the first one whose
    cost exceeds the budget or the step's row cap ends the scan (strict
    FIFO, so a long prefill is not bypassed for ever);
  * work conservation: a step that would run nothing admits the first
    slot-feasible prefill regardless of the budget;
  * a request leaves (its slot is freed) when its last block is committed,
    or when a block that committed its end token (eos) is done;
  * two comparison policies: `prefill_first` (no budget: every ready
    prefill that fits the row cap), `no_carry` (the budget is reset to
    `quantum` every step instead of accumulating).
"""

POLICIES = {"deficit": 0, "prefill_first": 1, "no_carry": 2}


class Request:
    def __init__(self, rid, prompt_len, resp_len, blk):
        self.rid, self.P, self.Lr = rid, prompt_len, resp_len
        self.T = prompt_len + resp_len
        self.nblocks = resp_len // blk
        self.block = 0
        self.slot = -1
        self.state = "queued"            # queued | ready | decoding | done


class Scheduler:
    def __init__(self, slots, blk, vic, quantum, budget_cap, max_step_rows, max_seq, policy="deficit",
                 dual_cache=0):
        assert slots >= 1 and blk >= 1 and vic >= 0 and quantum >= 0 and budget_cap >= quantum
        assert max_step_rows >= slots * (blk + 2 * vic) and max_seq <= max_step_rows
        self.S, self.blk, self.vic = slots, blk, vic
        self.Q, self.cap, self.M, self.max_seq = quantum, budget_cap, max_step_rows, max_seq
        self.policy, self.dual = policy, dual_cache
        self.D = 0
        self.free = list(range(slots))
        self.slot_req = [None] * slots
        self.queue = []                  # prefill FIFO of Request
        self.reqs = {}
        self.last = []
        self.finished = []

    def submit(self, rid, prompt_len, resp_len):
        if rid in self.reqs or resp_len < self.blk or resp_len % self.blk or prompt_len < 0 \
                or prompt_len + resp_len > self.max_seq:
            return False
        r = Request(rid, prompt_len, resp_len, self.blk)
        self.reqs[rid] = r
        self.queue.append(r)
        return True

    def window(self, r):
        b0 = r.P + r.block * self.blk
        return b0, max(0, b0 - self.vic), min(r.T, b0 + self.blk + self.vic)

    def _entry(self, r, kind):
        b0, ws, we = self.window(r)
        if kind == 1:
            return dict(slot=r.slot, req=r.rid, block=r.block, kind=1, q_pos0=0, q_rows=r.T, kv_rows=r.T, b0=b0)
        return dict(slot=r.slot, req=r.rid, block=r.block, kind=0, q_pos0=ws, q_rows=we - ws,
                    kv_rows=r.T if self.dual else we, b0=b0)

    def plan(self):
        if self.policy == "deficit":
            self.D = min(self.cap, self.D + self.Q)
        elif self.policy == "no_carry":
            self.D = self.Q
        entries, used = [], 0
        for s in range(self.S):
            r = self.slot_req[s]
            if r is not None and r.state == "decoding":
                e = self._entry(r, 0)
                entries.append(e)
                used += e["q_rows"]
                if self.policy != "prefill_first":
                    self.D -= e["q_rows"]
        admitted = []
        for r in self.queue:
            if r.slot < 0 and not self.free:
                continue
            fits_rows = used + r.T <= self.M
            fits_budget = self.policy == "prefill_first" or r.T <= self.D
            if not (fits_rows and fits_budget):
                break
            self._admit(r)
            admitted.append(r)
            used += r.T
            if self.policy != "prefill_first":
                self.D -= r.T
        if not entries and not admitted:
            for r in self.queue:
                if r.slot < 0 and not self.free:
                    continue
                self._admit(r)
                admitted.append(r)
                used += r.T
                if self.policy != "prefill_first":
                    self.D -= r.T
                break
        for r in admitted:
            self.queue.remove(r)
            entries.append(self._entry(r, 1))
        self.last = entries
        return entries

    def _admit(self, r):
        if r.slot < 0:
            r.slot = min(self.free)
            self.free.remove(r.slot)
            self.slot_req[r.slot] = r
        r.state = "decoding"

    def complete(self, remaining, eos):
        """remaining[slot]: masked positions left in the slot's block after
        the step; eos[slot]: the block holds a committed end token."""
        for e in self.last:
            r = self.reqs[e["req"]]
            if remaining[e["slot"]] > 0:
                continue
            if r.block + 1 < r.nblocks and not eos[e["slot"]]:
                r.block += 1
                r.state = "ready"
                self.queue.append(r)
            else:
                r.state = "done"
                self.slot_req[r.slot] = None
                self.free.append(r.slot)
                self.finished.append(r.rid)
                r.slot = -1
        self.last = []
