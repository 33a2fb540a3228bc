"""Python face of the native step-level scheduler (include/dllm_sched.h).

The deficit token-budget rules (Sangam abstract: in-flight decodes first,
whole prefills only when the accumulated budget allows, unused budget
carried forward) live in the C++ library; this class marshals arguments.
"""

from __future__ import annotations

import ctypes

import numpy as np

from . import _binding as B

POLICIES = {"deficit": 0, "prefill_first": 1, "no_carry": 2}
ENTRY_KEYS = ("slot", "req", "block", "kind", "q_pos0", "q_rows", "kv_rows", "b0")


class Scheduler:
    def __init__(self, slots, blk, vic, quantum, budget_cap, max_step_rows, max_seq, policy="deficit",
                 dual_cache=0):
        cfg = B.SchedConfig(slots, blk, vic, quantum, budget_cap, max_step_rows, max_seq, POLICIES[policy],
                            int(dual_cache))
        h = ctypes.c_void_p()
        B._ck(B.LIB.dllm_sched_create(ctypes.byref(cfg), ctypes.byref(h)), "dllm_sched_create")
        self.h = h
        self.S, self.blk, self.M = slots, blk, max_step_rows
        self._out = (B.SchedEntry * slots)()

    def submit(self, rid, prompt_len, resp_len) -> bool:
        return B.LIB.dllm_sched_submit(self.h, int(rid), int(prompt_len), int(resp_len)) == 0

    def plan_raw(self):
        n = B.LIB.dllm_sched_plan(self.h, self._out, self.S)
        if n < 0:
            raise B.DllmError(-n, "dllm_sched_plan")
        return self._out, n

    def plan(self):
        out, n = self.plan_raw()
        return [{k: getattr(out[i], k) for k in ENTRY_KEYS} for i in range(n)]

    def complete(self, remaining, eos=None):
        rem = np.ascontiguousarray(remaining, dtype=np.int32)
        assert rem.shape == (self.S,)
        eptr = None
        if eos is not None:
            e = np.ascontiguousarray(eos, dtype=np.uint8)
            eptr = e.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))
        rc = B.LIB.dllm_sched_complete(self.h, rem.ctypes.data_as(B._I32P), eptr)
        B._ck(rc, "dllm_sched_complete")

    @property
    def D(self) -> int:
        return int(B.LIB.dllm_sched_budget(self.h))

    def queued(self) -> int:
        return int(B.LIB.dllm_sched_queued(self.h))

    def finished(self):
        buf = (ctypes.c_int32 * 256)()
        got = []
        while True:
            n = B.LIB.dllm_sched_finished(self.h, buf, 256)
            got += list(buf[:n])
            if n < 256:
                return got

    def close(self):
        if self.h:
            B.LIB.dllm_sched_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pack(entries_raw, n, slots, blk):
    """q_off, kv_off [slots + 1] and row_req, row_pos [n * blk] (int32 numpy)
    of a planned step, batch index = slot."""
    q_off = np.zeros(slots + 1, np.int32)
    kv_off = np.zeros(slots + 1, np.int32)
    row_req = np.zeros(max(1, n * blk), np.int32)
    row_pos = np.zeros(max(1, n * blk), np.int32)
    P = B._I32P
    R = B.LIB.dllm_sched_pack(entries_raw, n, slots, blk, q_off.ctypes.data_as(P), kv_off.ctypes.data_as(P),
                              row_req.ctypes.data_as(P), row_pos.ctypes.data_as(P))
    if R < 0:
        raise B.DllmError(-R, "dllm_sched_pack")
    return q_off, kv_off, row_req[:R], row_pos[:R]
