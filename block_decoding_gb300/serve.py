"""Step-level serving loop over dllm_denoise_step.

Before every denoising step the native scheduler (include/dllm_sched.h:
deficit token budget, in-flight decodes first, whole prefills when the
carried budget allows -- Sangam abstract; admission and eviction between
steps -- serving study, design principles) plans which resident requests
decode and which prefills start. The plan is packed into one ragged batch
whose batch index is the cache slot (slots not in the plan get no rows and
keep their committed block state), run as one dllm_denoise_step, and the
per-slot commit counts come back to the host to drive the next plan.

A decode entry runs its window rows over keys [0, window end) (or the whole
sequence with the dual cache); a prefill entry runs every position of the
sequence over every key, and its block rows give the block's first commit.
Query, key and value rows are the first rows of fixed synthetic buffers
(the step costs are real, the activations are not a model's); the block
state of every slot is real and carried across steps.
"""

from __future__ import annotations

import time

import numpy as np
import torch

from . import _binding as B
from .sched import Scheduler, pack


class StepServer:
    def __init__(self, bufs, *, slots, blk, vic, params, quantum, budget_cap, max_step_rows, max_seq,
                 policy="deficit", dual_cache=1, eos_id=-1, device="cuda"):
        """bufs: device tensors q [>= max_step_rows][H][dh], k, v [>= slots *
        max_seq][H][dh], w_head, emb [V][d], hidden [>= slots * blk][d]
        (bf16)."""
        dev = torch.device(device)
        self.b = bufs
        self.S, self.blk, self.params = slots, blk, dict(params)
        self.H, self.dh = bufs["q"].shape[1], bufs["q"].shape[2]
        d = bufs["w_head"].shape[1]
        if bufs["q"].shape[0] < max_step_rows or bufs["k"].shape[0] < slots * max_seq \
                or bufs["hidden"].shape[0] < slots * blk:
            raise ValueError("step buffers smaller than the scheduler's limits")
        self.sched = Scheduler(slots, blk, vic, quantum, budget_cap, max_step_rows, max_seq, policy, dual_cache)
        mask_id = int(params["mask_id"])
        self.mask_id = mask_id
        self.mask = torch.zeros((slots, blk), dtype=torch.uint8, device=dev)   # all committed: idle
        self.tokens = torch.full((slots, blk), mask_id, dtype=torch.int32, device=dev)
        self.credit = torch.zeros((slots, blk), dtype=torch.float32, device=dev)
        self.prev = torch.full((slots, blk), -1, dtype=torch.int32, device=dev)
        self.next_emb = torch.zeros((slots, blk, d), dtype=torch.bfloat16, device=dev)
        self.n_commit = torch.zeros(slots, dtype=torch.int32, device=dev)
        R = slots * blk
        self.argmax = torch.empty(R, dtype=torch.int32, device=dev)
        self.conf = torch.empty(R, dtype=torch.float32, device=dev)
        self.pe = torch.empty((R, d), dtype=torch.float32, device=dev) if params["smoothing"] else None
        self.attn_out = torch.empty_like(bufs["q"][:max_step_rows])
        nmeta = 2 * (slots + 1) + 2 * R
        self.meta_host = torch.zeros(nmeta, dtype=torch.int32).pin_memory()
        self.meta_dev = torch.zeros(nmeta, dtype=torch.int32, device=dev)
        self.commit_host = torch.zeros(slots, dtype=torch.int32).pin_memory()
        self.tok_host = torch.zeros((slots, blk), dtype=torch.int32).pin_memory()
        self.remaining = np.zeros(slots, np.int32)
        self.eos_id = int(eos_id)
        self.ws = None
        self.dev = dev
        self.last = None           # host view of the last step, for tests

    def submit(self, rid, prompt_len, resp_len) -> bool:
        return self.sched.submit(rid, prompt_len, resp_len)

    def step(self, stream=None):
        """Plan, run and complete one step. Returns the planned entries
        (list of dicts) or None when nothing is runnable."""
        raw, n = self.sched.plan_raw()
        if n == 0:
            self.sched.complete(self.remaining)
            return None
        ents = [{k: getattr(raw[i], k) for k in ("slot", "req", "block", "kind", "q_pos0", "q_rows", "kv_rows",
                                                 "b0")} for i in range(n)]
        S, blk = self.S, self.blk
        q_off, kv_off, rr, rp = pack(raw, n, S, blk)
        if int(q_off[-1]) > self.attn_out.shape[0] or int(kv_off[-1]) > self.b["k"].shape[0]:
            raise RuntimeError("planned step exceeds the step buffers")
        R = n * blk
        m = self.meta_host.numpy()
        m[:S + 1] = q_off
        m[S + 1:2 * S + 2] = kv_off
        m[2 * S + 2:2 * S + 2 + R] = rr
        m[2 * S + 2 + R:2 * S + 2 + 2 * R] = rp
        self.meta_dev.copy_(self.meta_host, non_blocking=True)
        starts = [e["slot"] for e in ents if e["kind"] == 1]
        if starts:
            # a prefill starts the slot's block: every position masked, no history
            idx = torch.tensor(starts, dtype=torch.long).to(self.dev, non_blocking=True)
            self.mask.index_fill_(0, idx, 1)
            self.tokens.index_fill_(0, idx, self.mask_id)
            self.credit.index_fill_(0, idx, 0.0)
            self.prev.index_fill_(0, idx, -1)
        md = self.meta_dev
        a = B.step_args(q=self.b["q"], k=self.b["k"], v=self.b["v"], attn_out=self.attn_out,
                        q_off=md[:S + 1], kv_off=md[S + 1:2 * S + 2],
                        max_q=max(e["q_rows"] for e in ents), max_kv=max(e["kv_rows"] for e in ents),
                        hidden=self.b["hidden"][:R], w_head=self.b["w_head"], emb=self.b["emb"],
                        argmax=self.argmax[:R], conf=self.conf[:R],
                        pe=self.pe[:R] if self.pe is not None else None,
                        row_req=md[2 * S + 2:2 * S + 2 + R], row_pos=md[2 * S + 2 + R:2 * S + 2 + 2 * R],
                        mask=self.mask, tokens=self.tokens, credit=self.credit, prev=self.prev,
                        next_emb=self.next_emb, n_commit=self.n_commit, params=self.params)
        need = B.denoise_step_workspace(a)
        if self.ws is None or self.ws.numel() < need:
            self.ws = B.workspace(need, self.dev)
        self.last = dict(entries=ents, q_off=q_off, kv_off=kv_off, row_req=rr, row_pos=rp, R=R, args=a)
        B.denoise_step(a, self.ws, stream)
        self.commit_host.copy_(self.n_commit, non_blocking=True)
        if self.eos_id >= 0:
            self.tok_host.copy_(self.tokens, non_blocking=True)
        torch.cuda.current_stream(self.dev).synchronize()
        nc = self.commit_host.numpy()
        for e in ents:
            s = e["slot"]
            if e["kind"] == 1:
                self.remaining[s] = blk
            self.remaining[s] -= nc[s]
        eos = None
        if self.eos_id >= 0:
            eos = np.zeros(S, np.uint8)
            for e in ents:
                s = e["slot"]
                if self.remaining[s] == 0:
                    eos[s] = bool((self.tok_host.numpy()[s] == self.eos_id).any())
        self.sched.complete(self.remaining, eos)
        for e in ents:
            e["n_commit"] = int(nc[e["slot"]])
        return ents


def run_trace(server: StepServer, trace, max_steps=1_000_000, on_step=None, id_base=0):
    """Feed a request trace (``workloads.make_serve_trace``) through the
    server on a simulated clock that advances by each step's measured wall
    time (plan + launch + the host's read of the commit counts), jumping
    ahead to the next arrival when nothing is runnable. Returns per-request
    and per-step records."""
    arr = np.asarray(trace["arrival_ms"], dtype=np.float64)
    P, Lr = trace["prompt_len"], trace["resp_len"]
    n = len(arr)
    req = {i: dict(arrival=float(arr[i]), first=None, finish=None, tokens=0) for i in range(n)}
    steps = []
    now, nxt, done = 0.0, 0, 0
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    while done < n and len(steps) < max_steps:
        while nxt < n and arr[nxt] <= now:
            if not server.submit(id_base + nxt, int(P[nxt]), int(Lr[nxt])):
                raise ValueError(f"request {nxt} rejected by the scheduler")
            nxt += 1
        t0 = time.perf_counter()
        ev0.record()
        ents = server.step()
        ev1.record()
        ev1.synchronize()
        wall = (time.perf_counter() - t0) * 1e3
        if ents is None:
            if nxt >= n:
                raise RuntimeError("idle with requests outstanding")
            now = max(now, float(arr[nxt]))
            continue
        gpu = ev0.elapsed_time(ev1)
        now += wall
        for e in ents:
            r = req[e["req"] - id_base]
            r["tokens"] += e["n_commit"]
            if r["first"] is None:
                r["first"] = now
        for rid in server.sched.finished():
            req[rid - id_base]["finish"] = now
            done += 1
        steps.append(dict(t=now, wall_ms=wall, gpu_ms=gpu, n=len(ents),
                          prefills=sum(e["kind"] for e in ents), rows=sum(e["q_rows"] for e in ents),
                          budget=server.sched.D))
        if on_step is not None:
            on_step(server, ents)
    return dict(requests=req, steps=steps, makespan_ms=now)


def summarize(res):
    """Throughput and latency figures of ``run_trace``'s records."""
    reqs = [r for r in res["requests"].values() if r["finish"] is not None]
    lat = np.array([r["finish"] - r["arrival"] for r in reqs])
    ttfc = np.array([r["first"] - r["arrival"] for r in reqs])
    st = res["steps"]
    wall = np.array([s["wall_ms"] for s in st])
    gpu = np.array([s["gpu_ms"] for s in st])
    pre = np.array([s["prefills"] > 0 for s in st])
    toks = sum(r["tokens"] for r in reqs)
    q = lambda a, p: float(np.percentile(a, p)) if len(a) else None  # noqa: E731
    return dict(requests=len(reqs), committed_tokens=int(toks), makespan_ms=res["makespan_ms"],
                tok_per_s=toks / (res["makespan_ms"] / 1e3) if res["makespan_ms"] > 0 else None,
                latency_ms=dict(mean=float(lat.mean()), p50=q(lat, 50), p90=q(lat, 90), p99=q(lat, 99)),
                first_commit_ms=dict(mean=float(ttfc.mean()), p50=q(ttfc, 50), p90=q(ttfc, 90)),
                steps=len(st), step_wall_ms_mean=float(wall.mean()), step_gpu_ms_mean=float(gpu.mean()),
                step_gpu_ms_p99=q(gpu, 99),
                decode_only_step_gpu_ms=float(gpu[~pre].mean()) if (~pre).any() else None,
                prefill_step_gpu_ms=float(gpu[pre].mean()) if pre.any() else None,
                prefill_step_share=float(pre.mean()))
