"""GPU: scheduled steps (native scheduler -> packed ragged batch with batch
index = slot -> dllm_denoise_step) against the oracle step on the same
inputs, step by step; and a whole request trace through the serving loop."""

import numpy as np
import pytest
import torch

import oracle
from block_decoding_gb300.serve import StepServer, run_trace, summarize
from helpers import dev_bf16, host_bf16_bits
from parity import check_attention, check_commit, check_head
from workloads import bf16_bits_to_f64, make_serve_inputs, make_serve_trace

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

S, BLK, VIC, MAX_SEQ = 3, 8, 4, 96
M = S * (BLK + 2 * VIC) + MAX_SEQ


def _server(policy="deficit", dual=1, quantum=60, cap=150, seed=5):
    inp = make_serve_inputs(slots=S, blk=BLK, H=2, dh=64, V=512, q_rows=M, kv_rows=S * MAX_SEQ, seed=seed)
    bufs = {k: dev_bf16(inp[k]) for k in ("q", "k", "v", "w_head", "emb", "hidden")}
    srv = StepServer(bufs, slots=S, blk=BLK, vic=VIC, params=inp["params"], quantum=quantum, budget_cap=cap,
                     max_step_rows=M, max_seq=MAX_SEQ, policy=policy, dual_cache=dual)
    return inp, srv


def _host(srv):
    return dict(mask=srv.mask.cpu().numpy(), tokens=srv.tokens.cpu().numpy(), credit=srv.credit.cpu().numpy(),
                prev=srv.prev.cpu().numpy())


@pytest.mark.parametrize("dual", [1, 0])
def test_scheduled_steps_match_the_oracle(dual):
    inp, srv = _server(dual=dual)
    # (step index, prompt, response): ragged prompts, 1 to 4 blocks, more requests than slots
    arrivals = [(0, 20, 16), (0, 60, 8), (0, 5, 32), (2, 40, 16), (3, 0, 8), (5, 70, 24), (9, 33, 8)]
    toks = {}
    n_steps = n_prefill_steps = 0
    for k in range(400):
        for (t, P, L) in arrivals:
            if t == k:
                assert srv.submit(arrivals.index((t, P, L)), P, L)
        before = _host(srv)
        ents = srv.step()
        if ents is None:
            if k > max(a[0] for a in arrivals):
                break
            continue
        last = srv.last
        for e in ents:                       # the reset a prefill does before the step
            if e["kind"] == 1:
                s = e["slot"]
                before["mask"][s] = 1
                before["tokens"][s] = inp["params"]["mask_id"]
                before["credit"][s] = 0
                before["prev"][s] = -1
        R, nq, nkv = last["R"], int(last["q_off"][-1]), int(last["kv_off"][-1])
        ref_in = dict(q=inp["q"][:nq], k=inp["k"][:nkv], v=inp["v"][:nkv], q_off=last["q_off"],
                      kv_off=last["kv_off"], scale=inp["scale"], hidden=inp["hidden"][:R], w_head=inp["w_head"],
                      emb=inp["emb"], row_req=last["row_req"], row_pos=last["row_pos"], params=inp["params"],
                      B=S, blk=BLK, R=R, **before)
        ref = oracle.step.denoise_step(ref_in)
        torch.cuda.synchronize()
        check_attention(srv.attn_out[:nq].float().cpu().numpy(), ref["attn"])
        amb = ref["ambiguity"]
        check_head(srv.argmax[:R].cpu().numpy(), srv.conf[:R].cpu().numpy(), srv.pe[:R].cpu().numpy(),
                   ref["head"], amb_rows=amb["argmax_row"])
        after = dict(_host(srv), n_commit=srv.n_commit.cpu().numpy(), next_emb_bits=host_bf16_bits(srv.next_emb))
        check_commit(ref_in, after, ref["commit"], amb, inp["emb"], pe_ref=ref["head"]["pe"])
        # slots outside the plan are untouched
        planned = {e["slot"] for e in ents}
        for s in set(range(S)) - planned:
            assert np.array_equal(after["mask"][s], before["mask"][s]) and after["n_commit"][s] == 0
        for e in ents:
            toks[e["req"]] = toks.get(e["req"], 0) + e["n_commit"]
        n_steps += 1
        n_prefill_steps += any(e["kind"] for e in ents)
    assert sorted(srv.sched.finished()) == list(range(len(arrivals)))
    assert all(toks[i] == arrivals[i][2] for i in range(len(arrivals)))
    assert n_prefill_steps >= 1 and n_steps > n_prefill_steps


@pytest.mark.parametrize("policy", ["deficit", "prefill_first", "no_carry"])
def test_trace_runs_to_completion(policy):
    _, srv = _server(policy=policy, quantum=40, cap=200)
    trace = make_serve_trace(n=12, rate_per_s=2000.0, prompt_range=(0, 60), resp_choices=(8, 16, 32), seed=4)
    res = run_trace(srv, trace, max_steps=5000)
    sm = summarize(res)
    assert sm["requests"] == 12
    assert sm["committed_tokens"] == int(trace["resp_len"].sum())
    assert sm["latency_ms"]["mean"] > 0 and sm["steps"] > 0
