"""GPU parity of the end-to-end pieces: bf16 GEMM epilogues, the layer stack
with its prefix cache, and the block decode loop, against the oracle.

Activations are bf16 between kernels on the device and float64 in the
oracle, so hidden rows are compared norm-wise within E2E_TOL; decisions are
compared teacher-forced: every recorded device step is recomputed by the
oracle from the device's own state before that step, and the commit of the
step is replayed bit-exactly from the device's head outputs. One test runs
both loops free-running on the full end-to-end configuration and reports
the first step at which they differ.
"""

import numpy as np
import pytest
import torch

import block_decoding_gb300 as bd
import oracle
from helpers import dev, dev_bf16, host_bf16_bits, rownorm_rel
from oracle import model as om
from workloads import bf16_bits_to_f64, f32_to_bf16_bits, make_e2e_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

GEMM_TOL = 1e-2    # bf16 output rounding of an fp32-accumulated product
E2E_TOL = 3e-2     # hidden rows after several layers of bf16 activations
SMALL = dict(layers=2, d=256, H=4, dh=64, ffn=512, V=512, prompt_len=32, resp_len=64, blk=32, vic=16)


def _bf16(rng, shape, std=1.0):
    return f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))


@pytest.mark.parametrize("M,N,K", [(1, 1024, 1024), (17, 3072, 1024), (96, 1024, 4096), (300, 256, 512),
                                   (512, 1024, 1024)])
def test_gemm_plain_and_residual(M, N, K):
    rng = np.random.default_rng(M + N)
    A, W, R = _bf16(rng, (M, K)), _bf16(rng, (N, K), 0.02), _bf16(rng, (M, N))
    ref = bf16_bits_to_f64(A) @ bf16_bits_to_f64(W).T
    C = bd.gemm_bf16(dev_bf16(A), dev_bf16(W))
    torch.cuda.synchronize()
    assert rownorm_rel(bf16_bits_to_f64(host_bf16_bits(C)), ref).max() <= GEMM_TOL
    Rt = dev_bf16(R)
    bd.gemm_bf16(dev_bf16(A), dev_bf16(W), epilogue=1, aux=Rt, out=Rt)    # in place: x += A W^T
    torch.cuda.synchronize()
    assert rownorm_rel(bf16_bits_to_f64(host_bf16_bits(Rt)), ref + bf16_bits_to_f64(R)).max() <= GEMM_TOL
    assert bd.device_status() == 0


@pytest.mark.parametrize("M,F,K", [(5, 128, 256), (96, 4096, 1024), (512, 512, 1024)])
def test_gemm_swiglu(M, F, K):
    rng = np.random.default_rng(M + F)
    A, W = _bf16(rng, (M, K)), _bf16(rng, (2 * F, K), 0.05)
    g = bf16_bits_to_f64(A) @ bf16_bits_to_f64(W[:F]).T
    u = bf16_bits_to_f64(A) @ bf16_bits_to_f64(W[F:]).T
    ref = om.silu(g) * u
    C = bd.gemm_bf16(dev_bf16(A), dev_bf16(W), epilogue=2)
    torch.cuda.synchronize()
    assert C.shape == (M, F)
    assert rownorm_rel(bf16_bits_to_f64(host_bf16_bits(C)), ref).max() <= GEMM_TOL


def _weights(inp):
    return dict(emb=dev_bf16(inp["emb"]), w_head=dev_bf16(inp["w_head"]), H=inp["H"], rms_eps=inp["rms_eps"],
                rope_base=inp["rope_base"],
                wqkv=[dev_bf16(l["wqkv"]) for l in inp["layer_weights"]],
                wo=[dev_bf16(l["wo"]) for l in inp["layer_weights"]],
                wgu=[dev_bf16(l["wgu"]) for l in inp["layer_weights"]],
                wdown=[dev_bf16(l["wdown"]) for l in inp["layer_weights"]])


def test_model_forward_full_then_cached_window():
    inp = make_e2e_inputs(seed=3, **SMALL)
    T, d = 96, inp["d"]
    rng = np.random.default_rng(4)
    x = inp["emb"][rng.integers(0, inp["V"], T)]
    m = om.Model(inp)
    full_ref, kv = m.forward(bf16_bits_to_f64(x), np.arange(T))
    w = _weights(inp)
    desc, keep = bd.model_desc(w, T)
    kc = [torch.zeros((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(inp["layers"])]
    vc = [torch.zeros((T, d), dtype=torch.bfloat16, device="cuda") for _ in range(inp["layers"])]
    out = bd.model_forward(desc, dev_bf16(x), 0, kc, vc)
    torch.cuda.synchronize()
    assert rownorm_rel(bf16_bits_to_f64(host_bf16_bits(out)), full_ref).max() <= E2E_TOL
    # window [60, 96) over the cached rows [0, 60): the oracle uses its own
    # cache of the same rows, the device its bf16 cache
    ws = 60
    cache = [(k[:ws], v[:ws]) for (k, v) in kv]
    win_ref, _ = m.forward(bf16_bits_to_f64(x[ws:]), np.arange(ws, T), cache)
    out = bd.model_forward(desc, dev_bf16(x[ws:]), ws, kc, vc)
    torch.cuda.synchronize()
    assert rownorm_rel(bf16_bits_to_f64(host_bf16_bits(out)), win_ref).max() <= E2E_TOL
    assert bd.device_status() == 0


def _run_teacher_forced(inp, check_steps=None):
    """Decode on the device; recompute recorded steps with the oracle."""
    w = _weights(inp)
    dec = bd.BlockDecoder(w, torch.from_numpy(inp["prompt"]), resp_len=inp["resp_len"], blk=inp["blk"],
                          vic=inp["vic"], params=inp["params"], dual_cache=bool(inp["dual_cache"]))
    rec = []
    snap = {}

    def on_step(when, b, s, dd):
        if check_steps is not None and (b, s) not in check_steps:
            return
        cpu = lambda t: t.cpu().numpy()  # noqa: E731
        if when == "before":
            snap.update(tokens=cpu(dd.tokens), masked=cpu(dd.masked).astype(bool), bmask=cpu(dd.bmask),
                        btokens=cpu(dd.btokens), bcredit=cpu(dd.bcredit), bprev=cpu(dd.bprev),
                        bnext=host_bf16_bits(dd.bnext_emb))
        else:
            rec.append(dict(b=b, s=s, before=dict(snap), hidden=host_bf16_bits(dd.hidden), argmax=cpu(dd.argmax),
                            conf=cpu(dd.conf), pe=cpu(dd.pe), n=int(cpu(dd.n_commit)[0]), bmask=cpu(dd.bmask),
                            btokens=cpu(dd.btokens), bcredit=cpu(dd.bcredit), bprev=cpu(dd.bprev),
                            bnext=host_bf16_bits(dd.bnext_emb)))

    steps = dec.decode(on_step=on_step)
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    tokens, masked = dec.tokens.cpu().numpy(), dec.masked.cpu().numpy()
    return steps, tokens, masked, rec


def _check_records(inp, rec):
    m = om.Model(inp)
    prm = inp["params"]
    emb64 = m.emb
    caches = {}
    stats = dict(steps=0, argmax_cmp=0, argmax_excluded=0)
    for r in rec:
        b, s, bef = r["b"], r["s"], r["before"]
        block_emb = bf16_bits_to_f64(bef["bnext"]) if s > 0 else None
        if s == 0 or b not in caches:
            assert s == 0, "the window steps of a block need its refresh recorded"
            hb, caches[b] = om.forward_step(m, inp, bef["tokens"], bef["masked"], None, b, True, None)
        else:
            hb, _ = om.forward_step(m, inp, bef["tokens"], bef["masked"], block_emb, b, False, caches[b])
        # hidden rows of the block
        assert rownorm_rel(bf16_bits_to_f64(r["hidden"]), hb).max() <= E2E_TOL, (b, s)
        # head on the device's own hidden rows: argmax exact where the top-2 gap is clear
        head = oracle.head_confidence(bf16_bits_to_f64(r["hidden"]), m.w_head, emb64)
        gap, sc = oracle.step.top2_gap(head["z"])
        clear = gap >= oracle.step.ARGMAX_GAP_REL * sc
        assert np.array_equal(r["argmax"][clear], head["argmax"][clear]), (b, s)
        assert np.abs(r["conf"] - head["conf"]).max() <= 2e-3
        assert rownorm_rel(r["pe"], head["pe"]).max() <= 1e-2
        stats["argmax_cmp"] += int(clear.sum())
        stats["argmax_excluded"] += int((~clear).sum())
        # commit replayed from the device's head outputs: bit-exact
        blk = inp["blk"]
        com = oracle.commit(r["argmax"], r["conf"], r["pe"].astype(np.float64), np.zeros(blk, np.int32),
                            np.arange(blk, dtype=np.int32), bef["bmask"][None], bef["btokens"][None],
                            bef["bcredit"][None], bef["bprev"][None], emb64, prm)
        assert np.array_equal(r["bmask"], com["mask"][0]) and np.array_equal(r["btokens"], com["tokens"][0])
        assert np.array_equal(r["bcredit"], com["credit"][0]) and np.array_equal(r["bprev"], com["prev"][0])
        assert r["n"] == int(com["n_commit"][0]) >= 1
        stats["steps"] += 1
    return stats


@pytest.mark.parametrize("dual", [1, 0])
def test_decode_small_model_teacher_forced(dual):
    inp = make_e2e_inputs(seed=11, dual_cache=dual, **SMALL)
    steps, tokens, masked, rec = _run_teacher_forced(inp)
    assert not masked.any() and np.array_equal(tokens[:inp["prompt_len"]], inp["prompt"])
    assert steps == [inp["blk"]] * (inp["resp_len"] // inp["blk"])     # random weights: fallback only
    stats = _check_records(inp, rec)
    assert stats["steps"] == sum(steps)


def test_decode_small_model_zero_threshold_hierarchical():
    inp = make_e2e_inputs(seed=12, tau=0.0, **SMALL)
    steps, tokens, masked, rec = _run_teacher_forced(inp)
    assert not masked.any()
    assert steps == [6, 6]                          # ceil(log2(32 + 1)): centre-first bisection
    _check_records(inp, rec)


def test_decode_small_model_dual_cache_teacher_forced():
    """Window steps over prefix + window + suffix cache (block 0's window
    [16, 80) leaves a suffix [80, 96); block 1's reaches the end)."""
    inp = make_e2e_inputs(seed=15, dual_cache=1, **SMALL)
    steps, tokens, masked, rec = _run_teacher_forced(inp, check_steps={(0, 0), (0, 1), (0, 2), (1, 0), (1, 1)})
    assert not masked.any()
    _check_records(inp, rec)
    # every row of block 0's first window step is nearer the oracle with the
    # suffix cache than the oracle without it (those are about 5 % apart)
    m = om.Model(inp)
    st = {(r["b"], r["s"]): r for r in rec}
    r0, r1 = st[(0, 0)]["before"], st[(0, 1)]["before"]
    ref = {}
    for dual in (0, 1):
        cfg = dict(inp, dual_cache=dual)
        _, cache = om.forward_step(m, cfg, r0["tokens"], r0["masked"], None, 0, True, None)
        ref[dual], _ = om.forward_step(m, cfg, r1["tokens"], r1["masked"], bf16_bits_to_f64(r1["bnext"]), 0, False,
                                       cache)
    got = bf16_bits_to_f64(st[(0, 1)]["hidden"])
    assert (rownorm_rel(got, ref[1]) < rownorm_rel(got, ref[0])).all()


@pytest.mark.slow
def test_decode_end_to_end_config():
    """The 4-layer d=1024 model, 256 prompt + 8 blocks of 32, vicinity 32."""
    inp = make_e2e_inputs(seed=0)
    check = {(0, 0), (0, 1), (0, 2), (3, 0), (3, 7), (7, 0), (7, 30), (7, 31)}
    steps, tokens, masked, rec = _run_teacher_forced(inp, check_steps=check)
    assert not masked.any() and np.array_equal(tokens[:256], inp["prompt"])
    assert steps == [32] * 8
    # block caches of the checked window steps come from their refresh steps
    _check_records(inp, [r for r in rec if (r["b"], 0) in check])


@pytest.mark.slow
def test_decode_end_to_end_first_divergence():
    """Config 4, both loops free-running: the device's host-driven loop and
    the oracle's own loop (no teacher forcing) over block 0. Reports the
    first step at which their decisions differ; every earlier step must
    agree exactly, and the first difference must be one that the device's
    bf16 activations can flip: a commit of the same position with another
    token whose top-2 logit gap lies inside the band, or, when a step falls
    back to its single most confident position, a swap of two positions
    whose confidences (oracle) differ by less than the device's own error
    on them at that step."""
    inp = make_e2e_inputs(seed=0)
    w = _weights(inp)
    dec = bd.BlockDecoder(w, torch.from_numpy(inp["prompt"]), resp_len=inp["resp_len"], blk=inp["blk"],
                          vic=inp["vic"], params=inp["params"], dual_cache=bool(inp["dual_cache"]))
    dev_steps, snap = [], {}

    def on_step(when, b, s, dd):
        if when == "before":
            snap["mask"] = dd.bmask.cpu().numpy().astype(bool)
        else:
            after = dd.bmask.cpu().numpy().astype(bool)
            dev_steps.append(dict(sel=snap["mask"] & ~after, tokens=dd.btokens.cpu().numpy().copy(),
                                  conf=dd.conf.cpu().numpy().copy()))

    dec.decode(on_step=on_step, max_blocks=1)
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    ref = om.decode(inp, max_blocks=1, record=True)
    first = None
    for k, st in enumerate(ref["steps"]):
        sel_o, tok_o = st["commit"]["selected"][0], st["commit"]["tokens"][0]
        d = dev_steps[k]
        if not (np.array_equal(sel_o, d["sel"]) and np.array_equal(tok_o[sel_o], d["tokens"][sel_o])):
            first = k
            break
    n = len(ref["steps"])
    print(f"config 4, block 0: device and oracle loops agree on "
          f"{n if first is None else first} of {n} steps" + ("" if first is None else f"; first difference at step {first}"))
    if first is None:
        assert len(dev_steps) == n
        return
    st, d = ref["steps"][first], dev_steps[first]
    sel_o = st["commit"]["selected"][0]
    z, conf_o = st["head"]["z"], st["head"]["conf"]
    gap, _ = oracle.step.top2_gap(z)
    rel = gap / z.std(axis=1)
    explained = False
    same = sel_o & d["sel"]
    for j in np.flatnonzero(same):
        if st["commit"]["tokens"][0, j] != d["tokens"][j]:
            explained |= bool(rel[j] < E2E_GAP_BAND)
    only_o, only_d = np.flatnonzero(sel_o & ~d["sel"]), np.flatnonzero(d["sel"] & ~sel_o)
    for a in only_o:
        for b in only_d:
            margin = abs(conf_o[a] - conf_o[b])
            err = abs(d["conf"][a] - conf_o[a]) + abs(d["conf"][b] - conf_o[b])
            explained |= bool(margin <= err)
    print(f"  step {first}: oracle commits {np.flatnonzero(sel_o).tolist()}, device {np.flatnonzero(d['sel']).tolist()}")
    assert explained, "the first difference is not one that bf16 activations can flip"


def _decoder(inp, eos_id=-1):
    return bd.BlockDecoder(_weights(inp), torch.from_numpy(inp["prompt"]), resp_len=inp["resp_len"],
                           blk=inp["blk"], vic=inp["vic"], params=inp["params"], eos_id=eos_id)


def test_decode_graph_matches_host_loop_twice():
    """The device-side loop (one CUDA graph, no host read per step) commits
    exactly the tokens of the host-driven loop: same kernels, same order."""
    inp = make_e2e_inputs(seed=13, **SMALL)
    dec = _decoder(inp)
    steps = dec.decode()
    host_tokens = dec.tokens.cpu().numpy().copy()
    assert not dec.masked.cpu().numpy().any() and steps == [32, 32]
    for _ in range(2):
        dec.restart()
        dec.decode_graph()
        torch.cuda.synchronize()
        assert bd.device_status() == 0
        assert not dec.masked.cpu().numpy().any()
        assert np.array_equal(dec.tokens.cpu().numpy(), host_tokens)


def test_decode_graph_stops_after_eos():
    inp = make_e2e_inputs(seed=14, **SMALL)
    ref = _decoder(inp)
    ref.decode()
    toks = ref.tokens.cpu().numpy()
    Lp, blk = inp["prompt_len"], inp["blk"]
    eos = int(toks[Lp + 3])                       # a token block 0 commits
    later = toks[Lp + blk:]
    dec = _decoder(inp, eos_id=eos)
    dec.decode_graph()
    torch.cuda.synchronize()
    got_t, got_m = dec.tokens.cpu().numpy(), dec.masked.cpu().numpy()
    assert not got_m[Lp:Lp + blk].any()           # block 0 decoded as before
    assert np.array_equal(got_t[:Lp + blk], toks[:Lp + blk])
    if eos not in later:                          # block 1 would not have produced it anyway
        assert got_m[Lp + blk:].all()             # skipped: still masked
    host = _decoder(inp, eos_id=eos)
    host.decode()
    assert np.array_equal(host.masked.cpu().numpy(), got_m)
    assert np.array_equal(host.tokens.cpu().numpy(), got_t)


# --------------------------------------------------------------------------
# the device-side decode loop (one CUDA graph) against the oracle's loop
# --------------------------------------------------------------------------

# A decision is compared when its top-2 logit gap is at least this fraction
# of the row's logit standard deviation. The device rounds every activation
# to bf16 between kernels; for this model (weights N(0, 0.08^2)) a forward
# with every intermediate rounded so moves a top-2 gap by at most ~0.06
# standard deviations (median ~0.012), so the band keeps each compared
# decision about four such worst cases away from a flip.
E2E_GAP_BAND = 0.25
GRAPH_MODEL = dict(SMALL, resp_len=96, w_std=0.08)      # three blocks of 32
GRAPH_SEED = 27


def _graph_vs_oracle(inp, eos_id=-1):
    """Decode with the device graph, then replay the oracle's loop teacher-
    forced on the device's tokens: every oracle decision with a clear
    margin must be the device's token; the final mask must be the oracle's."""
    dec = _decoder(inp, eos_id=eos_id)
    dec.decode_graph()
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    tokens, masked = dec.tokens.cpu().numpy(), dec.masked.cpu().numpy().astype(bool)
    ref = om.decode(inp, record=True, eos_id=eos_id, teacher=tokens)
    assert np.array_equal(masked, ref["masked"])
    assert np.array_equal(tokens[ref["masked"]], np.full(int(ref["masked"].sum()), inp["params"]["mask_id"]))
    Lp, blk = inp["prompt_len"], inp["blk"]
    compared, excluded, bad = 0, 0, []
    for st in ref["steps"]:
        # tau = 0: every masked position is a candidate, so the positions a
        # step commits follow from the mask alone, on both sides
        assert np.array_equal(st["commit"]["cand"][0], st["state_in"]["mask"][0].astype(bool))
        z = st["head"]["z"]
        gap, _ = oracle.step.top2_gap(z)
        rel = gap / z.std(axis=1)
        b0 = Lp + st["block"] * blk
        for j in np.flatnonzero(st["commit"]["selected"][0]):
            if rel[j] < E2E_GAP_BAND:
                excluded += 1
            elif tokens[b0 + j] != st["commit"]["tokens"][0, j]:
                bad.append((st["block"], st["step"], int(j), float(rel[j])))
            else:
                compared += 1
    assert not bad, f"device tokens differ from clear oracle decisions (block, step, pos, gap/std): {bad[:10]}"
    print(f"decode graph vs oracle: {compared} decisions compared, {excluded} within the gap band")
    return compared, excluded, ref


def test_decode_graph_matches_the_oracle_loop():
    inp = make_e2e_inputs(seed=GRAPH_SEED, tau=0.0, **GRAPH_MODEL)
    compared, excluded, ref = _graph_vs_oracle(inp)
    assert not ref["masked"].any()
    assert compared + excluded == inp["resp_len"]
    assert excluded <= 0.5 * inp["resp_len"]
    # centre-first bisection: each block of 32 fills in ceil(log2(33)) steps
    assert len(ref["steps"]) == 3 * 6


def test_decode_graph_eos_matches_the_oracle_loop():
    """Early stop after EOS: the block that commits it finishes; the later
    blocks are skipped and stay masked, as in the oracle's loop."""
    inp = make_e2e_inputs(seed=GRAPH_SEED, tau=0.0, **GRAPH_MODEL)
    Lp, blk = inp["prompt_len"], inp["blk"]
    free = _decoder(inp)
    free.decode_graph()
    torch.cuda.synchronize()
    eos = int(free.tokens.cpu().numpy()[Lp + 15])      # block 0's first commit (its centre)
    compared, excluded, ref = _graph_vs_oracle(inp, eos_id=eos)
    assert not ref["masked"][:Lp + blk].any() and ref["masked"][Lp + blk:].all()
    assert {st["block"] for st in ref["steps"]} == {0}
    assert compared + excluded == blk
