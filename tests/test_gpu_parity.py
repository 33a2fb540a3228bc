"""GPU parity: the CUDA path against the oracle on the same seeded inputs.

Small cases cover several tiles, ragged tails and the edge cases (single
query, no cached prefix, empty requests, blk = 1 / 64, exact argmax ties
across tiles and CTAs, the hand-worked commit cases); the full-size
workloads compare every attention row and every head row, and the commit
both against the oracle's own decisions (ambiguous ones excluded and
counted) and fed with the device's own head outputs (bit-exact, nothing
excluded).
"""

import numpy as np
import pytest
import torch

import block_decoding_gb300 as bd
import oracle
from helpers import dev, dev_bf16, host_bf16_bits, rownorm_rel
from parity import check_attention, check_commit, check_head
from runner import run_step, upload_step
from workloads import bf16_bits_to_f64, f32_to_bf16_bits, make_step_inputs, step_config

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


# --------------------------------------------------------------------------
# commit (K3) with directly drawn confidences: bit-exact
# --------------------------------------------------------------------------

def _commit_case(rng, B, blk, V, d, frac_masked=0.7):
    mask = (rng.random((B, blk)) < frac_masked).astype(np.uint8)
    tokens = np.where(mask == 1, V - 1, rng.integers(0, V - 1, (B, blk))).astype(np.int32)
    rows = [(i, j) for i in range(B) for j in range(blk) if mask[i, j]]
    rng.shuffle(rows)
    # also add rows for a few unmasked positions: they must be ignored
    extra = [(i, j) for i in range(B) for j in range(blk) if not mask[i, j]][:3]
    rows = rows + extra
    row_req = np.array([r[0] for r in rows], np.int32)
    row_pos = np.array([r[1] for r in rows], np.int32)
    R = len(rows)
    argmax = rng.integers(0, V, R).astype(np.int32)
    prev = np.full((B, blk), -1, np.int32)
    credit = np.zeros((B, blk), np.float32)
    for r, (i, j) in enumerate(rows):
        if mask[i, j]:
            prev[i, j] = argmax[r] if rng.random() < 0.6 else rng.integers(-1, V)
            credit[i, j] = rng.uniform(0, 1.5)
    conf = rng.uniform(0.3, 1.0, R).astype(np.float32)
    pe = (rng.standard_normal((R, d)) * 0.01).astype(np.float32)
    emb = rng.integers(0, 1 << 16, (V, d), dtype=np.uint16) & 0xBFFF  # finite bf16
    return dict(mask=mask, tokens=tokens, row_req=row_req, row_pos=row_pos, argmax=argmax,
                prev=prev, credit=credit, conf=conf, pe=pe, emb=emb)


@pytest.mark.parametrize("blk", [1, 7, 32, 64])
@pytest.mark.parametrize("mode", [(0, 1), (1, 1), (1, 2), (1, 64)])
def test_commit_bit_exact(blk, mode):
    rng = np.random.default_rng(100 + blk + 7 * mode[1])
    B, V, d = 6, 50, 64
    c = _commit_case(rng, B, blk, V, d)
    params = dict(tau=0.9, lam=0.7, kappa=1.5, hierarchical=mode[0], hier_levels=mode[1],
                  smoothing=1, alpha=1.0, mask_id=V - 1)
    ref = oracle.commit(c["argmax"], c["conf"], c["pe"].astype(np.float64), c["row_req"], c["row_pos"],
                        c["mask"], c["tokens"], c["credit"], c["prev"], bf16_bits_to_f64(c["emb"]), params)
    g = dict(mask=dev(c["mask"]), tokens=dev(c["tokens"]), credit=dev(c["credit"]), prev=dev(c["prev"]))
    ne, nc = bd.commit(dev(c["argmax"]), dev(c["conf"]), dev(c["pe"]), dev(c["row_req"]), dev(c["row_pos"]),
                       g["mask"], g["tokens"], g["credit"], g["prev"], dev_bf16(c["emb"]), params)
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    assert np.array_equal(g["mask"].cpu().numpy(), ref["mask"])
    assert np.array_equal(g["tokens"].cpu().numpy(), ref["tokens"])
    assert np.array_equal(g["prev"].cpu().numpy(), ref["prev"])
    assert np.array_equal(g["credit"].cpu().numpy(), ref["credit"])        # float32 bit-exact
    assert np.array_equal(nc.cpu().numpy(), ref["n_commit"])
    ne = host_bf16_bits(ne)
    committed = ref["mask"] == 0
    assert np.array_equal(ne[committed], c["emb"][ref["tokens"][committed]])
    sm = ~committed
    if sm.any():
        assert rownorm_rel(bf16_bits_to_f64(ne[sm]), ref["next_emb"][sm]).max() < 5e-3


def test_commit_reports_missing_row_without_touching_state():
    rng = np.random.default_rng(5)
    c = _commit_case(rng, 2, 8, 20, 64, frac_masked=1.0)
    keep = c["row_req"] != 1
    keep[np.flatnonzero(c["row_req"] == 1)[1:]] = True   # request 1 loses one row
    params = dict(tau=0.9, lam=0.7, kappa=1.5, hierarchical=1, hier_levels=1,
                  smoothing=0, alpha=1.0, mask_id=19)
    g = dict(mask=dev(c["mask"]), tokens=dev(c["tokens"]), credit=dev(c["credit"]), prev=dev(c["prev"]))
    bd.device_status(clear=True)
    _, nc = bd.commit(dev(c["argmax"][keep]), dev(c["conf"][keep]), None, dev(c["row_req"][keep]),
                      dev(c["row_pos"][keep]), g["mask"], g["tokens"], g["credit"], g["prev"],
                      dev_bf16(c["emb"]), params)
    torch.cuda.synchronize()
    st = bd.device_status(clear=True)
    assert st & 0x1
    assert np.array_equal(g["mask"].cpu().numpy()[1], c["mask"][1])
    assert nc.cpu().numpy()[1] == 0 and nc.cpu().numpy()[0] >= 1


def _commit_on_device(c, params, stream=None):
    g = dict(mask=dev(c["mask"]), tokens=dev(c["tokens"]), credit=dev(c["credit"]), prev=dev(c["prev"]))
    ne, nc = bd.commit(dev(c["argmax"]), dev(c["conf"]), dev(c["pe"]), dev(c["row_req"]), dev(c["row_pos"]),
                       g["mask"], g["tokens"], g["credit"], g["prev"], dev_bf16(c["emb"]), params, stream=stream)
    return g, ne, nc


def _commit_matches_oracle(c, params, g, nc):
    ref = oracle.commit(c["argmax"], c["conf"], c["pe"].astype(np.float64), c["row_req"], c["row_pos"],
                        c["mask"], c["tokens"], c["credit"], c["prev"], bf16_bits_to_f64(c["emb"]), params)
    assert np.array_equal(g["mask"].cpu().numpy(), ref["mask"])
    assert np.array_equal(g["tokens"].cpu().numpy(), ref["tokens"])
    assert np.array_equal(g["prev"].cpu().numpy(), ref["prev"])
    assert np.array_equal(g["credit"].cpu().numpy(), ref["credit"])
    assert np.array_equal(nc.cpu().numpy(), ref["n_commit"])


def test_commit_arrival_counts_over_many_calls_and_two_streams():
    """The commit's last CTA per request (found with an arrival count, one
    count slot per call in turn) writes the state: 80 calls in a row (the 32
    slots reused more than twice, with request and block counts changing
    between calls) and two calls in flight at once on two streams all match
    the oracle exactly."""
    V, d = 40, 64
    params = dict(tau=0.9, lam=0.7, kappa=1.5, hierarchical=1, hier_levels=2,
                  smoothing=1, alpha=1.0, mask_id=V - 1)
    rng = np.random.default_rng(404)
    for call in range(80):
        B, blk = [(1, 32), (3, 7), (6, 1), (2, 64)][call % 4]
        c = _commit_case(rng, B, blk, V, d)
        g, _, nc = _commit_on_device(c, params)
        torch.cuda.synchronize()
        assert bd.device_status() == 0
        _commit_matches_oracle(c, params, g, nc)
    cases = [_commit_case(rng, 5, 32, V, d), _commit_case(rng, 4, 16, V, d)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for c, st in zip(cases, streams):
        with torch.cuda.stream(st):
            outs.append(_commit_on_device(c, params, stream=st))
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    for c, (g, _, nc) in zip(cases, outs):
        _commit_matches_oracle(c, params, g, nc)


@pytest.mark.parametrize("mode", ["off", "levels1", "levels2"])
def test_commit_handworked_cases_on_device(golden, mode):
    """The four hand-worked 3-position cases (distance ties broken by p, the
    centre first, the credit path, the fallback) as four requests of one
    dllm_commit call: selections, credit bits and counts exact."""
    g = golden("commit_handworked.json")
    cases = g["cases"]
    B, blk, V, d = len(cases), 3, 12, 64
    params = dict(tau=g["params"]["tau"], lam=g["params"]["lam"], kappa=g["params"]["kappa"],
                  hierarchical=0 if mode == "off" else 1, hier_levels=2 if mode == "levels2" else 1,
                  smoothing=0, alpha=1.0, mask_id=V - 1)
    mask = np.ones((B, blk), np.uint8)
    tokens = np.full((B, blk), V - 1, np.int32)
    prev = np.array([c["prev"] for c in cases], np.int32)
    credit = np.array([c["credit"] for c in cases], np.float32)
    # rows in reverse order: the row map, not the row order, places them
    rows = [(i, j) for i in range(B) for j in range(blk)][::-1]
    row_req = np.array([r[0] for r in rows], np.int32)
    row_pos = np.array([r[1] for r in rows], np.int32)
    argmax = np.array([cases[i]["argmax"][j] for i, j in rows], np.int32)
    conf = np.array([cases[i]["p"][j] for i, j in rows], np.float32)
    emb = f32_to_bf16_bits(np.random.default_rng(1).standard_normal((V, d)).astype(np.float32))
    ref = oracle.commit(argmax, conf, None, row_req, row_pos, mask, tokens, credit, prev,
                        bf16_bits_to_f64(emb), params)
    gm = dict(mask=dev(mask), tokens=dev(tokens), credit=dev(credit), prev=dev(prev))
    ne, nc = bd.commit(dev(argmax), dev(conf), None, dev(row_req), dev(row_pos), gm["mask"], gm["tokens"],
                       gm["credit"], gm["prev"], dev_bf16(emb), params)
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    m_out, cr_out = gm["mask"].cpu().numpy(), gm["credit"].cpu().numpy()
    for i, c in enumerate(cases):
        want = c["selected"][mode]
        assert sorted(np.flatnonzero(m_out[i] == 0).tolist()) == want, (c["name"], mode)
        for j in range(blk):
            if j not in want:
                assert abs(float(cr_out[i, j]) - c["credit_after"][j]) < g["abs_tol"], (c["name"], j)
    assert np.array_equal(m_out, ref["mask"])
    assert np.array_equal(gm["tokens"].cpu().numpy(), ref["tokens"])
    assert np.array_equal(gm["prev"].cpu().numpy(), ref["prev"])
    assert np.array_equal(cr_out, ref["credit"])
    assert np.array_equal(nc.cpu().numpy(), ref["n_commit"])
    committed = ref["mask"] == 0
    assert np.array_equal(host_bf16_bits(ne)[committed], emb[ref["tokens"][committed]])


# --------------------------------------------------------------------------
# head (K2)
# --------------------------------------------------------------------------

# (32, 256, 24576) and (48, 256, 24676): 192 and 193 vocabulary tiles on
# 148-160 SMs, so the logits GEMM runs its last tiles as K halves (the
# second one with a partial tile). R >= 128 runs both GEMMs on CTA pairs
# (R = 128: 128-row blocks, two 64-row halves); (300, 320, 1100): two row
# blocks (the second CTA's half of the second one wholly past R), nine
# vocabulary tiles and three d tiles (the last pair's second CTA wholly
# past V and d).
@pytest.mark.parametrize("R,d,V", [(16, 256, 2048), (1, 64, 1), (40, 512, 5003), (130, 1024, 1000),
                                   (32, 256, 24576), (48, 256, 24676), (128, 256, 3000), (300, 320, 1100)])
def test_head_matches_oracle(R, d, V):
    inp = make_step_inputs(B=1, H=d // 64, dh=64, V=V, blk=min(64, R), P=0, n_masked=None, seed=R + V)
    rng = np.random.default_rng(R)
    hid = inp["hidden"]
    if R > hid.shape[0]:
        hid = np.concatenate([hid, hid[rng.integers(0, hid.shape[0], R - hid.shape[0])]])
    hid = hid[:R]
    ref = oracle.head_confidence(bf16_bits_to_f64(hid), bf16_bits_to_f64(inp["w_head"]),
                                 bf16_bits_to_f64(inp["emb"]))
    gap, sc = oracle.step.top2_gap(ref["z"])
    amb = gap < oracle.step.ARGMAX_GAP_REL * sc
    a, c, pe = bd.head_confidence(dev_bf16(hid), dev_bf16(inp["w_head"]), dev_bf16(inp["emb"]))
    torch.cuda.synchronize()
    check_head(a.cpu().numpy(), c.cpu().numpy(), pe.cpu().numpy(), ref, amb_rows=amb)


@pytest.mark.parametrize("R", [40, 130, 300])
def test_head_exact_ties_take_the_lowest_index(R):
    """W_head rows duplicated exactly: the duplicate logits are equal bit for
    bit on the device, in the same 32-row vocabulary quarter, another
    quarter of the same 128-row tile, another tile (another CTA) and far
    apart (another statistics chunk). The argmax must be the lower index
    whatever the order in which tiles, CTAs and chunks merge; R = 40 takes
    the separate statistics pass, R = 130 and 300 the statistics fused into
    the logits GEMM on CTA pairs (300: two row blocks). The regular parity check excludes such rows (top-2 gap 0)."""
    d, V = 256, 5003
    rng = np.random.default_rng(R)
    w = (rng.standard_normal((V, d)) / np.sqrt(d)).astype(np.float32)
    pairs = [(64 + 3, 64 + 8), (640 + 10, 640 + 50), (1300, 1600), (200, 2900), (4990, 30)]
    for lo, hi in pairs:
        w[hi] = w[lo]
    w_bits = f32_to_bf16_bits(w)
    wf = bf16_bits_to_f64(w_bits)
    k = np.arange(R) % len(pairs)
    tok = np.array([pairs[i][r % 2] for r, i in enumerate(k)])      # plant either copy
    want = np.array([min(pairs[i]) for i in k], np.int32)
    hid = 0.05 * rng.standard_normal((R, d)) + 8.0 * wf[tok] / np.linalg.norm(wf[tok], axis=1)[:, None]
    hid_bits = f32_to_bf16_bits(hid.astype(np.float32))
    emb = f32_to_bf16_bits((0.02 * rng.standard_normal((V, d))).astype(np.float32))
    ref = oracle.head_confidence(bf16_bits_to_f64(hid_bits), wf, bf16_bits_to_f64(emb))
    gap, _ = oracle.step.top2_gap(ref["z"])
    assert (gap < 1e-9).all()                         # the exact tie is the row's top 2
    a, c, pe = bd.head_confidence(dev_bf16(hid_bits), dev_bf16(w_bits), dev_bf16(emb))
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    assert np.array_equal(a.cpu().numpy(), want)
    assert np.abs(c.cpu().numpy() - ref["conf"]).max() <= 2e-3
    assert rownorm_rel(pe.cpu().numpy(), ref["pe"]).max() <= 1e-2


# --------------------------------------------------------------------------
# attention (K1)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dh", [64, 128])
def test_attention_ragged(dh):
    inp = make_step_inputs(B=5, H=3, dh=dh, V=64, blk=8, P=[0, 5, 300, 1000, 77],
                           vl=[0, 3, 16, 32, 0], vr=[0, 1, 16, 0, 120], seed=dh)
    ref = oracle.block_attention(bf16_bits_to_f64(inp["q"]), bf16_bits_to_f64(inp["k"]),
                                 bf16_bits_to_f64(inp["v"]), inp["q_off"], inp["kv_off"], inp["scale"])
    o = bd.block_attn(dev_bf16(inp["q"]), dev_bf16(inp["k"]), dev_bf16(inp["v"]), dev(inp["q_off"]),
                      dev(inp["kv_off"]), inp["max_q"], inp["max_kv"], inp["scale"], out_fp32=True)
    torch.cuda.synchronize()
    check_attention(o.cpu().numpy(), ref)
    ob = bd.block_attn(dev_bf16(inp["q"]), dev_bf16(inp["k"]), dev_bf16(inp["v"]), dev(inp["q_off"]),
                       dev(inp["kv_off"]), inp["max_q"], inp["max_kv"], inp["scale"])
    torch.cuda.synchronize()
    check_attention(ob.float().cpu().numpy(), ref)


@pytest.mark.parametrize("dh", [64, 128])
def test_attention_two_query_tiles_and_many_splits(dh):
    # request 0: W = 196 (two 128-row query tiles), L = 3196 (25 key tiles,
    # so the work is split across many CTAs and merged by the combine pass)
    inp = make_step_inputs(B=2, H=2, dh=dh, V=64, blk=32, P=[3000, 10], vl=[64, 0], vr=[100, 0], seed=7)
    ref = oracle.block_attention(bf16_bits_to_f64(inp["q"]), bf16_bits_to_f64(inp["k"]),
                                 bf16_bits_to_f64(inp["v"]), inp["q_off"], inp["kv_off"], inp["scale"])
    o = bd.block_attn(dev_bf16(inp["q"]), dev_bf16(inp["k"]), dev_bf16(inp["v"]), dev(inp["q_off"]),
                      dev(inp["kv_off"]), inp["max_q"], inp["max_kv"], inp["scale"], out_fp32=True)
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    check_attention(o.cpu().numpy(), ref)


@pytest.mark.parametrize("dh", [64, 128])
def test_attention_rising_scores_move_the_reference_max(dh):
    """Key norms growing 13-fold along the sequence, plus one late spike: a
    row's running max rises by far more than 2^8 over the key tiles, so the
    reference max moves (and O is rescaled) many times, in every key split."""
    from workloads import f32_to_bf16_bits
    inp = make_step_inputs(B=2, H=2, dh=dh, V=64, blk=32, P=[3000, 10], vl=[64, 0], vr=[100, 0], seed=11)
    k = bf16_bits_to_f64(inp["k"])
    rows = k.shape[0]
    k = k * (1.0 + 12.0 * np.arange(rows) / rows)[:, None, None]
    k[rows - 150] *= 3.0
    inp["k"] = f32_to_bf16_bits(k.astype(np.float32))
    ref = oracle.block_attention(bf16_bits_to_f64(inp["q"]), bf16_bits_to_f64(inp["k"]),
                                 bf16_bits_to_f64(inp["v"]), inp["q_off"], inp["kv_off"], inp["scale"])
    o = bd.block_attn(dev_bf16(inp["q"]), dev_bf16(inp["k"]), dev_bf16(inp["v"]), dev(inp["q_off"]),
                      dev(inp["kv_off"]), inp["max_q"], inp["max_kv"], inp["scale"], out_fp32=True)
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    check_attention(o.cpu().numpy(), ref)


def test_attention_offsets_beyond_buffers_are_clipped():
    inp = make_step_inputs(B=1, H=2, dh=64, V=64, blk=16, P=40, seed=8)
    kv_off = inp["kv_off"].copy()
    kv_off[1] += 1000                       # claims 1000 rows that are not there
    rows = int(inp["kv_off"][1])
    ref = oracle.block_attention(bf16_bits_to_f64(inp["q"]), bf16_bits_to_f64(inp["k"]),
                                 bf16_bits_to_f64(inp["v"]), inp["q_off"], inp["kv_off"], inp["scale"])
    bd.device_status(clear=True)
    o = bd.block_attn(dev_bf16(inp["q"]), dev_bf16(inp["k"][:rows]), dev_bf16(inp["v"][:rows]),
                      dev(inp["q_off"]), dev(kv_off), inp["max_q"], rows + 1000, inp["scale"], out_fp32=True)
    torch.cuda.synchronize()
    assert bd.device_status(clear=True) & 0x20
    check_attention(o.cpu().numpy(), ref)


def test_attention_empty_and_single():
    # request 0: one query, one key; request 1: no queries; request 2: queries, keys
    H, dh = 2, 64
    q_off = np.array([0, 1, 1, 4], np.int32)
    kv_off = np.array([0, 1, 5, 9], np.int32)
    rng = np.random.default_rng(9)
    from workloads import f32_to_bf16_bits
    q = f32_to_bf16_bits(rng.standard_normal((4, H, dh)).astype(np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((9, H, dh)).astype(np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((9, H, dh)).astype(np.float32))
    ref = oracle.block_attention(bf16_bits_to_f64(q), bf16_bits_to_f64(k), bf16_bits_to_f64(v),
                                 q_off, kv_off, 0.125)
    o = bd.block_attn(dev_bf16(q), dev_bf16(k), dev_bf16(v), dev(q_off), dev(kv_off), 3, 4, 0.125,
                      out_fp32=True)
    torch.cuda.synchronize()
    check_attention(o.cpu().numpy(), ref)
    np.testing.assert_allclose(o.cpu().numpy()[0], bf16_bits_to_f64(v)[0], rtol=1e-6)


# --------------------------------------------------------------------------
# whole step on the small workloads
# --------------------------------------------------------------------------

@pytest.mark.parametrize("cal", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_step_tiny(cal, seed):
    inp = step_config("tiny", seed=seed, cal=cal)
    ref = oracle.denoise_step(inp)
    out = run_step(inp)
    check_attention(out["attn"], ref["attn"])
    amb = ref["ambiguity"]
    check_head(out["argmax"], out["conf"], out["pe"], ref["head"], amb_rows=amb["argmax_row"])
    check_commit(inp, out, ref["commit"], amb, inp["emb"], pe_ref=ref["head"]["pe"])


def test_step_mid_batched_hierarchy_off():
    inp = make_step_inputs(B=4, H=4, dh=128, V=3001, blk=32, P=[40, 0, 333, 129], vl=8, vr=8,
                           n_masked=20, cal=True, seed=3, hierarchical=0)
    ref = oracle.denoise_step(inp)
    out = run_step(inp)
    check_attention(out["attn"], ref["attn"])
    check_head(out["argmax"], out["conf"], out["pe"], ref["head"], amb_rows=ref["ambiguity"]["argmax_row"])
    check_commit(inp, out, ref["commit"], ref["ambiguity"], inp["emb"], pe_ref=ref["head"]["pe"])


# --------------------------------------------------------------------------
# full-size workloads
# --------------------------------------------------------------------------

def _teacher_forced_commit(inp, out):
    """Oracle commit fed with the device's own head outputs: bit-exact."""
    ref = oracle.commit(out["argmax"], out["conf"], out["pe"].astype(np.float64), inp["row_req"],
                        inp["row_pos"], inp["mask"], inp["tokens"], inp["credit"], inp["prev"],
                        bf16_bits_to_f64(inp["emb"]), inp["params"])
    assert np.array_equal(out["mask"], ref["mask"])
    assert np.array_equal(out["tokens"], ref["tokens"])
    assert np.array_equal(out["prev"], ref["prev"])
    assert np.array_equal(out["credit"], ref["credit"])
    assert np.array_equal(out["n_commit"], ref["n_commit"])
    com = ref["mask"] == 0
    assert np.array_equal(out["next_emb_bits"][com], inp["emb"][ref["tokens"][com]])
    if (~com).any():
        assert rownorm_rel(bf16_bits_to_f64(out["next_emb_bits"][~com]), ref["next_emb"][~com]).max() < 5e-3
    return ref


@pytest.mark.slow
@pytest.mark.parametrize("name,cal", [("llada8b_b1", False), ("llada8b_b1", True), ("llada8b_b16", False),
                                      ("llada8b_b16", True), ("longctx_8k", True)])
def test_step_full_size(name, cal):
    """Every attention row and every head row against the oracle, then the
    commit twice: against the oracle's own decisions under its ambiguity
    record, and replayed from the device's head outputs (bit-exact)."""
    inp = step_config(name, cal=cal)
    out = run_step(inp)
    ref = oracle.denoise_step(inp)
    check_attention(out["attn"], ref["attn"])
    amb = ref["ambiguity"]
    check_head(out["argmax"], out["conf"], out["pe"], ref["head"], amb_rows=amb["argmax_row"])
    info = check_commit(inp, out, ref["commit"], amb, inp["emb"], pe_ref=ref["head"]["pe"])
    print(f"{name}{'_cal' if cal else ''}: {info}, ambiguity counts {amb['counts']}")
    _teacher_forced_commit(inp, out)
