"""GPU parity of dllm_moe_ffn against the MoE oracle.

Routing: the device's expert sets equal the oracle's wherever the k-th and
(k+1)-th logits are further apart than fp32 rounding of the logit sums can
move them; weights within 1e-4. Outputs: compared with the oracle evaluated
on the device's own routing (so a near-tie routing flip cannot hide an
arithmetic error), norm-wise per row within 1e-2 (the expert activations
between the two GEMMs are bf16).
"""

import numpy as np
import pytest
import torch

import block_decoding_gb300 as bd
from helpers import dev_bf16, rownorm_rel
from oracle import moe
from workloads import MOE_CONFIGS, bf16_bits_to_f64, make_moe_inputs

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

MOE_TOL = 1e-2
W_TOL = 1e-4
GAP_REL = 1e-4


def _run(inp, out_fp32=True):
    g = {k: dev_bf16(inp[k]) for k in ("h", "w_router", "w13", "w2")}
    out, ids, w = bd.moe_ffn(g["h"], g["w_router"], g["w13"], g["w2"], inp["topk"], out_fp32=out_fp32)
    torch.cuda.synchronize()
    assert bd.device_status() == 0
    return out.float().cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def _check_routing(inp, ids, w, rows=None):
    h = bf16_bits_to_f64(inp["h"] if rows is None else inp["h"][rows])
    ref_ids, ref_w, z = moe.route(h, bf16_bits_to_f64(inp["w_router"]), inp["topk"])
    if rows is not None:
        ids, w = ids[rows], w[rows]
    gap, sc = moe.topk_gap(z, inp["topk"])
    clear = gap >= GAP_REL * sc
    for t in np.flatnonzero(clear):
        assert sorted(ids[t]) == sorted(ref_ids[t]), t
        got = dict(zip(ids[t].tolist(), w[t].tolist()))
        for e, x in zip(ref_ids[t].tolist(), ref_w[t].tolist()):
            assert abs(got[e] - x) <= W_TOL, (t, e)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-5)
    assert ((ids >= 0) & (ids < inp["E"])).all()
    assert all(len(set(r)) == len(r) for r in ids.tolist())
    return int((~clear).sum())


def _oracle_rows(inp, ids, w, rows):
    """Oracle outputs of the given rows on the device's routing, converting
    each expert's weights only when a sampled row uses it."""
    F = inp["F"]
    h = bf16_bits_to_f64(inp["h"][rows])
    y = np.zeros((len(rows), inp["d"]))
    for e in sorted(set(ids[rows].ravel().tolist())):
        w13 = bf16_bits_to_f64(inp["w13"][e])
        w2 = bf16_bits_to_f64(inp["w2"][e])
        for i, t in enumerate(rows):
            for j in np.flatnonzero(ids[t] == e):
                y[i] += float(w[t, j]) * moe.expert(h[i:i + 1], w13, w2, F)[0]
    return y


CASES = [
    dict(MOE_CONFIGS["tiny"]),                              # BN 16
    dict(n=1, d=128, E=4, F=128, topk=1),                   # one token, one expert
    dict(n=33, d=256, E=6, F=256, topk=6),                  # every expert chosen
    dict(n=300, d=256, E=16, F=256, topk=4),                # BN 128, ragged token blocks
    dict(n=70, d=384, E=1, F=128, topk=1),                  # a dense FFN
    dict(n=2048, d=128, E=32, F=128, topk=8),               # 16384 assignments: two id batches per scan thread
    dict(n=61, d=128, E=256, F=128, topk=16),               # most experts and the largest top-k
]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"n{c['n']}_d{c['d']}_E{c['E']}_F{c['F']}_k{c['topk']}")
def test_moe_ffn_matches_oracle(cfg):
    inp = make_moe_inputs(seed=21, **cfg)
    out, ids, w = _run(inp)
    _check_routing(inp, ids, w)
    y, _, _ = moe.moe_ffn(bf16_bits_to_f64(inp["h"]), None, bf16_bits_to_f64(inp["w13"]),
                          bf16_bits_to_f64(inp["w2"]), cfg["topk"], ids=ids, weights=w.astype(np.float64))
    assert rownorm_rel(out, y).max() <= MOE_TOL


def test_moe_ffn_skewed_routing_and_bf16_out():
    """A zero router sends every token to experts 0..k-1 (exact ties, lowest
    index): k experts with every token (several token blocks each), the rest
    with none."""
    cfg = dict(n=90, d=256, E=12, F=128, topk=3)
    inp = make_moe_inputs(seed=22, **cfg)
    inp["w_router"] = np.zeros_like(inp["w_router"])
    out, ids, w = _run(inp, out_fp32=False)
    assert (ids == np.arange(3)).all() and np.allclose(w, 1.0 / 3)
    y, _, _ = moe.moe_ffn(bf16_bits_to_f64(inp["h"]), np.zeros((12, 256)), bf16_bits_to_f64(inp["w13"]),
                          bf16_bits_to_f64(inp["w2"]), 3)
    assert rownorm_rel(out, y).max() <= MOE_TOL


@pytest.mark.parametrize("name", ["llada_moe_window", "llada_moe_refresh"])
def test_moe_ffn_full_size_sampled_rows(name):
    """d 2048, 64 experts, top-8, width 1024: routing of every token; outputs
    of a sample of tokens against the oracle on the device's routing."""
    inp = make_moe_inputs(seed=23, **MOE_CONFIGS[name])
    out, ids, w = _run(inp)
    _check_routing(inp, ids, w)
    rows = np.random.default_rng(5).choice(inp["n"], size=6, replace=False)
    y = _oracle_rows(inp, ids, w, rows)
    assert rownorm_rel(out[rows], y).max() <= MOE_TOL
    assert np.isfinite(out).all()


def test_moe_ffn_bitwise_repeatable():
    """The expert-sorted order inside a segment follows the order in which
    the scan's atomics land and may differ from call to call; the outputs
    must not: every grouped-GEMM output row depends on its own input row
    alone, and the combine sums a token's k rows in rank order. Many
    assignments per expert (2048 tokens, top-8 of 16) make a different
    order likely."""
    inp = make_moe_inputs(seed=24, n=2048, d=256, E=16, F=256, topk=8)
    g = {k: dev_bf16(inp[k]) for k in ("h", "w_router", "w13", "w2")}
    runs = []
    for _ in range(3):
        out, ids, w = bd.moe_ffn(g["h"], g["w_router"], g["w13"], g["w2"], inp["topk"])
        torch.cuda.synchronize()
        runs.append((out.clone(), ids.clone(), w.clone()))
    assert bd.device_status() == 0
    for out, ids, w in runs[1:]:
        assert torch.equal(ids, runs[0][1]) and torch.equal(w, runs[0][2])
        assert torch.equal(out, runs[0][0])
