"""Parity rules between the CUDA path and the oracle (test infrastructure).

Floating-point outputs: attention O and P.E within 1e-2 norm-wise relative
error per row (||x - y|| / ||y||; elementwise relative error is
ill-conditioned for P.E, a near-cancelling sum), confidence within 2e-3
absolute. Integer outputs (argmax, committed sets, tokens, mask, prev) are
bit-exact except where the oracle's ambiguity record says the two sides may
legitimately decide differently; those are counted, printed and returned,
and at most MAX_EXCLUDED_FRAC of the decisions (rounded down) may be
excluded, so that a widened exclusion rule cannot hide a wrong result.
"""

import numpy as np

from helpers import rownorm_rel
from workloads import bf16_bits_to_f64

ATTN_TOL = 1e-2
PE_TOL = 1e-2
CONF_TOL = 2e-3
CREDIT_TOL = 2e-3 * 4  # credit <- lambda*credit + p accumulates the conf error
MAX_EXCLUDED_FRAC = 0.05


def _bound_excluded(what, n_excluded, n_total):
    limit = int(MAX_EXCLUDED_FRAC * n_total)
    print(f"{what}: {n_excluded} of {n_total} excluded as ambiguous (limit {limit})")
    assert n_excluded <= limit, f"{what}: {n_excluded} of {n_total} excluded > {limit}"


def check_attention(o_gpu, o_ref, tol=ATTN_TOL):
    err = rownorm_rel(o_gpu, o_ref)
    assert err.max() <= tol, f"attention rel err {err.max():.3e} > {tol}"
    return float(err.max())


def check_head(argmax, conf, pe, head_ref, rows=None, amb_rows=None):
    """argmax exact outside ambiguous rows; conf abs; pe norm-wise."""
    ref_a = head_ref["argmax"] if rows is None else head_ref["argmax"][rows]
    ref_c = head_ref["conf"] if rows is None else head_ref["conf"][rows]
    ok = np.ones(len(ref_a), bool) if amb_rows is None else ~amb_rows
    bad = np.flatnonzero((np.asarray(argmax) != ref_a) & ok)
    assert bad.size == 0, f"argmax differs at rows {bad[:10]}"
    cerr = np.abs(np.asarray(conf, np.float64) - ref_c)
    assert cerr.max() <= CONF_TOL, f"conf err {cerr.max():.3e}"
    out = dict(conf_err=float(cerr.max()), argmax_excluded=int((~ok).sum()))
    _bound_excluded("argmax rows", out["argmax_excluded"], len(ref_a))
    if pe is not None:
        ref_pe = head_ref["pe"] if rows is None else head_ref["pe"][rows]
        perr = rownorm_rel(pe, ref_pe)
        assert perr.max() <= PE_TOL, f"pe rel err {perr.max():.3e}"
        out["pe_err"] = float(perr.max())
    return out


def check_commit(inp, state_gpu, com_ref, amb, emb_bits, pe_ref=None):
    """Compare the committed state and next-step embeddings of one step.

    Per request the device's committed set must be one of the selections
    the oracle's ambiguity record allows (``choices``: exactly the oracle's
    own when nothing is ambiguous); a request the record excludes whole is
    counted, not compared. Tokens, prev and credit follow the oracle's
    per-position decision record (argmax, post-update credit), except at
    positions whose argmax is ambiguous. pe_ref (the oracle's P.E rows)
    checks the smoothed next-step rows of every position the device left
    masked; without it only those both sides left masked are checked.
    """
    mask0 = inp["mask"].astype(bool)
    B, blk = mask0.shape
    sel_gpu = mask0 & (state_gpu["mask"] == 0)
    n_choice = 0
    for i in range(B):
        if amb["request"][i]:
            continue
        got = frozenset(np.flatnonzero(sel_gpu[i]).tolist())
        ch = amb["choices"][i]
        assert got in ch, f"request {i}: committed {sorted(got)}, allowed {[sorted(c) for c in ch][:8]}"
        n_choice += int(len(ch) > 1)
    arg_ok = ~amb["argmax_pos"]
    a_ref = com_ref["a"]
    m = sel_gpu & arg_ok
    assert np.array_equal(state_gpu["tokens"][m], a_ref[m]), "tokens"
    # untouched positions stay untouched
    assert np.array_equal(state_gpu["tokens"][~mask0], inp["tokens"][~mask0])
    assert np.array_equal(state_gpu["mask"][~mask0], inp["mask"][~mask0])
    still = mask0 & ~sel_gpu & arg_ok
    assert np.array_equal(state_gpu["prev"][still], a_ref[still]), "prev"
    cr_err = np.abs(state_gpu["credit"][still].astype(np.float64) - com_ref["credit_upd"][still])
    assert cr_err.size == 0 or cr_err.max() <= CREDIT_TOL, f"credit err {cr_err.max():.3e}"
    assert (state_gpu["credit"][sel_gpu] == 0).all() and (state_gpu["prev"][sel_gpu] == -1).all()
    for i in range(B):
        assert state_gpu["n_commit"][i] == sel_gpu[i].sum() >= (1 if mask0[i].any() else 0)
    # next-step embeddings
    ne = state_gpu["next_emb_bits"]                        # [B][blk][d] uint16
    emb = emb_bits
    committed = ~mask0 | sel_gpu
    for i in range(B):
        for j in range(blk):
            if committed[i, j]:
                tok = state_gpu["tokens"][i, j]
                assert np.array_equal(ne[i, j], emb[tok]), f"next_emb row ({i},{j})"
    prm = inp["params"]
    sm = mask0 & ~sel_gpu
    if pe_ref is None:
        sm &= ~com_ref["selected"]
        want = com_ref["next_emb"][sm] if sm.any() else None
    elif sm.any():
        row_of = {(int(i), int(j)): r for r, (i, j) in enumerate(zip(inp["row_req"], inp["row_pos"]))}
        base = bf16_bits_to_f64(emb[int(prm["mask_id"])])
        want = np.stack([base + (float(prm["alpha"]) * np.asarray(pe_ref[row_of[(int(i), int(j))]], np.float64)
                                 if prm["smoothing"] else 0.0) for i, j in np.argwhere(sm)])
    if sm.any():
        err = rownorm_rel(bf16_bits_to_f64(ne[sm]), want)
        assert err.max() <= PE_TOL, f"smoothed next_emb err {err.max():.3e}"
    out = dict(selection_excluded=int(amb["selection"].sum()),
               requests_excluded=int(amb["request"].sum()),
               requests_with_choices=n_choice,
               n_commit=int(state_gpu["n_commit"].sum()))
    _bound_excluded("selections", out["selection_excluded"], int(mask0.sum()))
    return out
