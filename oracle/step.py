"""Oracle: one whole denoise step, and the ambiguity record used by parity.

The step (dInfer article: vicinity KV refresh, then the decoding strategy):
attention of the window queries over the cached prefix + fresh window K/V,
the LM head with its softmax statistics and P.E over the masked block rows,
then the commit. In these single-step workloads the head's hidden rows are
inputs of their own (planted rows), so the attention output does not feed
the head; the end-to-end model in ``oracle.model`` connects them.
"""

import numpy as np

from workloads import bf16_bits_to_f64

from .attention import block_attention
from .commit import commit, masked_spans
from .head import head_confidence

# Bands inside which the two sides may decide differently for legitimate
# rounding reasons (bf16 inputs, float32 accumulation on the device).
THRESH_BAND = 1e-3       # |p - tau| or |credit - kappa| (absolute)
ARGMAX_GAP_REL = 1e-4    # top-2 logit gap < 1e-4 * max(1, |m|)
FALLBACK_GAP_REL = 1e-3  # (p1 - p2) / p1 between the two best masked positions


def step_inputs_f64(inp, rows=None):
    """float64 views of a workload's bf16 arrays (rows: subset of head rows)."""
    out = dict(q=bf16_bits_to_f64(inp["q"]), k=bf16_bits_to_f64(inp["k"]),
               v=bf16_bits_to_f64(inp["v"]))
    hid = inp["hidden"] if rows is None else inp["hidden"][rows]
    out["hidden"] = bf16_bits_to_f64(hid)
    out["w_head"] = bf16_bits_to_f64(inp["w_head"])
    out["emb"] = bf16_bits_to_f64(inp["emb"])
    return out


def denoise_step(inp, f64=None, with_attention=True):
    """Run attention, head and commit for a workload dict from ``workloads``."""
    f = f64 if f64 is not None else step_inputs_f64(inp)
    res = {}
    if with_attention:
        res["attn"] = block_attention(f["q"], f["k"], f["v"], inp["q_off"],
                                      inp["kv_off"], inp["scale"])
    prm = inp["params"]
    head = head_confidence(f["hidden"], f["w_head"],
                           f["emb"] if prm["smoothing"] else None)
    res["head"] = head
    res["commit"] = commit(head["argmax"], head["conf"], head["pe"],
                           inp["row_req"], inp["row_pos"], inp["mask"],
                           inp["tokens"], inp["credit"], inp["prev"],
                           f["emb"], prm)
    res["ambiguity"] = ambiguity(inp, head, res["commit"])
    return res


def top2_gap(z):
    """Per row: (largest - second largest logit), and max(1, |largest|).

    A row with a single logit has no second one: its gap is infinite.
    """
    z = np.asarray(z, np.float64)
    if z.shape[1] < 2:
        return np.full(z.shape[0], np.inf), np.maximum(1.0, np.abs(z[:, 0]))
    part = np.partition(z, -2, axis=1)
    t1, t2 = part[:, -1], part[:, -2]
    return t1 - t2, np.maximum(1.0, np.abs(t1))


def _close(pa, pb):
    """Two confidences within FALLBACK_GAP_REL of the larger one."""
    return abs(pa - pb) < FALLBACK_GAP_REL * max(pa, pb)


# Enumeration caps: a request with more ambiguous positions, or more
# reachable selections, than this is excluded whole instead.
MAX_FLIPS = 8
MAX_ALTERNATIVES = 256


def hierarchical_choices(cand, p, l, r, levels):
    """Every selection HS(l, r, levels) can return when each close tie may
    go either way.

    Walks the recursion of ``commit.hierarchical_select``: at each sub-range
    the pick is the candidate nearest the centre, and an equal distance on
    both sides is broken by the higher p. When the two equidistant
    candidates' p are within FALLBACK_GAP_REL, a device whose float32
    confidences differ from the oracle's by rounding may take either, and
    the later picks of the range follow from that choice. Returns a set of
    frozensets, or None past MAX_ALTERNATIVES.
    """
    if levels <= 0 or r <= l:
        return {frozenset()}
    inside = [s for s in range(l, r) if cand[s]]
    if not inside:
        return {frozenset()}
    c = l + (r - l - 1) // 2
    dmin = min(abs(s - c) for s in inside)
    near = [s for s in inside if abs(s - c) == dmin]
    if len(near) == 2 and _close(float(p[near[0]]), float(p[near[1]])):
        picks = near
    else:
        picks = [min(inside, key=lambda t: (abs(t - c), -float(p[t]), t))]
    out = set()
    for s in picks:
        left = hierarchical_choices(cand, p, l, s, levels - 1)
        right = hierarchical_choices(cand, p, s + 1, r, levels - 1)
        if left is None or right is None:
            return None
        for a in left:
            for b in right:
                out.add(frozenset({s}) | a | b)
                if len(out) > MAX_ALTERNATIVES:
                    return None
    return out


def hierarchical_close_tie(cand, p, l, r, levels):
    """Does the centre-first walk HS(l, r, levels) meet a close tie?"""
    ch = hierarchical_choices(cand, p, l, r, levels)
    return ch is None or len(ch) > 1


def selection_choices(cand, p, was, prm):
    """Every selected set one request's commit can reach from these
    candidates: threshold (S = C) or hierarchical selection with close ties
    either way, then the fallback when nothing is selected (the most
    confident masked position, and every other one within FALLBACK_GAP_REL
    of it). Returns a set of frozensets, or None past MAX_ALTERNATIVES."""
    blk = len(was)
    if prm["hierarchical"]:
        sels = {frozenset()}
        for (l, r) in masked_spans(was):
            ch = hierarchical_choices(cand, p, l, r, int(prm["hier_levels"]))
            if ch is None:
                return None
            sels = {a | b for a in sels for b in ch}
            if len(sels) > MAX_ALTERNATIVES:
                return None
    else:
        sels = {frozenset(j for j in range(blk) if cand[j])}
    if frozenset() in sels and was.any():
        sels.discard(frozenset())
        ps = [float(p[j]) for j in range(blk) if was[j]]
        top = max(ps)
        sels |= {frozenset({j}) for j in range(blk) if was[j] and _close(float(p[j]), top)}
    return sels


def ambiguity(inp, head, com):
    """Which decisions a correct device result may legitimately take differently.

    Per position (masked before the step): its argmax is ambiguous when the
    top-2 logits are within ARGMAX_GAP_REL * max(1, |max logit|); it is near
    a threshold when |p - tau| or |credit - kappa| < THRESH_BAND, where p is
    the float32 confidence and credit the float32 value after the update,
    both as the commit decided with them. Either makes the position's
    candidacy uncertain. Per request, ``choices[i]`` is the set of selected
    sets the commit can reach with every uncertain candidacy taken either
    way and every close tie (hierarchical centre tie, fallback) broken
    either way (``selection_choices``); a correct device selects one of
    them, and when there is only one it must select exactly that. A request
    with more than MAX_FLIPS uncertain positions, or more than
    MAX_ALTERNATIVES reachable selections, is excluded whole (``request``,
    ``selection``) and counted.
    """
    prm = inp["params"]
    B, blk = inp["mask"].shape
    gap, scale = top2_gap(head["z"])
    argmax_amb_row = gap < ARGMAX_GAP_REL * scale
    pos_amb = np.zeros((B, blk), dtype=bool)
    arg_amb = np.zeros((B, blk), dtype=bool)
    for r in range(len(inp["row_req"])):
        i, j = int(inp["row_req"][r]), int(inp["row_pos"][r])
        if not inp["mask"][i, j]:
            continue
        p = float(com["p"][i, j])
        cr = float(com["credit_upd"][i, j])
        near = abs(p - prm["tau"]) < THRESH_BAND or abs(cr - prm["kappa"]) < THRESH_BAND
        pos_amb[i, j] = near or bool(argmax_amb_row[r])
        arg_amb[i, j] = bool(argmax_amb_row[r])
    sel_amb = np.zeros((B, blk), dtype=bool)   # positions whose selection is not compared
    req_amb = np.zeros(B, dtype=bool)
    choices = [None] * B
    n_alt = 0
    for i in range(B):
        was = inp["mask"][i].astype(bool)
        flips = np.flatnonzero(pos_amb[i] & was)
        if len(flips) > MAX_FLIPS:
            req_amb[i], sel_amb[i] = True, was
            continue
        alts = set()
        for bits in range(1 << len(flips)):
            cand = com["cand"][i].copy()
            for k, j in enumerate(flips):
                if bits >> k & 1:
                    cand[j] = not cand[j]
            sels = selection_choices(cand, com["p"][i], was, prm)
            if sels is None:
                alts = None
                break
            alts |= sels
            if len(alts) > MAX_ALTERNATIVES:
                alts = None
                break
        if alts is None:
            req_amb[i], sel_amb[i] = True, was
            continue
        choices[i] = alts
        n_alt += int(len(alts) > 1)
    return dict(argmax_row=argmax_amb_row, position=pos_amb, argmax_pos=arg_amb,
                selection=sel_amb, request=req_amb, choices=choices,
                counts=dict(argmax_rows=int(argmax_amb_row.sum()),
                            near_threshold=int((pos_amb & ~arg_amb).sum()),
                            requests_with_choices=n_alt,
                            selection_positions=int(sel_amb.sum()),
                            requests=int(req_amb.sum())))
