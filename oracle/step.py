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


def hierarchical_close_tie(cand, p, l, r, levels):
    """Does the centre-first walk HS(l, r, levels) meet a close tie?

    Walks the same recursion as ``commit.hierarchical_select``; at each
    sub-range the pick is the candidate nearest the centre, and an equal
    distance on both sides is broken by the higher p. When the two
    equidistant candidates' p are within FALLBACK_GAP_REL, a device whose
    float32 confidences differ from the oracle's by rounding may break the
    tie the other way, and every later pick of the range follows from it.
    """
    if levels <= 0 or r <= l:
        return False
    inside = [s for s in range(l, r) if cand[s]]
    if not inside:
        return False
    c = l + (r - l - 1) // 2
    dmin = min(abs(s - c) for s in inside)
    near = [s for s in inside if abs(s - c) == dmin]
    if len(near) == 2 and _close(float(p[near[0]]), float(p[near[1]])):
        return True
    s = min(inside, key=lambda t: (abs(t - c), -float(p[t]), t))
    return (hierarchical_close_tie(cand, p, l, s, levels - 1)
            or hierarchical_close_tie(cand, p, s + 1, r, levels - 1))


def ambiguity(inp, head, com):
    """Which decisions a correct device result may legitimately take differently.

    Per position (masked before the step): its argmax is ambiguous when the
    top-2 logits are within ARGMAX_GAP_REL * max(1, |max logit|); it is near
    a threshold when |p - tau| or |credit - kappa| < THRESH_BAND, where p is
    the float32 confidence and credit the float32 value after the update,
    both as the commit decided with them. Per request:
      * fallback taken: ambiguous (every masked position) when the two best
        confidences are within FALLBACK_GAP_REL or any position is;
      * hierarchy off (S = C): only the ambiguous positions, unless no
        candidate is left once they are removed (a flip could then empty C
        and call the fallback): then the whole request;
      * hierarchy on: every maximal masked span that holds an ambiguous
        position or whose centre-first walk meets a close tie of equidistant
        candidates; the whole request when no unambiguous candidate is left.
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
    tie_spans = 0
    for i in range(B):
        was = inp["mask"][i].astype(bool)
        if not was.any():
            continue
        if com["fallback"][i]:
            ps = sorted((float(com["p"][i, j]) for j in range(blk) if was[j]), reverse=True)
            close = len(ps) > 1 and _close(ps[0], ps[1])
            if close or pos_amb[i][was].any():
                req_amb[i] = True
                sel_amb[i] = was
            continue
        no_clean_cand = not (com["cand"][i] & ~pos_amb[i]).any()
        if not prm["hierarchical"]:
            sel_amb[i] = pos_amb[i]
        else:
            for (l, r) in masked_spans(was):
                tie = hierarchical_close_tie(com["cand"][i], com["p"][i], l, r,
                                             int(prm["hier_levels"]))
                tie_spans += int(tie)
                if tie or pos_amb[i, l:r].any():
                    sel_amb[i, l:r] = True
        if no_clean_cand and pos_amb[i][was].any():
            req_amb[i] = True
            sel_amb[i] = was
    return dict(argmax_row=argmax_amb_row, position=pos_amb, argmax_pos=arg_amb,
                selection=sel_amb, request=req_amb,
                counts=dict(argmax_rows=int(argmax_amb_row.sum()),
                            near_threshold=int((pos_amb & ~arg_amb).sum()),
                            tie_spans=tie_spans,
                            selection_positions=int(sel_amb.sum()),
                            requests=int(req_amb.sum())))
