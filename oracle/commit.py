"""Oracle: the parallel-decode commit of one denoise step.

Sources (dInfer article, "the art of decoding"):
  * threshold parallel decoding: every masked position whose confidence
    reaches tau is committed in the same iteration;
  * credit decoding: a token that has been predicted stably over several
    iterations accumulates credit and may be committed although its current
    confidence is lower; the update is credit <- lambda*credit + p while the
    argmax is unchanged, reset on change, commit when p >= tau or
    credit >= kappa;
  * hierarchical decoding: the region to decode is split in two recursively
    and the centre of each sub-region is decoded first, which spaces new
    tokens apart and fills a region in about logarithmically many steps;
  * iteration smoothing: still-masked positions carry their probability-
    weighted information into the next iteration.

Readings where the article is silent:
  * reset on change sets credit to the current p (history dropped, the
    current observation kept); "no history" is prev = -1;
  * hierarchical selection runs HS(l, r, levels) on each maximal run of
    consecutive masked positions of the block: no candidate in [l, r) or no
    level left gives nothing; otherwise pick the candidate nearest the
    centre c = l + (r - l - 1) // 2 (ties: higher p, then lower position)
    and recurse on both sides with one level less;
  * at least one commit per step: if nothing is selected, the masked
    position with the highest p (lowest position on ties) is committed;
  * next-step input embeddings: committed positions get E[token]; masked
    ones get E[mask_id] + alpha*PE (smoothing on) or E[mask_id].

Decision precision: the credit update and the comparisons are taken in
float32 (a product then a sum, each rounded), the precision the kernel takes
them in, so that a decision is the same on both sides for the same inputs.
"""

import numpy as np

F32 = np.float32


def masked_spans(mask_row):
    """Maximal runs [l, r) of consecutive masked positions."""
    spans, j, n = [], 0, len(mask_row)
    while j < n:
        if mask_row[j]:
            l = j
            while j < n and mask_row[j]:
                j += 1
            spans.append((l, j))
        else:
            j += 1
    return spans


def hierarchical_select(cand, p, l, r, levels):
    """HS(l, r, levels): centre-first recursive bisection over candidates.

    cand: bool per position; p: float32 confidence per position.
    """
    if levels <= 0 or r <= l:
        return set()
    inside = [s for s in range(l, r) if cand[s]]
    if not inside:
        return set()
    c = l + (r - l - 1) // 2
    s = min(inside, key=lambda t: (abs(t - c), -float(p[t]), t))
    return ({s} | hierarchical_select(cand, p, l, s, levels - 1)
            | hierarchical_select(cand, p, s + 1, r, levels - 1))


def commit(argmax, conf, pe, row_req, row_pos, mask, tokens, credit, prev,
           emb, params):
    """Apply one commit to the per-request block state.

    argmax [R] int, conf [R] (cast to float32), pe [R][d] or None,
    row_req/row_pos [R]: head row r belongs to request row_req[r], block
    position row_pos[r]. Rows at unmasked positions are ignored; a masked
    position without a row, or two rows for one position, is an error.
    mask [B][blk] (1 = masked), tokens/prev int32, credit float32.
    emb [V][d]. Returns the new state, next_emb [B][blk][d] (float64),
    n_commit [B] and the decision record: cand, selected, fallback, the
    float32 p and argmax of each masked position, and credit_upd, its
    credit after the update and before the commit resets it.
    """
    mask = np.array(mask, dtype=np.uint8)
    tokens = np.array(tokens, dtype=np.int32)
    credit = np.array(credit, dtype=F32)
    prev = np.array(prev, dtype=np.int32)
    emb = np.asarray(emb, np.float64)
    B, blk = mask.shape
    d = emb.shape[1]
    tau, lam, kappa = F32(params["tau"]), F32(params["lam"]), F32(params["kappa"])
    alpha = float(params["alpha"])
    mask_id = int(params["mask_id"])
    smoothing = bool(params["smoothing"])
    hier = bool(params["hierarchical"])
    levels = int(params["hier_levels"])
    if smoothing and pe is None:
        raise ValueError("smoothing needs P.E")

    row_of = np.full((B, blk), -1, dtype=np.int64)
    for r in range(len(row_req)):
        i, j = int(row_req[r]), int(row_pos[r])
        if not (0 <= i < B and 0 <= j < blk):
            raise ValueError("row outside the block")
        if not mask[i, j]:
            continue
        if row_of[i, j] >= 0:
            raise ValueError("two rows for one masked position")
        row_of[i, j] = r

    next_emb = np.zeros((B, blk, d), dtype=np.float64)
    n_commit = np.zeros(B, dtype=np.int32)
    cand = np.zeros((B, blk), dtype=bool)
    selected = np.zeros((B, blk), dtype=bool)
    fallback = np.zeros(B, dtype=bool)
    pvals = np.zeros((B, blk), dtype=F32)
    avals = np.full((B, blk), -1, dtype=np.int32)
    credit_upd = np.zeros((B, blk), dtype=F32)   # after the update, before the writes

    for i in range(B):
        was_masked = mask[i].astype(bool).copy()
        # 1. credit update and candidates, masked positions only
        for j in range(blk):
            if not was_masked[j]:
                continue
            r = row_of[i, j]
            if r < 0:
                raise ValueError("masked position without a head row")
            a = int(argmax[r])
            p = F32(conf[r])
            if prev[i, j] == a:
                cr = F32(F32(lam * credit[i, j]) + p)
            else:
                cr = p
            credit[i, j] = cr
            credit_upd[i, j] = cr
            prev[i, j] = a
            pvals[i, j] = p
            avals[i, j] = a
            cand[i, j] = bool(p >= tau) or bool(cr >= kappa)
        # 2. selection
        if hier:
            S = set()
            for (l, r) in masked_spans(was_masked):
                S |= hierarchical_select(cand[i], pvals[i], l, r, levels)
        else:
            S = {j for j in range(blk) if cand[i, j]}
        # 3. at least one commit while something is masked
        if not S and was_masked.any():
            js = [j for j in range(blk) if was_masked[j]]
            S = {max(js, key=lambda t: (float(pvals[i, t]), -t))}
            fallback[i] = True
        # 4. writes
        for j in range(blk):
            if was_masked[j] and j in S:
                tokens[i, j] = avals[i, j]
                mask[i, j] = 0
                credit[i, j] = F32(0.0)
                prev[i, j] = -1
                selected[i, j] = True
                next_emb[i, j] = emb[avals[i, j]]
            elif was_masked[j]:
                e = emb[mask_id].copy()
                if smoothing:
                    e = e + alpha * np.asarray(pe[row_of[i, j]], np.float64)
                next_emb[i, j] = e
            else:
                next_emb[i, j] = emb[tokens[i, j]]
        n_commit[i] = len(S)

    return dict(mask=mask, tokens=tokens, credit=credit, prev=prev,
                next_emb=next_emb, n_commit=n_commit, cand=cand,
                selected=selected, fallback=fallback, p=pvals, a=avals,
                credit_upd=credit_upd)
