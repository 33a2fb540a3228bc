"""Oracle (test infrastructure only): the mixture-of-experts FFN of a
LLaDA-MoE-like block, float64 NumPy.

The pages name the model family (dInfer abstract: LLaDA-MoE; TIDE abstract:
MoE dLLMs, expert activation) and expert parallelism (dInfer article,
system optimisations) but give no formula. Readings, the common top-k MoE:
  * router logits = h . W_r^T over E experts; probabilities = softmax of
    the logits; the k experts of highest probability are chosen (ties: lower
    expert index); their weights are their probabilities renormalised to sum
    to one;
  * expert e is a SwiGLU FFN: silu(h . W1_e^T) * (h . W3_e^T), then . W2_e^T
    (the same block as the dense FFN of ``oracle.model``);
  * the output of a token is the weighted sum of its k experts' outputs.
"""

import numpy as np

from .model import silu


def route(h, w_router, topk):
    """Top-k routing: (ids [n][k] ascending by rank, weights [n][k], logits)."""
    z = h @ w_router.T                                   # [n][E]
    p = np.exp(z - z.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    E = z.shape[1]
    # highest probability first, lower expert index first on ties
    order = np.lexsort((np.broadcast_to(np.arange(E), z.shape), -p), axis=1)
    ids = order[:, :topk].astype(np.int32)
    pk = np.take_along_axis(p, ids, axis=1)
    return ids, pk / pk.sum(axis=1, keepdims=True), z


def expert(h, w13, w2, F):
    """SwiGLU expert on rows h: w13 = [gate rows; up rows] [2F][d], w2 [d][F]."""
    gu = h @ w13.T
    return (silu(gu[:, :F]) * gu[:, F:]) @ w2.T


def moe_ffn(h, w_router, w13, w2, topk, ids=None, weights=None):
    """y [n][d] = sum_j weight_j * expert_{id_j}(h). w13 [E][2F][d], w2
    [E][d][F]. ids / weights: given routing (else computed by ``route``)."""
    if ids is None:
        ids, weights, _ = route(h, w_router, topk)
    E, F2, _ = w13.shape
    F = F2 // 2
    y = np.zeros((h.shape[0], w2.shape[1]))
    for e in range(E):
        tok, slot = np.nonzero(ids == e)
        if tok.size:
            y[tok] += weights[tok, slot][:, None] * expert(h[tok], w13[e], w2[e], F)
    return y, ids, weights


def topk_gap(z, topk):
    """Gap between the k-th and (k+1)-th largest router logits per token (a
    routing decision closer than rounding can flip), and the logits' scale."""
    s = np.sort(z, axis=1)[:, ::-1]
    if z.shape[1] <= topk:
        return np.full(z.shape[0], np.inf), np.abs(s).max(axis=1)
    return s[:, topk - 1] - s[:, topk], np.maximum(1.0, np.abs(s[:, 0]))
