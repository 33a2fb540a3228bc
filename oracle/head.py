"""Oracle: LM head, vocabulary softmax statistics and the expected embedding.

dInfer article, decoding problems (3): a plain decoder keeps only the most
confident token of each position and discards the rest of the distribution.
Its iteration smoothing feeds the probability-weighted information of the
still-undecoded positions into the next iteration. Readings: the confidence
is the largest softmax probability (temperature 1, no bias), ties in the
argmax go to the lowest vocabulary index, and the "probability-weighted
information" is the expected embedding P.E = sum_v p_v E_v.
"""

import numpy as np


def lm_head_logits(hidden, w_head):
    """z[r, v] = <hidden[r], w_head[v]>; hidden [R][d], w_head [V][d]."""
    return np.asarray(hidden, np.float64) @ np.asarray(w_head, np.float64).T


def vocab_softmax_stats(z):
    """Per row: m = max z, a = lowest argmax, l = sum exp(z - m), conf = 1/l.

    conf equals the largest softmax probability exp(m - m) / l.
    """
    z = np.asarray(z, np.float64)
    m = z.max(axis=1)
    a = np.argmax(z, axis=1).astype(np.int32)   # first maximum = lowest index
    l = np.exp(z - m[:, None]).sum(axis=1)
    conf = 1.0 / l
    return m, a, l, conf


def expected_embedding(z, m, l, emb):
    """PE[r] = sum_v softmax(z[r])_v * emb[v]; emb [V][d]."""
    p = np.exp(np.asarray(z, np.float64) - m[:, None]) / l[:, None]
    return p @ np.asarray(emb, np.float64)


def head_confidence(hidden, w_head, emb=None):
    """The whole head for R rows: logits, stats, and P.E when emb is given."""
    z = lm_head_logits(hidden, w_head)
    m, a, l, conf = vocab_softmax_stats(z)
    pe = expected_embedding(z, m, l, emb) if emb is not None else None
    return dict(z=z, m=m, l=l, argmax=a, conf=conf, pe=pe)
