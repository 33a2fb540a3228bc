"""Oracle: non-causal block attention over cached prefix + fresh window.

dInfer article, "vicinity KV refresh": each iteration recomputes K/V only for
the current block and a small neighbourhood and keeps the distant cache
fixed. Sangam abstract: bidirectional attention, so nothing is causal. So per
request the key set is the P cached prefix rows followed by the W fresh
window rows (left vicinity, block, right vicinity), and every window query
attends to all of them.
"""

import numpy as np


def block_attention(q, k, v, q_off, kv_off, scale):
    """O = softmax(Q K^T * scale) V per request and head, no mask.

    q: [sum W][H][dh], k, v: [sum L][H][dh] (float64). Request i owns query
    rows q_off[i]:q_off[i+1] and key rows kv_off[i]:kv_off[i+1]. A request
    with queries but no keys gets zeros (empty sum).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(q)
    B = len(q_off) - 1
    H = q.shape[1]
    for i in range(B):
        q0, q1 = int(q_off[i]), int(q_off[i + 1])
        k0, k1 = int(kv_off[i]), int(kv_off[i + 1])
        if q1 == q0 or k1 == k0:
            continue
        for h in range(H):
            s = (q[q0:q1, h, :] @ k[k0:k1, h, :].T) * scale      # scores [W, L]
            s = s - s.max(axis=1, keepdims=True)
            e = np.exp(s)
            a = e / e.sum(axis=1, keepdims=True)                   # softmax over keys
            out[q0:q1, h, :] = a @ v[k0:k1, h, :]
    return out
