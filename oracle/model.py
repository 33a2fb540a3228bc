"""Oracle: the end-to-end block decode loop of a small random transformer.

What the pages fix:
  * masked diffusion decoding in blocks, with prefills that recur per block
    and an approximate K/V cache reused across the decodes in between
    (Sangam abstract; dInfer article, "vicinity KV refresh");
  * each iteration recomputes only the current block and a small
    neighbourhood; the distant cache stays fixed (vicinity KV refresh);
  * the decoding strategy of ``oracle.commit`` (threshold, credit,
    hierarchical) and iteration smoothing.
Readings (the pages are silent on the model and the loop's details):
  * bidirectional pre-norm transformer: RMSNorm (eps 1e-6, weight 1), fused
    q/k/v projection, rotary embedding (rotate-half pairs (i, i + dh/2),
    base 10000, absolute positions) on q and k, non-causal softmax attention,
    output projection + residual, RMSNorm, SwiGLU FFN silu(gate) * up, down
    projection + residual; final RMSNorm, untied LM head; no biases;
  * at the start of block b a full forward over all positions (prompt,
    committed tokens, masked positions with their current input embedding)
    refreshes the cache: the K/V of every layer for positions before the
    window are kept; the same forward's block rows feed the block's first
    commit;
  * every later step of the block runs the layers on the window only
    (left vicinity, block, right vicinity clipped at the sequence end); the
    K/V of the positions outside the window stay as the refresh left them
    and the window attends over all of them: cached prefix + fresh window +
    cached suffix (the "dual cache", the default: the vicinity refresh
    keeps the distant cache on both sides unchanged). The prefix-only
    variant (dual_cache = 0) attends over cached prefix + window and drops
    the positions right of the window;
  * input embeddings: committed positions E[token]; masked block positions
    the commit's next-step embedding (E[mask] + alpha * P.E); masked
    positions outside the block E[mask];
  * a block starts with prev = -1, credit = 0.
Float64 throughout; no intermediate rounding.
"""

import numpy as np

from workloads import bf16_bits_to_f64

from .attention import block_attention
from .commit import commit
from .head import head_confidence


def rmsnorm(x, eps):
    """x / sqrt(mean(x^2) + eps) over the last axis (weight 1)."""
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope(x, pos, base):
    """Rotary embedding of x [n][H][dh] at integer positions pos [n]."""
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = base ** (-np.arange(half, dtype=np.float64) * 2.0 / dh)
    ang = np.asarray(pos, np.float64)[:, None] * inv_freq[None, :]      # [n][half]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


class Model:
    """The random-init transformer of ``workloads.make_e2e_inputs`` in float64."""

    def __init__(self, inp):
        self.inp = inp
        self.d, self.H, self.dh, self.ffn = inp["d"], inp["H"], inp["dh"], inp["ffn"]
        self.eps, self.base = inp["rms_eps"], inp["rope_base"]
        self.emb = bf16_bits_to_f64(inp["emb"])
        self.w_head = bf16_bits_to_f64(inp["w_head"])
        self.layers = [{k: bf16_bits_to_f64(v) for k, v in lw.items()} for lw in inp["layer_weights"]]

    def layer(self, li, x, pos, k_prefix=None, v_prefix=None, k_suffix=None, v_suffix=None):
        """One layer on rows x [n][d]; keys = prefix (if any) + these rows
        + suffix (if any).

        Returns the new rows and this layer's K, V of the rows [n][H][dh].
        """
        W = self.layers[li]
        n, d, H, dh = x.shape[0], self.d, self.H, self.dh
        h = rmsnorm(x, self.eps)
        qkv = h @ W["wqkv"].T
        q = rope(qkv[:, :d].reshape(n, H, dh), pos, self.base)
        k = rope(qkv[:, d:2 * d].reshape(n, H, dh), pos, self.base)
        v = qkv[:, 2 * d:].reshape(n, H, dh)
        kk = np.concatenate([a for a in (k_prefix, k, k_suffix) if a is not None], axis=0)
        vv = np.concatenate([a for a in (v_prefix, v, v_suffix) if a is not None], axis=0)
        o = block_attention(q, kk, vv, [0, n], [0, kk.shape[0]], 1.0 / np.sqrt(dh))
        x = x + o.reshape(n, d) @ W["wo"].T
        h2 = rmsnorm(x, self.eps)
        gu = h2 @ W["wgu"].T
        x = x + (silu(gu[:, :self.ffn]) * gu[:, self.ffn:]) @ W["wdown"].T
        return x, k, v

    def forward(self, x, pos, cache=None, suffix=None):
        """All layers; cache / suffix = per-layer (K, V) of the rows before /
        after these rows, or None.

        Returns final normed hidden rows and the per-layer (K, V) of the rows.
        """
        kv = []
        for li in range(len(self.layers)):
            kp, vp = (None, None) if cache is None else cache[li]
            ks, vs = (None, None) if suffix is None else suffix[li]
            x, k, v = self.layer(li, x, pos, kp, vp, ks, vs)
            kv.append((k, v))
        return rmsnorm(x, self.eps), kv


def input_rows(model, tokens, masked, block_emb, b0, blk, rows):
    """Input embeddings of the given positions (see the module readings)."""
    mask_id = model.inp["params"]["mask_id"]
    out = np.empty((len(rows), model.d))
    for n, p in enumerate(rows):
        if b0 <= p < b0 + blk and block_emb is not None:
            out[n] = block_emb[p - b0]
        elif masked[p]:
            out[n] = model.emb[mask_id]
        else:
            out[n] = model.emb[tokens[p]]
    return out


def window(inp, b):
    """Block start b0 and the window [ws, we) of block b."""
    T = inp["prompt_len"] + inp["resp_len"]
    b0 = inp["prompt_len"] + b * inp["blk"]
    return b0, max(0, b0 - inp["vic"]), min(T, b0 + inp["blk"] + inp["vic"])


def forward_step(model, inp, tokens, masked, block_emb, b, refresh, cache):
    """Final-normed block rows of one step and the cache after it.

    refresh: every position runs and the cache becomes the K/V of the rows
    before the window and (inp["dual_cache"], default 1) of the rows after
    it; otherwise the window runs over the given cache. The cache is opaque
    to callers: pass back what the block's refresh returned.
    """
    T = inp["prompt_len"] + inp["resp_len"]
    blk = inp["blk"]
    dual = bool(inp.get("dual_cache", 1))
    b0, ws, we = window(inp, b)
    if refresh:
        rows = np.arange(T)
        x = input_rows(model, tokens, masked, None, b0, blk, rows)
        hid, kv = model.forward(x, rows)
        cache = dict(prefix=[(k[:ws], v[:ws]) for (k, v) in kv],
                     suffix=[(k[we:], v[we:]) for (k, v) in kv] if dual else None)
        return hid[b0:b0 + blk], cache
    rows = np.arange(ws, we)
    x = input_rows(model, tokens, masked, block_emb, b0, blk, rows)
    hid, _ = model.forward(x, rows, cache["prefix"], cache["suffix"])
    return hid[b0 - ws:b0 - ws + blk], cache


def eos_committed(inp, tokens, masked, upto, eos_id):
    """A committed response position before `upto` holds eos_id."""
    Lp = inp["prompt_len"]
    if eos_id < 0 or upto <= Lp:
        return False
    seg = slice(Lp, upto)
    return bool(((tokens[seg] == eos_id) & ~masked[seg]).any())


def decode(inp, max_blocks=None, record=False, max_steps_per_block=None, eos_id=-1, teacher=None):
    """Block decode loop; returns the final tokens and a per-step record.

    eos_id >= 0: early stop (dInfer article, "system optimisations": the
    loop ends once the end-of-sequence token is out). Before each block the
    committed response positions are checked; when one holds eos_id, no
    later block is decoded and its positions stay masked. The stop is taken
    between blocks: the block that commits EOS is finished first.

    teacher: optional [T] token ids (teacher forcing, for comparing another
    implementation's decode with this one decision by decision). Every
    position this loop commits takes teacher's token instead of its own
    argmax, in the state, the sequence and the next-step input embedding;
    the step record keeps this loop's own decision (``commit["tokens"]``).
    """
    model = Model(inp)
    prm = inp["params"]
    Lp, Lr, blk = inp["prompt_len"], inp["resp_len"], inp["blk"]
    T = Lp + Lr
    mask_id = prm["mask_id"]
    tokens = np.full(T, mask_id, np.int32)
    tokens[:Lp] = inp["prompt"]
    masked = np.zeros(T, bool)
    masked[Lp:] = True
    steps = []
    nblocks = Lr // blk if max_blocks is None else min(max_blocks, Lr // blk)
    for b in range(nblocks):
        b0 = Lp + b * blk
        if eos_committed(inp, tokens, masked, b0, eos_id):
            break
        bstate = dict(mask=masked[b0:b0 + blk][None].astype(np.uint8), tokens=tokens[b0:b0 + blk][None].copy(),
                      credit=np.zeros((1, blk), np.float32), prev=np.full((1, blk), -1, np.int32))
        block_emb = None
        cache = None
        step = 0
        while bstate["mask"].any():
            hb, cache = forward_step(model, inp, tokens, masked, block_emb, b, step == 0, cache)
            head = head_confidence(hb, model.w_head, model.emb if prm["smoothing"] else None)
            com = commit(head["argmax"], head["conf"], head["pe"], np.zeros(blk, np.int32),
                         np.arange(blk, dtype=np.int32), bstate["mask"], bstate["tokens"], bstate["credit"],
                         bstate["prev"], model.emb, prm)
            if record:
                steps.append(dict(block=b, step=step, hidden=hb, head=head, commit=com,
                                  state_in={k: v.copy() for k, v in bstate.items()}))
            bstate = dict(mask=com["mask"], tokens=com["tokens"].copy(), credit=com["credit"], prev=com["prev"])
            block_emb = com["next_emb"][0].copy()
            if teacher is not None:
                for j in np.flatnonzero(com["selected"][0]):
                    t = int(teacher[b0 + j])
                    bstate["tokens"][0, j] = t
                    block_emb[j] = model.emb[t]
            tokens[b0:b0 + blk] = bstate["tokens"][0]
            masked[b0:b0 + blk] = bstate["mask"][0].astype(bool)
            step += 1
            if max_steps_per_block is not None and step >= max_steps_per_block:
                break
    return dict(tokens=tokens, masked=masked, steps=steps)
