"""Seeded synthetic workloads for the block-decoding denoise step.

Every array is drawn from one ``numpy.random.default_rng(seed)`` (PCG64)
stream in the fixed order documented on each function, as float32, and then
rounded to bfloat16 with round-to-nearest-even. The bf16 bit patterns
(``uint16`` arrays) are what both the oracle and the GPU path consume.

Shapes follow the LLaDA-8B-like workloads that the dInfer and LLaDA serving
pages measure on (dInfer abstract; "Serving masked diffusion LLMs",
Key Findings 3): 32 heads x 128, vocabulary 126464, block 32, batch 1 or 16.
No benchmark item (HumanEval, GSM8K, ShareGPT, arXiv) is used: the values
are random, with a planted token per hidden row so that the head's argmax
and confidence have structure.
"""

from __future__ import annotations

import math

import numpy as np

# Rows drawn per chunk for the vocabulary-sized matrices. Part of the recipe:
# the draw sequence depends on it, so it never changes silently.
_VOCAB_CHUNK_ROWS = 8192


# --------------------------------------------------------------------------
# bfloat16 bit helpers (storage format only)
# --------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float64 (exact)."""
    return bf16_bits_to_f32(b).astype(np.float64)


def _normal_bf16(rng, shape, std):
    n = int(np.prod(shape))
    x = rng.standard_normal(n, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return f32_to_bf16_bits(x).reshape(shape)


def _normal_bf16_rows(rng, rows, cols, std):
    """[rows][cols] normal matrix drawn in fixed chunks of rows."""
    out = np.empty((rows, cols), dtype=np.uint16)
    for r0 in range(0, rows, _VOCAB_CHUNK_ROWS):
        r1 = min(rows, r0 + _VOCAB_CHUNK_ROWS)
        out[r0:r1] = _normal_bf16(rng, (r1 - r0, cols), std)
    return out


def _as_list(x, B):
    if isinstance(x, (list, tuple, np.ndarray)):
        assert len(x) == B
        return [int(v) for v in x]
    return [int(x)] * B


# --------------------------------------------------------------------------
# single denoise step workloads
# --------------------------------------------------------------------------

def calibrated_scale(V: int) -> float:
    """Factor applied to the planted coefficient c in the "cal" variants.

    With hidden = 0.5*N(0, I) + c*w_v/|w_v| and W ~ N(0, 1/d), the planted
    logit is about c and the other V-1 logits are about N(0, 1/4), so the
    confidence is about e^c / (e^c + V e^(1/8)). Scaling c by
    ln(9 V e^(1/8)) / 4 puts c = 4 at confidence 0.9, so that thresholds,
    credit and hierarchical selection all get exercised.
    """
    return math.log(9.0 * V * math.exp(0.125)) / 4.0


def _planted_hidden(rng, w_head, R, V, c_max, cal):
    """R hidden rows 0.5*noise + c*w_v/|w_v| around planted vocabulary rows
    (draws: planted ids, c, noise -- in that order)."""
    d = w_head.shape[1]
    planted = rng.integers(0, V, size=R).astype(np.int32)
    c = rng.uniform(0.0, c_max, size=R).astype(np.float32)
    if cal:
        c = (c * np.float32(calibrated_scale(V))).astype(np.float32)
    noise = rng.standard_normal((R, d), dtype=np.float32)
    wv = bf16_bits_to_f32(w_head[planted])
    wn = np.sqrt((wv.astype(np.float64) ** 2).sum(axis=1)).astype(np.float32)
    hid32 = np.float32(0.5) * noise + c[:, None] * (wv / wn[:, None])
    return planted, c, f32_to_bf16_bits(hid32)


def make_step_inputs(*, B=1, H=4, dh=64, V=2048, blk=32, P=128, vl=0, vr=0,
                     n_masked=None, c_max=6.0, cal=False, seed=0,
                     P_range=None, block_index=None, resp_len=256,
                     tau=0.9, lam=0.7, kappa=1.5, hierarchical=1,
                     hier_levels=1, smoothing=1, alpha=1.0, e_std=0.02,
                     name="custom"):
    """Inputs of one batched denoise step.

    Draw order from ``default_rng(seed)``:
      0. (``P_range`` given) P_i ~ U{lo..hi}, B draws.
      1. q  [sum W][H][dh] ~ N(0, 1)
      2. k  [sum L][H][dh] ~ N(0, 1)
      3. v  [sum L][H][dh] ~ N(0, 1)
      4. w_head [V][d] ~ N(0, 1/d) (std 1/sqrt(d)), in chunks of 8192 rows
      5. emb    [V][d] ~ N(0, e_std^2), same chunking
      6. per request: a permutation of blk (first n_masked are masked) when
         n_masked < blk, then blk token ids ~ U{0..V-2} for the committed slots
      7. planted token v_r ~ U{0..V-1}, R draws
      8. c_r ~ U(0, c_max), R draws (times ``calibrated_scale(V)`` if cal)
      9. noise [R][d] ~ N(0, 1); hidden = 0.5*noise + c*w_v/|w_v| (w_v as bf16)
     10. coin_r ~ U(0,1), ids_r ~ U{0..V-1}, credit_r ~ U(0, kappa) (0 if
         kappa is infinite); prev = v_r if coin < 1/2 else ids_r

    Per request i the key rows are P_i cached prefix rows followed by
    W_i = vl_i + blk + vr_i fresh window rows; q holds the W_i window rows.
    With ``block_index`` given, vr_i = min(vr, resp_len - blk*(b_i+1)).
    The head rows are the masked block positions, request-major, positions
    ascending (row_req / row_pos).
    """
    rng = np.random.default_rng(seed)
    d = H * dh
    if P_range is not None:
        P = [int(x) for x in rng.integers(P_range[0], P_range[1] + 1, size=B)]
    P = _as_list(P, B)
    vl = _as_list(vl, B)
    vr = _as_list(vr, B)
    if block_index is not None:
        block_index = _as_list(block_index, B)
        vr = [max(0, min(vr[i], resp_len - blk * (block_index[i] + 1))) for i in range(B)]
    W = [vl[i] + blk + vr[i] for i in range(B)]
    L = [P[i] + W[i] for i in range(B)]
    q_off = np.zeros(B + 1, dtype=np.int32)
    kv_off = np.zeros(B + 1, dtype=np.int32)
    q_off[1:] = np.cumsum(W)
    kv_off[1:] = np.cumsum(L)
    sumW, sumL = int(q_off[-1]), int(kv_off[-1])

    q = _normal_bf16(rng, (sumW, H, dh), 1.0)
    k = _normal_bf16(rng, (sumL, H, dh), 1.0)
    v = _normal_bf16(rng, (sumL, H, dh), 1.0)
    w_head = _normal_bf16_rows(rng, V, d, 1.0 / math.sqrt(d))
    emb = _normal_bf16_rows(rng, V, d, e_std)

    nm = blk if n_masked is None else int(n_masked)
    mask_id = V - 1
    mask = np.zeros((B, blk), dtype=np.uint8)
    tokens = np.zeros((B, blk), dtype=np.int32)
    for i in range(B):
        if nm < blk:
            perm = rng.permutation(blk)
            masked = np.zeros(blk, dtype=bool)
            masked[perm[:nm]] = True
        else:
            masked = np.ones(blk, dtype=bool)
        ids = rng.integers(0, max(V - 1, 1), size=blk).astype(np.int32)
        mask[i] = masked
        tokens[i] = np.where(masked, mask_id, ids)

    row_req, row_pos = [], []
    for i in range(B):
        for j in range(blk):
            if mask[i, j]:
                row_req.append(i)
                row_pos.append(j)
    row_req = np.asarray(row_req, dtype=np.int32)
    row_pos = np.asarray(row_pos, dtype=np.int32)
    R = len(row_req)

    planted, c, hidden = _planted_hidden(rng, w_head, R, V, c_max, cal)

    coin = rng.random(R)
    ids = rng.integers(0, V, size=R).astype(np.int32)
    if math.isinf(kappa):
        cr0 = np.zeros(R, dtype=np.float32)
    else:
        cr0 = rng.uniform(0.0, kappa, size=R).astype(np.float32)
    prev = np.full((B, blk), -1, dtype=np.int32)
    credit = np.zeros((B, blk), dtype=np.float32)
    for r in range(R):
        i, j = row_req[r], row_pos[r]
        prev[i, j] = planted[r] if coin[r] < 0.5 else ids[r]
        credit[i, j] = cr0[r]

    params = dict(tau=float(tau), lam=float(lam), kappa=float(kappa),
                  hierarchical=int(hierarchical), hier_levels=int(hier_levels),
                  smoothing=int(smoothing), alpha=float(alpha), mask_id=int(mask_id))
    return dict(name=name, seed=seed, B=B, H=H, dh=dh, d=d, V=V, blk=blk,
                P=P, vl=vl, vr=vr, W=W, L=L, q_off=q_off, kv_off=kv_off,
                max_q=max(W), max_kv=max(L), R=R, scale=1.0 / math.sqrt(dh),
                q=q, k=k, v=v, w_head=w_head, emb=emb, hidden=hidden,
                row_req=row_req, row_pos=row_pos, planted=planted, c=c,
                mask=mask, tokens=tokens, credit=credit, prev=prev,
                params=params)


# The four single-step workloads: a tiny case, the LLaDA-8B-shaped step at
# batch 1 and at batch 16 (ragged prefixes, each request at a different block
# of a 256-token response), and an 8K-prefix long-context step.
STEP_CONFIGS = {
    "tiny": dict(B=1, H=4, dh=64, V=2048, blk=32, P=128, vl=0, vr=0,
                 n_masked=16, c_max=6.0),
    "llada8b_b1": dict(B=1, H=32, dh=128, V=126464, blk=32, P=512, vl=32, vr=32,
                       c_max=6.0),
    "llada8b_b16": dict(B=16, H=32, dh=128, V=126464, blk=32, P_range=(256, 1024),
                        vl=32, vr=32, block_index=[i % 8 for i in range(16)],
                        resp_len=256, c_max=6.0),
    "longctx_8k": dict(B=1, H=32, dh=128, V=126464, blk=64, P=8192, vl=64, vr=64,
                       c_max=4.0),
}


def step_config(name: str, seed: int = 0, cal: bool = False, **over):
    """One of ``STEP_CONFIGS`` (optionally the calibrated "cal" variant)."""
    kw = dict(STEP_CONFIGS[name])
    kw.update(over)
    return make_step_inputs(seed=seed, cal=cal, name=name + ("_cal" if cal else ""), **kw)


# --------------------------------------------------------------------------
# end-to-end block decode workload (small random bidirectional transformer)
# --------------------------------------------------------------------------

def make_e2e_inputs(*, seed=0, layers=4, d=1024, H=16, dh=64, ffn=4096,
                    V=32768, prompt_len=256, resp_len=256, blk=32, vic=32,
                    w_std=0.02, tau=0.9, lam=0.7, kappa=1.5, hierarchical=1,
                    hier_levels=1, smoothing=1, alpha=1.0, dual_cache=1):
    """Random-init weights and a random prompt for the block decode loop.

    dual_cache: 1 = window steps attend over the whole sequence, the K/V
    outside the window staying as the block's refresh left them; 0 = over
    the cached prefix and the window only (a flag; nothing is drawn).
    Draw order from ``default_rng(seed)``: prompt ids ~ U{0..V-2}; emb [V][d];
    w_head [V][d]; then per layer wqkv [3d][d] (q rows, k rows, v rows),
    wo [d][d], wgu [2 ffn][d] (gate rows, then up rows), wdown [d][ffn];
    all N(0, w_std^2). RMSNorm weights are ones and are not drawn.
    """
    assert H * dh == d
    rng = np.random.default_rng(seed)
    mask_id = V - 1
    prompt = rng.integers(0, V - 1, size=prompt_len).astype(np.int32)
    emb = _normal_bf16_rows(rng, V, d, w_std)
    w_head = _normal_bf16_rows(rng, V, d, w_std)
    lw = []
    for _ in range(layers):
        lw.append(dict(
            wqkv=_normal_bf16(rng, (3 * d, d), w_std),
            wo=_normal_bf16(rng, (d, d), w_std),
            wgu=_normal_bf16(rng, (2 * ffn, d), w_std),
            wdown=_normal_bf16(rng, (d, ffn), w_std),
        ))
    params = dict(tau=float(tau), lam=float(lam), kappa=float(kappa),
                  hierarchical=int(hierarchical), hier_levels=int(hier_levels),
                  smoothing=int(smoothing), alpha=float(alpha), mask_id=int(mask_id))
    return dict(seed=seed, layers=layers, d=d, H=H, dh=dh, ffn=ffn, V=V,
                prompt_len=prompt_len, resp_len=resp_len, blk=blk, vic=vic,
                dual_cache=int(dual_cache), prompt=prompt, emb=emb, w_head=w_head, layer_weights=lw,
                rope_base=10000.0, rms_eps=1e-6, params=params)


# --------------------------------------------------------------------------
# step-level serving: a request trace and the step buffers it runs over
# --------------------------------------------------------------------------

SERVE_MIXES = {
    # short prompts, long responses: decodes dominate
    "decode_heavy": dict(prompt_range=(64, 512), resp_choices=(128, 256)),
    # long prompts, short responses: recurring whole-sequence prefills dominate
    "prefill_heavy": dict(prompt_range=(2048, 8192), resp_choices=(64, 128)),
}


def make_serve_trace(*, n, rate_per_s, prompt_range, resp_choices, seed=0):
    """Poisson arrivals of n requests (times in ms, first at 0).

    Draw order from ``default_rng(seed)``: n - 1 exponential gaps with mean
    1000 / rate_per_s ms; prompt lengths ~ U{lo..hi}; response lengths
    uniform over resp_choices."""
    rng = np.random.default_rng(seed)
    gaps = rng.exponential(1000.0 / rate_per_s, size=max(0, n - 1))
    arrival = np.concatenate([[0.0], np.cumsum(gaps)])
    prompt = rng.integers(prompt_range[0], prompt_range[1] + 1, size=n).astype(np.int32)
    resp = np.asarray(resp_choices, dtype=np.int32)[rng.integers(0, len(resp_choices), size=n)]
    return dict(arrival_ms=arrival, prompt_len=prompt, resp_len=resp)


def make_serve_inputs(*, slots, blk, H, dh, V, q_rows, kv_rows, c_max=6.0, cal=True, e_std=0.02, seed=0,
                      tau=0.9, lam=0.7, kappa=1.5, hierarchical=1, hier_levels=1, smoothing=1, alpha=1.0):
    """Fixed step buffers for a scheduled run: every step's query, key and
    value rows are the first rows of q / k / v, and its head rows the first
    rows of hidden (one block of blk rows per scheduled slot).

    Draw order from ``default_rng(seed)``: q [q_rows][H][dh], k, v
    [kv_rows][H][dh] ~ N(0, 1); w_head [V][d] ~ N(0, 1/d); emb [V][d] ~
    N(0, e_std^2); then slots*blk planted hidden rows (as in
    ``make_step_inputs``)."""
    rng = np.random.default_rng(seed)
    d = H * dh
    q = _normal_bf16(rng, (q_rows, H, dh), 1.0)
    k = _normal_bf16(rng, (kv_rows, H, dh), 1.0)
    v = _normal_bf16(rng, (kv_rows, H, dh), 1.0)
    w_head = _normal_bf16_rows(rng, V, d, 1.0 / math.sqrt(d))
    emb = _normal_bf16_rows(rng, V, d, e_std)
    planted, c, hidden = _planted_hidden(rng, w_head, slots * blk, V, c_max, cal)
    params = dict(tau=float(tau), lam=float(lam), kappa=float(kappa),
                  hierarchical=int(hierarchical), hier_levels=int(hier_levels),
                  smoothing=int(smoothing), alpha=float(alpha), mask_id=int(V - 1))
    return dict(slots=slots, blk=blk, H=H, dh=dh, d=d, V=V, scale=1.0 / math.sqrt(dh), q=q, k=k, v=v,
                w_head=w_head, emb=emb, hidden=hidden, planted=planted, c=c, params=params)


# --------------------------------------------------------------------------
# mixture-of-experts FFN (LLaDA-MoE-like shapes, random weights)
# --------------------------------------------------------------------------

# Window step of block decoding (blk 32 + 2 x 32 vicinity) and a refresh of
# 512 positions through a 64-expert top-8 FFN of width 1024 on d = 2048.
MOE_CONFIGS = {
    "tiny": dict(n=40, d=256, E=8, F=128, topk=2),
    "llada_moe_window": dict(n=96, d=2048, E=64, F=1024, topk=8),
    "llada_moe_refresh": dict(n=512, d=2048, E=64, F=1024, topk=8),
}


def make_moe_inputs(*, n, d, E, F, topk, seed=0, w_std=0.02, router_std=None):
    """Inputs of one MoE FFN: normed rows and random expert weights.

    Draw order from ``default_rng(seed)``: h [n][d] ~ N(0, 1); w_router
    [E][d] ~ N(0, router_std^2) (default 1/sqrt(d): unit-scale logits);
    w13 [E][2F][d] (per expert the F gate rows, then the F up rows) and w2
    [E][d][F] ~ N(0, w_std^2), drawn expert by expert."""
    rng = np.random.default_rng(seed)
    rs = (1.0 / math.sqrt(d)) if router_std is None else router_std
    h = _normal_bf16(rng, (n, d), 1.0)
    w_router = _normal_bf16(rng, (E, d), rs)
    w13 = np.empty((E, 2 * F, d), dtype=np.uint16)
    w2 = np.empty((E, d, F), dtype=np.uint16)
    for e in range(E):
        w13[e] = _normal_bf16(rng, (2 * F, d), w_std)
        w2[e] = _normal_bf16(rng, (d, F), w_std)
    return dict(seed=seed, n=n, d=d, E=E, F=F, topk=topk, h=h, w_router=w_router, w13=w13, w2=w2)
