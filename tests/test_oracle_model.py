"""Pins for the end-to-end oracle: transformer pieces and the block loop (CPU)."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import model as om
from workloads import make_e2e_inputs

TINY = dict(layers=2, d=64, H=2, dh=32, ffn=128, V=128, prompt_len=16, resp_len=32, blk=16, vic=8)


def test_rmsnorm_matches_torch():
    x = np.random.default_rng(0).standard_normal((5, 24)) * 3
    ref = F.rms_norm(torch.from_numpy(x), (24,), eps=1e-6).numpy()
    np.testing.assert_allclose(om.rmsnorm(x, 1e-6), ref, rtol=1e-13)
    assert np.allclose(np.sqrt(np.mean(om.rmsnorm(x, 0.0) ** 2, axis=-1)), 1.0)


def test_silu_matches_torch():
    x = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(om.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-13, atol=1e-300)


def test_rope_is_a_rotation_by_position():
    rng = np.random.default_rng(1)
    n, H, dh = 6, 2, 8
    x = rng.standard_normal((n, H, dh))
    pos = np.array([0, 1, 2, 5, 100, 511])
    y = om.rope(x, pos, 10000.0)
    # complex form: pair (i, i + dh/2) as x_i + 1j x_{i+dh/2}, rotated by pos * base^(-2i/dh)
    half = dh // 2
    zc = x[..., :half] + 1j * x[..., half:]
    th = pos[:, None, None] * 10000.0 ** (-2.0 * np.arange(half) / dh)
    ref = zc * np.exp(1j * th)
    np.testing.assert_allclose(y[..., :half], ref.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[..., half:], ref.imag, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[0], x[0], rtol=1e-15)
    # scores depend on relative position only
    q, k = rng.standard_normal((1, 1, dh)), rng.standard_normal((1, 1, dh))
    s1 = (om.rope(q, [7], 1e4) * om.rope(k, [3], 1e4)).sum()
    s2 = (om.rope(q, [104], 1e4) * om.rope(k, [100], 1e4)).sum()
    assert abs(s1 - s2) < 1e-12


def _torch_layer(x, pos, W, H, dh, ffn, eps):
    """The same layer from torch primitives (SDPA, rms_norm, silu, complex rope)."""
    t = lambda a: torch.from_numpy(np.asarray(a, np.float64))  # noqa: E731
    x = t(x)
    n, d = x.shape
    h = F.rms_norm(x, (d,), eps=eps)
    qkv = h @ t(W["wqkv"]).T

    def rot(a):
        a = a.reshape(n, H, dh)
        c = torch.complex(a[..., :dh // 2], a[..., dh // 2:])
        th = t(pos)[:, None, None] * 10000.0 ** (-2.0 * torch.arange(dh // 2, dtype=torch.float64) / dh)
        c = c * torch.polar(torch.ones_like(th), th)
        return torch.cat([c.real, c.imag], -1)
    q, k, v = rot(qkv[:, :d]), rot(qkv[:, d:2 * d]), qkv[:, 2 * d:].reshape(n, H, dh)
    o = F.scaled_dot_product_attention(q.permute(1, 0, 2), k.permute(1, 0, 2), v.permute(1, 0, 2))
    x = x + o.permute(1, 0, 2).reshape(n, d) @ t(W["wo"]).T
    gu = F.rms_norm(x, (d,), eps=eps) @ t(W["wgu"]).T
    x = x + (F.silu(gu[:, :ffn]) * gu[:, ffn:]) @ t(W["wdown"]).T
    return x.numpy()


def test_layer_matches_torch_primitives():
    inp = make_e2e_inputs(seed=2, **TINY)
    m = om.Model(inp)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((12, m.d))
    pos = np.arange(12) + 4
    y, _, _ = m.layer(0, x, pos)
    ref = _torch_layer(x, pos, m.layers[0], m.H, m.dh, m.ffn, m.eps)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-10)


def test_cached_window_equals_full_forward_at_the_sequence_end():
    """Keys = cached prefix + fresh window reproduce the full forward when the
    window reaches the end of the sequence and nothing changed."""
    inp = make_e2e_inputs(seed=4, **TINY)
    m = om.Model(inp)
    T = 48
    rng = np.random.default_rng(5)
    x = rng.standard_normal((T, m.d))
    full, kv = m.forward(x, np.arange(T))
    ws = 30
    cache = [(k[:ws], v[:ws]) for (k, v) in kv]
    win, _ = m.forward(x[ws:], np.arange(ws, T), cache)
    np.testing.assert_allclose(win, full[ws:], rtol=1e-11, atol=1e-11)


def test_dual_cache_window_equals_full_forward_mid_sequence():
    """With a suffix cache too, a window in the middle of the sequence sees
    every key the full forward saw, so unchanged inputs reproduce it; the
    prefix-only cache does not (the suffix keys are missing)."""
    inp = make_e2e_inputs(seed=4, **TINY)
    m = om.Model(inp)
    T, ws, we = 48, 12, 30
    x = np.random.default_rng(6).standard_normal((T, m.d))
    full, kv = m.forward(x, np.arange(T))
    pre = [(k[:ws], v[:ws]) for (k, v) in kv]
    suf = [(k[we:], v[we:]) for (k, v) in kv]
    win, _ = m.forward(x[ws:we], np.arange(ws, we), pre, suf)
    np.testing.assert_allclose(win, full[ws:we], rtol=1e-11, atol=1e-11)
    win_pre, _ = m.forward(x[ws:we], np.arange(ws, we), pre)
    assert np.abs(win_pre - full[ws:we]).max() > 1e-3


@pytest.mark.parametrize("dual", [0, 1])
def test_forward_step_window_after_refresh(dual):
    """A window step right after the refresh with the refresh's own block
    inputs reproduces the refresh's block rows exactly with the dual cache,
    and only up to the dropped right-hand keys without it."""
    inp = make_e2e_inputs(seed=8, dual_cache=dual, **TINY)
    m = om.Model(inp)
    T = inp["prompt_len"] + inp["resp_len"]
    mask_id = inp["params"]["mask_id"]
    tokens = np.full(T, mask_id, np.int32)
    tokens[:inp["prompt_len"]] = inp["prompt"]
    masked = np.zeros(T, bool)
    masked[inp["prompt_len"]:] = True
    b = 0
    b0, ws, we = om.window(inp, b)
    assert we < T                               # the suffix is not empty
    h_ref, cache = om.forward_step(m, inp, tokens, masked, None, b, True, None)
    blk_in = om.input_rows(m, tokens, masked, None, b0, inp["blk"], np.arange(b0, b0 + inp["blk"]))
    h_win, _ = om.forward_step(m, inp, tokens, masked, blk_in, b, False, cache)
    err = np.abs(h_win - h_ref).max()
    if dual:
        assert err < 1e-11
    else:
        assert err > 1e-3


def test_decode_dual_cache_commits_everything():
    inp = make_e2e_inputs(seed=6, dual_cache=1, **TINY)
    res = om.decode(inp, record=True)
    assert not res["masked"].any()
    per_block = [sum(1 for s in res["steps"] if s["block"] == b) for b in range(2)]
    assert per_block == [16, 16]


def test_decode_commits_every_block_with_fallback_only():
    inp = make_e2e_inputs(seed=6, **TINY)
    res = om.decode(inp, record=True)
    assert not res["masked"].any()
    assert np.array_equal(res["tokens"][:16], inp["prompt"])
    per_block = [sum(1 for s in res["steps"] if s["block"] == b) for b in range(2)]
    assert per_block == [16, 16]               # random weights: p << tau, one commit per step
    assert all(s["commit"]["fallback"][0] for s in res["steps"])


@pytest.mark.parametrize("hier,steps", [(0, 1), (1, math.ceil(math.log2(17)))])
def test_decode_zero_threshold(hier, steps):
    inp = make_e2e_inputs(seed=7, tau=0.0, hierarchical=hier, **TINY)
    res = om.decode(inp, record=True)
    per_block = [sum(1 for s in res["steps"] if s["block"] == b) for b in range(2)]
    assert per_block == [steps, steps]


def _per_block(res, nblocks):
    return [sum(1 for s in res["steps"] if s["block"] == b) for b in range(nblocks)]


def test_decode_eos_stops_after_the_block_that_commits_it():
    """Early stop after EOS (dInfer article, system optimisations): the
    block that commits EOS finishes, no later block is decoded."""
    inp = make_e2e_inputs(seed=6, **TINY)
    Lp, blk = inp["prompt_len"], inp["blk"]
    free = om.decode(inp, record=True)
    eos = int(free["tokens"][Lp + 3])                    # committed in block 0
    res = om.decode(inp, record=True, eos_id=eos)
    assert np.array_equal(res["tokens"][:Lp + blk], free["tokens"][:Lp + blk])
    assert not res["masked"][:Lp + blk].any()
    assert res["masked"][Lp + blk:].all()
    assert (res["tokens"][Lp + blk:] == inp["params"]["mask_id"]).all()
    assert _per_block(res, 2) == [16, 0]                 # block 0 ran all its steps


def test_decode_eos_in_the_prompt_or_never_committed_does_not_stop():
    inp = make_e2e_inputs(seed=6, **TINY)
    Lp = inp["prompt_len"]
    free = om.decode(inp)
    resp = set(free["tokens"][Lp:].tolist())
    in_prompt = [int(t) for t in inp["prompt"] if int(t) not in resp]
    never = [t for t in range(inp["V"] - 1) if t not in resp and t not in set(inp["prompt"].tolist())]
    assert in_prompt and never
    for eos in (in_prompt[0], never[0]):
        res = om.decode(inp, eos_id=eos)
        assert np.array_equal(res["tokens"], free["tokens"]) and not res["masked"].any()


def test_decode_eos_first_committed_in_a_middle_block():
    cfg = dict(TINY, resp_len=48)                        # three blocks of 16
    inp = make_e2e_inputs(seed=9, **cfg)
    Lp, blk = inp["prompt_len"], inp["blk"]
    free = om.decode(inp)
    b0_tokens = set(free["tokens"][Lp:Lp + blk].tolist())
    later = [int(t) for t in free["tokens"][Lp + blk:Lp + 2 * blk] if int(t) not in b0_tokens]
    assert later
    res = om.decode(inp, record=True, eos_id=later[0])
    assert np.array_equal(res["tokens"][:Lp + 2 * blk], free["tokens"][:Lp + 2 * blk])
    assert res["masked"][Lp + 2 * blk:].all() and not res["masked"][:Lp + 2 * blk].any()
    assert _per_block(res, 3) == [16, 16, 0]


def test_teacher_forcing_with_the_own_tokens_changes_nothing():
    inp = make_e2e_inputs(seed=7, tau=0.0, **TINY)
    free = om.decode(inp, record=True)
    forced = om.decode(inp, record=True, teacher=free["tokens"])
    assert np.array_equal(forced["tokens"], free["tokens"])
    assert len(forced["steps"]) == len(free["steps"])
    for a, b in zip(forced["steps"], free["steps"]):
        assert np.array_equal(a["head"]["z"], b["head"]["z"])


def test_teacher_forcing_takes_the_teacher_token_and_keeps_the_own_decision():
    inp = make_e2e_inputs(seed=7, tau=0.0, **TINY)
    Lp, V = inp["prompt_len"], inp["V"]
    free = om.decode(inp, record=True)
    first = free["steps"][0]
    j = int(np.flatnonzero(first["commit"]["selected"][0])[0])     # the first commit of block 0
    teacher = free["tokens"].copy()
    teacher[Lp + j] = (teacher[Lp + j] + 1) % (V - 1)
    forced = om.decode(inp, record=True, teacher=teacher)
    assert forced["tokens"][Lp + j] == teacher[Lp + j]
    assert forced["steps"][0]["commit"]["tokens"][0, j] == free["tokens"][Lp + j]
    # the changed token is an input of the next step: its hidden rows move
    assert np.abs(forced["steps"][1]["hidden"] - free["steps"][1]["hidden"]).max() > 1e-6
    # with tau = 0 and hierarchy the positions committed per step follow from
    # the mask alone, so both runs commit the same positions at each step
    for a, b in zip(forced["steps"], free["steps"]):
        assert np.array_equal(a["commit"]["selected"], b["commit"]["selected"])
