"""Pins for the oracle's block attention (CPU only).

The oracle is checked against things other than itself: a hand-worked case,
a brute-force loop over scalar scores, textbook special cases, and
PyTorch's float64 scaled_dot_product_attention on ragged multi-request inputs.
"""

import math

import numpy as np
import pytest
import torch

from oracle import block_attention


def _brute(q, k, v, q_off, kv_off, scale):
    out = np.zeros_like(q)
    for i in range(len(q_off) - 1):
        for h in range(q.shape[1]):
            for t in range(q_off[i], q_off[i + 1]):
                keys = range(kv_off[i], kv_off[i + 1])
                s = [scale * math.fsum(q[t, h, x] * k[u, h, x] for x in range(q.shape[2]))
                     for u in keys]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                tot = math.fsum(e)
                for x in range(q.shape[2]):
                    out[t, h, x] = math.fsum(e[n] / tot * v[u, h, x] for n, u in enumerate(keys))
    return out


def _ragged(rng, W, L, H, dh):
    q_off = np.concatenate([[0], np.cumsum(W)]).astype(np.int32)
    kv_off = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    q = rng.standard_normal((q_off[-1], H, dh))
    k = rng.standard_normal((kv_off[-1], H, dh))
    v = rng.standard_normal((kv_off[-1], H, dh))
    return q, k, v, q_off, kv_off


def test_handworked(golden):
    g = golden("attention_handworked.json")
    q = np.array(g["q"], float)[:, None, :]
    k = np.array(g["k"], float)[:, None, :]
    v = np.array(g["v"], float)[:, None, :]
    o = block_attention(q, k, v, [0, 2], [0, 3], g["scale"])
    np.testing.assert_allclose(o[:, 0, :], np.array(g["out"]), atol=g["abs_tol"])


def test_brute_force_ragged():
    rng = np.random.default_rng(1)
    q, k, v, qo, ko = _ragged(rng, [3, 1, 2], [5, 1, 7], 2, 3)
    o = block_attention(q, k, v, qo, ko, 0.37)
    np.testing.assert_allclose(o, _brute(q, k, v, qo, ko, 0.37), rtol=1e-12, atol=1e-12)


def test_one_key_returns_value():
    rng = np.random.default_rng(2)
    q, k, v, qo, ko = _ragged(rng, [4], [1], 3, 8)
    o = block_attention(q, k, v, qo, ko, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(v[0], o.shape), rtol=1e-13)


def test_identical_keys_and_zero_scale_give_mean():
    rng = np.random.default_rng(3)
    q, k, v, qo, ko = _ragged(rng, [2], [6], 2, 4)
    k[:] = k[0]
    o = block_attention(q, k, v, qo, ko, 0.9)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), rtol=1e-12)
    q, k, v, qo, ko = _ragged(rng, [2], [6], 2, 4)
    o = block_attention(q, k, v, qo, ko, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0), o.shape), rtol=1e-12)


@pytest.mark.parametrize("seed", [0, 1])
def test_matches_torch_sdpa_float64(seed):
    rng = np.random.default_rng(10 + seed)
    W, L, H, dh = [5, 9, 1], [40, 13, 70], 3, 16
    q, k, v, qo, ko = _ragged(rng, W, L, H, dh)
    scale = 1.0 / math.sqrt(dh)
    o = block_attention(q, k, v, qo, ko, scale)
    for i in range(3):
        tq = torch.from_numpy(q[qo[i]:qo[i + 1]]).permute(1, 0, 2)
        tk = torch.from_numpy(k[ko[i]:ko[i + 1]]).permute(1, 0, 2)
        tv = torch.from_numpy(v[ko[i]:ko[i + 1]]).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=False, scale=scale)
        np.testing.assert_allclose(o[qo[i]:qo[i + 1]], ref.permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-12)


def test_empty_requests():
    rng = np.random.default_rng(4)
    q, k, v, qo, ko = _ragged(rng, [0, 2, 0], [3, 4, 0], 1, 2)
    o = block_attention(q, k, v, qo, ko, 1.0)
    assert o.shape == (2, 1, 2)
    assert np.all(np.isfinite(o))
