"""The whole-step oracle and the seeded workload generator (CPU only)."""

import numpy as np
import pytest

import oracle
from workloads import (bf16_bits_to_f32, f32_to_bf16_bits, make_step_inputs,
                       step_config)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3, 65504.0], np.float32)
    b = f32_to_bf16_bits(x)
    back = bf16_bits_to_f32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: even mantissa (1.0) wins
    assert back[1] == np.float32(1.0)
    assert back[2] == np.float32(1.0078125)
    assert back[0] == 1.0 and back[3] == -2.5
    rel = np.abs(back - x) / np.abs(x)
    assert (rel <= 2.0 ** -8).all()         # half an ulp of an 8-bit significand


def test_generator_is_deterministic_and_shaped():
    a = step_config("tiny", seed=3)
    b = step_config("tiny", seed=3)
    for key in ("q", "k", "v", "w_head", "emb", "hidden", "mask", "prev", "credit"):
        assert np.array_equal(a[key], b[key])
    assert a["R"] == 16 and a["mask"].sum() == 16
    assert a["q"].shape == (32, 4, 64) and a["k"].shape == (160, 4, 64)
    assert list(a["row_pos"]) == sorted(a["row_pos"])
    c = step_config("tiny", seed=4)
    assert not np.array_equal(a["q"], c["q"])


def test_ragged_batch_offsets():
    inp = make_step_inputs(B=16, H=2, dh=64, V=300, blk=32, P_range=(256, 1024),
                           vl=32, vr=32, block_index=[i % 8 for i in range(16)])
    W = np.diff(inp["q_off"])
    L = np.diff(inp["kv_off"])
    assert all(256 <= p <= 1024 for p in inp["P"])
    assert list(W) == [32 + 32 + min(32, 224 - 32 * (i % 8)) for i in range(16)]
    assert list(L - W) == inp["P"]
    assert inp["R"] == 16 * 32


def test_tiny_step_oracle_runs_and_keeps_invariants():
    inp = step_config("tiny")
    res = oracle.denoise_step(inp)
    com = res["commit"]
    assert res["attn"].shape == (32, 4, 64)
    assert com["n_commit"][0] >= 1
    assert np.array_equal(com["mask"], inp["mask"] & ~com["selected"])
    assert ((com["tokens"] == inp["tokens"]) | com["selected"]).all()
    # planted rows: the argmax is the planted token whenever c is large
    big = inp["c"] >= np.quantile(inp["c"], 0.5)
    assert (res["head"]["argmax"][big] == inp["planted"][big]).mean() > 0.5


def test_literal_configs_only_fall_back():
    """With the literal planted-row recipe no confidence reaches tau."""
    inp = step_config("tiny")
    res = oracle.denoise_step(inp, with_attention=False)
    assert res["head"]["conf"].max() < 0.9
    assert res["commit"]["fallback"].all()
    assert res["commit"]["n_commit"].tolist() == [1]


def test_calibrated_variant_reaches_thresholds():
    inp = step_config("tiny", cal=True, seed=1)
    res = oracle.denoise_step(inp, with_attention=False)
    assert (res["head"]["conf"] >= 0.9).any()
    assert res["commit"]["n_commit"][0] >= 1
