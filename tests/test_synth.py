"""Seeded input generator: determinism, bf16 rounding, and the planted structure (no GPU)."""
import numpy as np
import torch

from speculative_decoding_drafter_gb300.synth import (CONFIGS, SelectorConfig, bf16_bits_to_f32,
                                                      f32_to_bf16_bits, make_inputs)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-6, 6, 100000),
                        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 1e-40, 1.00390625, 1.01171875], np.float32)])
    x = x.astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(f32_to_bf16_bits(x), want)
    assert np.array_equal(bf16_bits_to_f32(want), torch.from_numpy(want.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_tiny_config_is_deterministic_and_shaped():
    a, b = make_inputs("tiny", 0), make_inputs("tiny", 0)
    c = CONFIGS["tiny"]
    shapes = {"hidden": (c.R, c.H), "W_vocab": (c.V, c.H), "W_sel": (c.D, c.H), "pred_cb": (c.V, c.D),
              "succ_cb": (c.V, c.D)}
    for n, s in shapes.items():
        assert a[n].shape == s and a[n].dtype == np.uint16
        assert np.array_equal(a[n], b[n])
    assert a["anchor"].shape == (c.B,) and a["anchor"].dtype == np.int32
    assert np.all((a["anchor"] >= 0) & (a["anchor"] < c.V))
    assert not np.array_equal(make_inputs("tiny", 1)["hidden"], a["hidden"])
    w = bf16_bits_to_f32(a["W_vocab"])
    assert abs(w.std() * np.sqrt(c.H) - 1.0) < 0.02
    assert abs(bf16_bits_to_f32(a["pred_cb"]).std() - 0.1) < 0.002


def test_duplicate_plant_copies_vocabulary_rows_bitwise():
    cfg = SelectorConfig("dup_small", 8, 5, 64, 2048, 8, 16, "dup_logits")
    x = make_inputs(cfg, 3)
    assert len(x["plant"]["pairs"]) == 2
    for r, v, u in x["plant"]["pairs"]:
        assert u != v
        assert np.array_equal(x["W_vocab"][u], x["W_vocab"][v])


def test_rank_boost_plant_raises_the_token():
    cfg = SelectorConfig("boost_small", 2, 4, 128, 3000, 8, 16, "rank_boost")
    x = make_inputs(cfg, 5)
    h = bf16_bits_to_f32(x["hidden"]).astype(np.float64)
    w = bf16_bits_to_f32(x["W_vocab"]).astype(np.float64)
    for r, v in zip(x["plant"]["rows"], x["plant"]["tokens"]):
        lg = w @ h[r]
        assert int(np.sum(lg > lg[v])) <= 1  # moved from rank 2..8 to the top (or next to it)


def test_scaled_rows_plant_multiplies_by_four():
    cfg = SelectorConfig("scaled_small", 4, 5, 32, 256, 4, 8, "scaled_rows")
    x = make_inputs(cfg, 2)
    base = make_inputs(SelectorConfig("plain_small", 4, 5, 32, 256, 4, 8), 2)
    rows = x["plant"]["rows"]
    assert len(rows) == 2
    assert np.array_equal(bf16_bits_to_f32(x["hidden"][rows]), 4 * bf16_bits_to_f32(base["hidden"][rows]))
    others = np.setdiff1d(np.arange(20), rows)
    assert np.array_equal(x["hidden"][others], base["hidden"][others])
