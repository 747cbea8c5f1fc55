"""Pins of the CPU oracle to facts other than itself (no GPU needed).

Each test fixes one step of the selector head against a closed form, a
hand-derived example, a library routine on a special case, brute force on
tiny inputs, or an invariant the pages state.  They are chosen so that a
plausible slip in the oracle (a dropped term, a swapped codebook, a wrong
predecessor or gate row, a transposed lattice, a reversed tie-break, an
argmax turned argmin) fails at least one of them; tests/test_oracle_mutants.py
checks exactly that by compiling such slips into the oracle.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from speculative_decoding_drafter_gb300.synth import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    """float values that are exact in bf16 -> bf16 bits (asserts exactness)."""
    a = np.asarray(x, dtype=np.float32)
    bits = f32_to_bf16_bits(a)
    assert np.array_equal(bf16_bits_to_f32(bits), a), "fixture value is not exact in bf16"
    return bits


def rand_bf16(rng, shape, std=1.0):
    return f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))


def nearest_f32(q: Fraction) -> np.float32:
    """Correctly rounded float32 of an exact rational (nearest, ties to even)."""
    f = np.float32(float(q))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]

    def key(c):
        return (abs(Fraction(float(c)) - q), int(np.array(c, dtype=np.float32).view(np.uint32)) & 1)

    return min(cands, key=key)


# ---------------------------------------------------------------- worked example


def load_worked_example():
    with open(os.path.join(GOLDEN, "worked_example.json")) as fh:
        ex = json.load(fh)
    d = ex["dims"]
    inp = {n: bf(ex[n]) for n in ("hidden", "W_vocab", "W_sel", "pred_cb", "succ_cb")}
    inp["anchor"] = np.asarray(ex["anchor"], np.int32)
    return ex, d, inp


def test_worked_example_every_step():
    ex, d, inp = load_worked_example()
    out = oracle.select(inp["hidden"], inp["W_vocab"], inp["W_sel"], inp["pred_cb"], inp["succ_cb"],
                        inp["anchor"], d["k"], d["T"])
    e = ex["expected"]
    assert np.array_equal(out["logits"], np.asarray(e["logits"], np.float32))
    assert np.array_equal(out["topk_ids"], np.asarray(e["topk_ids"], np.int32))
    assert np.array_equal(out["topk_vals"], np.asarray(e["topk_vals"], np.float32))
    assert np.array_equal(out["gate"], np.asarray(e["gate"], np.float64))
    assert np.array_equal(out["lattice"], np.asarray(e["lattice"], np.float32))
    assert np.array_equal(out["draft"], np.asarray(e["draft"], np.int32))
    # plain DFlash (independent top-1 per position) differs: the selector re-orders
    assert np.array_equal(out["topk_ids"][:, 0][None, :], np.asarray(e["dflash1_top1"], np.int32))
    assert not np.array_equal(out["draft"], np.asarray(e["dflash1_top1"], np.int32))


# ---------------------------------------------------------------- step 1: logits


def test_logits_equal_correctly_rounded_exact_sum():
    rng = np.random.default_rng(11)
    R, H, V = 3, 24, 40
    hid = rand_bf16(rng, (R, H))
    W = rand_bf16(rng, (V, H), 1 / np.sqrt(H))
    got = oracle.logits(hid, W)
    hf, wf = bf16_bits_to_f32(hid), bf16_bits_to_f32(W)
    for r in range(R):
        for v in range(V):
            exact = sum(Fraction(float(hf[r, h])) * Fraction(float(wf[v, h])) for h in range(H))
            assert got[r, v] == nearest_f32(exact), (r, v)


def test_logits_one_hot_vocab_rows_select_hidden_entries():
    rng = np.random.default_rng(12)
    R, H, V = 4, 16, 48
    hid = rand_bf16(rng, (R, H))
    W = np.zeros((V, H), np.float32)
    W[np.arange(V), np.arange(V) % H] = 1.0
    got = oracle.logits(hid, bf(W))
    want = bf16_bits_to_f32(hid)[:, np.arange(V) % H]
    assert np.array_equal(got, want)


# ---------------------------------------------------------------- step 2: top-k


def test_topk_equals_stable_library_sort_with_ties_and_signed_zeros():
    rng = np.random.default_rng(13)
    R, V, k = 6, 300, 12
    lg = rng.standard_normal((R, V)).astype(np.float32)
    lg[0, 7] = lg[0, 3]  # exact duplicates: lower id must come first
    lg[1, 50:60] = 5.0  # a run of equal maxima
    lg[2, :] = -3.0 - np.abs(lg[2])  # row 2: all negative except two zeros
    lg[2, 20], lg[2, 10] = np.float32(0.0), np.float32(-0.0)  # -0 == +0 is a tie: id 10 first
    ids, vals = oracle.topk(lg, k)
    for r in range(R):
        order = np.lexsort((np.arange(V), -lg[r].astype(np.float64)))  # stable: ties by id
        assert np.array_equal(ids[r], order[:k].astype(np.int32))
        assert np.array_equal(vals[r], lg[r, order[:k]])
    assert list(ids[1, :10]) == list(range(50, 60))
    assert list(ids[2, :2]) == [10, 20]


def test_topk_with_k_equal_to_V_is_the_full_order():
    rng = np.random.default_rng(14)
    V = 64
    lg = np.round(rng.standard_normal((2, V)) * 2).astype(np.float32)  # many ties
    ids, vals = oracle.topk(lg, V)
    for r in range(2):
        want = sorted(range(V), key=lambda v: (-float(lg[r, v]), v))
        assert list(ids[r]) == want


def test_topk_rejects_non_finite_logits():
    lg = np.zeros((1, 8), np.float32)
    lg[0, 3] = np.nan
    with pytest.raises(ValueError):
        oracle.topk(lg, 2)


# ---------------------------------------------------------------- step 3: gate


def test_gate_of_identity_projection_is_the_hidden_prefix():
    rng = np.random.default_rng(15)
    R, H, D = 5, 32, 8
    hid = rand_bf16(rng, (R, H))
    Wsel = np.zeros((D, H), np.float32)
    Wsel[np.arange(D), np.arange(D)] = 1.0
    g = oracle.gate(hid, bf(Wsel))
    assert np.array_equal(g, bf16_bits_to_f32(hid)[:, :D].astype(np.float64))


def test_gate_is_linear_in_the_projection():
    rng = np.random.default_rng(16)
    hid = rand_bf16(rng, (3, 40))
    Wsel = rand_bf16(rng, (8, 40), 0.2)
    W2 = f32_to_bf16_bits(bf16_bits_to_f32(Wsel) * np.float32(2.0))  # exact
    assert np.array_equal(oracle.gate(hid, W2), 2.0 * oracle.gate(hid, Wsel))


# ---------------------------------------------------------------- steps 4-5: lattice


def _lattice_case(rng, B=2, T=3, k=3, V=20, D=6):
    cand = np.stack([rng.choice(V, size=k, replace=False) for _ in range(B * T)]).astype(np.int32)
    U = rng.standard_normal((B * T, k)).astype(np.float32)
    g = rng.standard_normal((B * T, D))
    anchor = rng.integers(0, V, size=B).astype(np.int32)
    return cand, U, g, anchor


def test_lattice_with_zero_codebook_is_the_unary_on_every_predecessor_row():
    rng = np.random.default_rng(17)
    B, T, k, V, D = 2, 4, 3, 20, 6
    cand, U, g, anchor = _lattice_case(rng, B, T, k, V, D)
    succ = rand_bf16(rng, (V, D))
    for pred, sc in ((np.zeros((V, D), np.uint16), succ), (succ, np.zeros((V, D), np.uint16))):
        lat = oracle.lattice(cand, U, g, pred, sc, anchor, T)
        assert np.array_equal(lat[:, :k], cand.astype(np.float32))
        scores = lat[:, k:].reshape(B * T, k, k)
        assert np.array_equal(scores, np.broadcast_to(U[:, None, :], scores.shape))


def test_lattice_one_hot_codebooks_closed_form():
    """A(a) = e_alpha(a), B(b) = 2 e_beta(b): pairwise = 2 g[r, alpha(prev)] [alpha(prev) == beta(cand)]."""
    rng = np.random.default_rng(18)
    B, T, k, V, D = 3, 4, 4, 12, 5
    cand, U, g, anchor = _lattice_case(rng, B, T, k, V, D)
    g = np.round(g * 8) / 8  # dyadic: every score exact in float32
    alpha = (np.arange(V) * 3 + 1) % D
    beta = (np.arange(V) * 2) % D
    pred = np.zeros((V, D), np.float32)
    pred[np.arange(V), alpha] = 1.0
    succ = np.zeros((V, D), np.float32)
    succ[np.arange(V), beta] = 2.0
    lat = oracle.lattice(cand, U, g, bf(pred), bf(succ), anchor, T)
    for b in range(B):
        for t in range(T):
            r = b * T + t
            for i in range(k):
                prev = anchor[b] if t == 0 else cand[r - 1, i]
                for j in range(k):
                    c = cand[r, j]
                    want = np.float32(float(U[r, j]) + (2.0 * g[r, alpha[prev]] if alpha[prev] == beta[c] else 0.0))
                    assert lat[r, k + i * k + j] == want, (b, t, i, j)


def test_lattice_first_position_rows_are_identical_and_anchor_conditioned():
    rng = np.random.default_rng(19)
    B, T, k, V, D = 2, 3, 4, 30, 8
    cand, U, g, anchor = _lattice_case(rng, B, T, k, V, D)
    pred = rand_bf16(rng, (V, D), 0.5)
    succ = rand_bf16(rng, (V, D), 0.5)
    lat = oracle.lattice(cand, U, g, pred, succ, anchor, T)
    for b in range(B):
        rows = lat[b * T, k:].reshape(k, k)
        assert np.all(rows == rows[0])
        # swapping the anchor for another token changes position 0 only
        a2 = anchor.copy()
        a2[b] = (anchor[b] + 1) % V
        lat2 = oracle.lattice(cand, U, g, pred, succ, a2, T)
        assert not np.array_equal(lat2[b * T], lat[b * T])
        mask = np.ones(B * T, bool)
        mask[b * T] = False
        assert np.array_equal(lat2[mask], lat[mask])


# ---------------------------------------------------------------- step 6: walk


def test_walk_follows_a_designed_lattice():
    """S[t][i][j] = -|j - f_t(i)|: the greedy path is j_t = f_t(j_{t-1}), with j_0 = c."""
    B, T, k = 2, 6, 5
    f = lambda t, i, b: (2 * i + t + b) % k  # noqa: E731
    c0 = [3, 1]
    lat = np.zeros((B * T, k + k * k), np.float32)
    want = np.zeros((B, T), np.int32)
    for b in range(B):
        jp = None
        for t in range(T):
            r = b * T + t
            lat[r, :k] = 1000 * b + 10 * t + np.arange(k)
            for i in range(k):
                target = c0[b] if t == 0 else f(t, i, b)
                lat[r, k + i * k: k + (i + 1) * k] = -np.abs(np.arange(k) - target)
            j = c0[b] if t == 0 else f(t, jp, b)
            want[b, t] = 1000 * b + 10 * t + j
            jp = j
    draft, choice = oracle.walk(lat, B, T, k)
    assert np.array_equal(draft, want)


def test_walk_first_maximum_wins_on_ties():
    k = 4
    lat = np.zeros((2, k + k * k), np.float32)
    lat[:, :k] = [[10, 11, 12, 13], [20, 21, 22, 23]]
    lat[0, k:] = np.tile([0.0, 2.0, 2.0, 1.0], k)
    lat[1, k + 1 * k: k + 2 * k] = [5.0, 1.0, 5.0, 5.0]
    draft, choice = oracle.walk(lat, 1, 2, k)
    assert draft.tolist() == [[11, 20]]


def test_walk_against_brute_force_over_all_paths():
    """Greedy path score <= the best of all k^T paths; equal when the pairwise term is zero."""
    rng = np.random.default_rng(20)
    B, T, k, V, D = 3, 4, 3, 16, 4
    hid = rand_bf16(rng, (B * T, 8))
    W = rand_bf16(rng, (V, 8))
    Wsel = rand_bf16(rng, (D, 8), 0.5)
    anchor = rng.integers(0, V, B).astype(np.int32)
    for zero in (False, True):
        pred = np.zeros((V, D), np.uint16) if zero else rand_bf16(rng, (V, D), 0.7)
        succ = rand_bf16(rng, (V, D), 0.7)
        out = oracle.select(hid, W, Wsel, pred, succ, anchor, k, T)
        S = out["lattice64"]
        for b in range(B):
            def score(path):
                s = S[b * T, 0, path[0]]
                for t in range(1, T):
                    s += S[b * T + t, path[t - 1], path[t]]
                return s
            best = max(score(p) for p in itertools.product(range(k), repeat=T))
            greedy = score(out["choice"][b])
            assert greedy <= best + 1e-12
            if zero:
                assert abs(greedy - best) < 1e-12
                assert np.all(out["choice"][b] == 0)


# ---------------------------------------------------------------- whole-path invariants


def _tiny_inputs(rng, B=2, T=5, H=32, V=64, D=8, dup=True):
    hid = rand_bf16(rng, (B * T, H))
    W = rand_bf16(rng, (V, H), 1 / np.sqrt(H))
    if dup:
        W[9] = W[4]  # exact tie between ids 4 and 9
    Wsel = rand_bf16(rng, (D, H), 1 / np.sqrt(H))
    pred = rand_bf16(rng, (V, D), 0.3)
    succ = rand_bf16(rng, (V, D), 0.3)
    anchor = rng.integers(0, V, B).astype(np.int32)
    return hid, W, Wsel, pred, succ, anchor


def test_zeroed_codebooks_reduce_the_walk_to_per_position_top1():
    """Plain DFlash keeps one independent top-1 token per position (llama.cpp page, mental model)."""
    rng = np.random.default_rng(21)
    B, T, k = 3, 5, 4
    hid, W, Wsel, pred, succ, anchor = _tiny_inputs(rng, B, T)
    z = np.zeros_like(pred)
    lg = oracle.logits(hid, W)
    top1 = np.array([np.lexsort((np.arange(lg.shape[1]), -lg[r].astype(np.float64)))[0]
                     for r in range(B * T)]).reshape(B, T)
    for p, s in ((z, succ), (pred, z), (z, z)):
        out = oracle.select(hid, W, Wsel, p, s, anchor, k, T)
        assert np.array_equal(out["draft"], top1)


def test_k_equal_one_is_top1():
    rng = np.random.default_rng(22)
    B, T = 2, 4
    hid, W, Wsel, pred, succ, anchor = _tiny_inputs(rng, B, T)
    out = oracle.select(hid, W, Wsel, pred, succ, anchor, 1, T)
    lg = out["logits"]
    want = np.array([np.lexsort((np.arange(lg.shape[1]), -lg[r].astype(np.float64)))[0]
                     for r in range(B * T)]).reshape(B, T)
    assert np.array_equal(out["draft"], want)
    assert out["lattice"].shape == (B * T, 2)


def test_adding_a_per_position_constant_to_the_logits_keeps_the_draft():
    rng = np.random.default_rng(23)
    B, T, k = 2, 5, 4
    hid, W, Wsel, pred, succ, anchor = _tiny_inputs(rng, B, T)
    lg = oracle.logits(hid, W)
    base = oracle.select_from_logits(lg, hid, Wsel, pred, succ, anchor, k, T)
    shift = np.float32(64.0) * np.arange(1, B * T + 1, dtype=np.float32)[:, None]  # exact in float32
    moved = oracle.select_from_logits(lg + shift, hid, Wsel, pred, succ, anchor, k, T)
    assert np.array_equal(base["topk_ids"], moved["topk_ids"])
    assert np.array_equal(base["draft"], moved["draft"])


def test_sequences_are_block_local():
    rng = np.random.default_rng(24)
    B, T, k = 4, 3, 3
    hid, W, Wsel, pred, succ, anchor = _tiny_inputs(rng, B, T)
    out = oracle.select(hid, W, Wsel, pred, succ, anchor, k, T)
    perm = np.array([2, 0, 3, 1])
    rows = (perm[:, None] * T + np.arange(T)[None, :]).reshape(-1)
    out2 = oracle.select(hid[rows], W, Wsel, pred, succ, anchor[perm], k, T)
    assert np.array_equal(out2["draft"], out["draft"][perm])
    assert np.array_equal(out2["lattice"], out["lattice"][rows])


# ---------------------------------------------------------------- step 7: confidence, p_min, sampling


def _rows_lattice(scores_per_step, ids_per_step, k):
    """One sequence whose every predecessor row at step t holds scores_per_step[t]."""
    T = len(scores_per_step)
    lat = np.zeros((T, k + k * k), np.float32)
    for t in range(T):
        lat[t, :k] = ids_per_step[t]
        lat[t, k:] = np.tile(np.asarray(scores_per_step[t], np.float32), k)
    return lat


def test_greedy_confidence_of_two_candidates_is_the_logistic_function():
    import math

    for s0, s1, tau in ((1.5, 0.25, 1.0), (-2.0, 3.0, 0.5), (0.0, 0.0, 2.0)):
        lat = _rows_lattice([[s0, s1]], [[7, 9]], 2)
        draft, n, conf = oracle.walk_sample(lat, 1, 1, 2, temperature=tau)
        pick = 0 if s0 >= s1 else 1
        want = 1.0 / (1.0 + math.exp(-abs(np.float32(s0) - np.float32(s1)) / tau))
        assert draft[0, 0] == [7, 9][pick]
        assert conf[0, 0] == pytest.approx(want, rel=1e-12)
        assert n[0] == 1


def test_sampling_follows_the_inverse_cdf_of_a_designed_row():
    # softmax(log p) = p: cumulative 0.1, 0.3, 0.6, 1.0
    row = np.log(np.array([0.1, 0.2, 0.3, 0.4])).astype(np.float32)
    for u, want in ((0.05, 0), (0.15, 1), (0.35, 2), (0.95, 3), (0.0, 0), (0.999, 3)):
        lat = _rows_lattice([row], [[10, 11, 12, 13]], 4)
        draft, n, conf = oracle.walk_sample(lat, 1, 1, 4, uniforms=np.array([[u]], np.float32))
        assert draft[0, 0] == 10 + want, u


def test_sampling_frequencies_match_the_softmax():
    from scipy.special import softmax

    rng = np.random.default_rng(31)
    k, n_draws, tau = 6, 20000, 0.7
    row = rng.standard_normal(k).astype(np.float32)
    lat = np.tile(_rows_lattice([row], [np.arange(k)], k), (n_draws, 1))  # n_draws sequences of one step
    u = rng.random((n_draws, 1)).astype(np.float32)
    draft, n, conf = oracle.walk_sample(lat, n_draws, 1, k, temperature=tau, uniforms=u)
    p = softmax(row.astype(np.float64) / tau)
    freq = np.bincount(draft[:, 0], minlength=k) / n_draws
    assert np.all(np.abs(freq - p) <= 4 * np.sqrt(p * (1 - p) / n_draws) + 1e-9)
    assert np.allclose(conf[:, 0], p[draft[:, 0]])


def test_p_min_stops_the_walk_where_confidence_first_drops():
    k, T = 3, 5
    sharp, flat = [4.0, 0.0, 0.0], [0.1, 0.0, 0.05]
    steps = [sharp, sharp, sharp, flat, sharp]
    lat = _rows_lattice(steps, [[100 + 10 * t + j for j in range(k)] for t in range(T)], k)
    base, _ = oracle.walk(lat, 1, T, k)
    draft, n, conf = oracle.walk_sample(lat, 1, T, k, p_min=0.5)
    assert n[0] == 3
    assert draft[0, :3].tolist() == base[0, :3].tolist()
    assert draft[0, 3:].tolist() == [-1, -1]
    assert conf[0, 3] < 0.5 and conf[0, 4] == 0.0
    d0, n0, _ = oracle.walk_sample(lat, 1, T, k, p_min=0.0)
    assert n0[0] == T and np.array_equal(d0, base)
    d1, n1, _ = oracle.walk_sample(lat, 1, T, k, p_min=1.01)
    assert n1[0] == 0 and np.all(d1 == -1)


def test_sampling_at_vanishing_temperature_is_greedy_and_shift_invariant():
    rng = np.random.default_rng(32)
    B, T, k = 3, 6, 5
    lat = np.zeros((B * T, k + k * k), np.float32)
    lat[:, :k] = np.arange(B * T * k).reshape(B * T, k)
    lat[:, k:] = (np.round(rng.standard_normal((B * T, k * k)) * 64) / 64).astype(np.float32)  # dyadic
    for b in range(B):
        lat[b * T, k:] = np.tile(lat[b * T, k:2 * k], k)
    greedy, _ = oracle.walk(lat, B, T, k)
    u = rng.random((B, T)).astype(np.float32)
    cold, n, _ = oracle.walk_sample(lat, B, T, k, temperature=1e-6, uniforms=u)
    assert np.array_equal(cold, greedy)
    shifted = lat.copy()
    shifted[:, k:] += np.float32(8.0)  # exact: the scores are multiples of 1/64 below 16
    a = oracle.walk_sample(lat, B, T, k, temperature=0.9, uniforms=u)
    b = oracle.walk_sample(shifted, B, T, k, temperature=0.9, uniforms=u)
    assert np.array_equal(a[0], b[0]) and np.allclose(a[2], b[2], rtol=1e-12)


# ---------------------------------------------------------------- dynamic local convolution


def _conv_inputs(rng, B, T, C, G, with_prev=True):
    x = rand_bf16(rng, (B * T, C))
    xp = rand_bf16(rng, (B, C)) if with_prev else None
    base = rand_bf16(rng, (2, C), 0.5)
    dyn = (rng.standard_normal((B * T, 2, C // G)) * 0.1).astype(np.float32)
    return x, xp, base, dyn


def test_conv_identity_and_shift_taps():
    rng = np.random.default_rng(41)
    B, T, C, G = 3, 5, 32, 16
    x, xp, _, _ = _conv_inputs(rng, B, T, C, G)
    zero = np.zeros((B * T, 2, C // G), np.float32)
    xf, xpf = bf16_bits_to_f32(x).astype(np.float64), bf16_bits_to_f32(xp).astype(np.float64)
    ident = bf(np.stack([np.ones(C), np.zeros(C)]))
    assert np.array_equal(oracle.dynamic_conv(x, xp, ident, zero, T, G), xf)
    shift = bf(np.stack([np.zeros(C), np.ones(C)]))
    y = oracle.dynamic_conv(x, xp, shift, zero, T, G)
    for b in range(B):
        assert np.array_equal(y[b * T], xpf[b])  # position 0 reads the last verified token
        assert np.array_equal(y[b * T + 1:(b + 1) * T], xf[b * T:(b + 1) * T - 1])  # never the previous block
    y0 = oracle.dynamic_conv(x, None, shift, zero, T, G)
    assert np.all(y0[::T] == 0.0)


def test_conv_dynamic_correction_is_shared_by_each_group_of_channels():
    B, T, C, G = 2, 3, 48, 16
    x = bf(np.ones((B * T, C)))
    xp = bf(np.ones((B, C)))
    base = bf(np.zeros((2, C)))
    dyn = np.arange(B * T * 2 * (C // G), dtype=np.float32).reshape(B * T, 2, C // G)
    y = oracle.dynamic_conv(x, xp, base, dyn, T, G)
    for r in range(B * T):
        for c in range(C):
            assert y[r, c] == dyn[r, 0, c // G] + dyn[r, 1, c // G]


def test_conv_tap_weights_combine_base_and_correction():
    B, T, C, G = 1, 2, 16, 16
    x = bf(np.full((B * T, C), 2.0))
    xp = bf(np.full((B, C), 3.0))
    base = bf(np.stack([np.full(C, 0.5), np.full(C, 0.25)]))
    dyn = np.zeros((B * T, 2, 1), np.float32)
    dyn[:, 0, 0], dyn[:, 1, 0] = 0.5, -0.25
    y = oracle.dynamic_conv(x, xp, base, dyn, T, G)
    # t=0: (0.5+0.5)*2 + (0.25-0.25)*3 = 2 ; t=1: 1*2 + 0*2 = 2
    assert np.all(y == 2.0)
    dyn[:, 1, 0] = 0.75
    y = oracle.dynamic_conv(x, xp, base, dyn, T, G)
    assert np.all(y[0] == 2.0 + 1.0 * 3.0) and np.all(y[1] == 2.0 + 1.0 * 2.0)


def test_conv_rms_normalisation_is_scale_invariant_and_closed_form():
    rng = np.random.default_rng(42)
    B, T, C, G = 2, 4, 64, 16
    x, xp, base, dyn = _conv_inputs(rng, B, T, C, G)
    gamma = bf(np.ones(C))
    y1 = oracle.dynamic_conv(x, xp, base, dyn, T, G, gamma=gamma, eps=0.0)
    x4 = f32_to_bf16_bits(bf16_bits_to_f32(x) * np.float32(4.0))
    xp4 = f32_to_bf16_bits(bf16_bits_to_f32(xp) * np.float32(4.0))
    assert np.allclose(oracle.dynamic_conv(x4, xp4, base, dyn, T, G, gamma=gamma, eps=0.0), y1, rtol=1e-13, atol=0)
    # a constant row a normalises to sign(a) * gamma
    xc = bf(np.full((B * T, C), -3.0))
    ident = bf(np.stack([np.ones(C), np.zeros(C)]))
    g2 = bf(np.full(C, 2.0))
    y = oracle.dynamic_conv(xc, None, ident, np.zeros_like(dyn), T, G, gamma=g2, eps=0.0)
    assert np.allclose(y, -2.0, rtol=1e-15)
