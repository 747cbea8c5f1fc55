"""Seeded synthetic inputs for the DFlash2 candidate-selector head.

This module only draws tensors.  It holds none of the selector's arithmetic
(no top-k, no gate, no lattice, no walk); the CUDA path and the CPU oracle
both consume what it returns, byte for byte.

Why synthetic: the workloads of "DFlash 2: Keep Drafting Parallel" (Tables
1-5: GSM8K, MATH-500, HumanEval, MBPP, MT-Bench on Qwen3-4B / Qwen3.5-4B /
Qwen3.8-27B / Muse Glimmer drafters) need trained drafter weights and
datasets.  Tensors with the selector head's shapes stand in for them: block
of 8 or 16 draft positions, vocabularies of ~152k-262k, selector rank 256-512,
top-16 candidates (section "A Lightweight Path Selector").

Recipe (every config):
  * hidden  [B*T, H]  ~ N(0, 1)                      -> bf16 (round to nearest even)
  * W_vocab [V, H]    ~ N(0, 1/sqrt(H))  (std)       -> bf16
  * W_sel   [D, H]    ~ N(0, 1/sqrt(H))  (std)       -> bf16
  * pred_cb [V, D]    ~ N(0, 0.1)        (std)       -> bf16
  * succ_cb [V, D]    ~ N(0, 0.1)        (std)       -> bf16
  * anchor  [B]       ~ uniform integers in [0, V)
Each tensor is drawn in float32 from its own PCG64 stream
(SeedSequence([seed, tensor_id, chunk])), so the bytes are identical on x86
and Arm and independent of thread count.  Per-config structure:
  * "rank_boost": per sequence, one seeded position gets the token at a seeded
    rank in [2, 8] raised by 2 sigma of its row's logits (hidden += 2 sigma *
    w_v / |w_v|^2 before the bf16 rounding), to exercise re-ordering.
  * "dup_logits": 5% of rows (seeded) pick their rank-rho token v
    (rho in [1, k/2]) and a partner u > v; W_vocab[u] := W_vocab[v] bitwise,
    so logit_u == logit_v exactly for every summation order that treats both
    vocabulary rows alike: this exercises the lower-id tie-break.
  * "scaled_rows": 10% of positions (seeded) are multiplied by 4 (exact in
    bf16) to sharpen their logits.
The two plants that need a row's logits to pick a token compute them here with
a float32 numpy matmul.  That is input shaping, not the method under test: the
chosen token only decides which bytes both sides receive.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
from dataclasses import dataclass

import numpy as np

__all__ = ["SelectorConfig", "CONFIGS", "make_inputs", "make_conv_inputs", "bf16_bits_to_f32", "f32_to_bf16_bits"]


@dataclass(frozen=True)
class SelectorConfig:
    """Shape of one selector-head workload: B sequences of T draft positions."""

    name: str
    B: int
    T: int
    H: int
    V: int
    k: int
    D: int
    plant: str = "none"

    @property
    def R(self) -> int:
        return self.B * self.T


CONFIGS = {
    # tiny selector: parity case the oracle finishes in well under a second
    "tiny": SelectorConfig("tiny", 1, 8, 256, 4096, 4, 64),
    # 8B-class drafter head at batch 1 (weight-streaming regime)
    "8b_b1": SelectorConfig("8b_b1", 1, 16, 4096, 151936, 8, 256, "rank_boost"),
    # 8B-class batched: 512 rows, duplicate logits for the tie-break
    "8b_b32": SelectorConfig("8b_b32", 32, 16, 4096, 151936, 16, 256, "dup_logits"),
    # 27B-class head: block of 8 (7 speculative tokens + anchor row)
    "27b_b8": SelectorConfig("27b_b8", 8, 8, 5120, 152064, 8, 256),
    # large-vocabulary, compute-bound: 1024 rows
    "large_vocab": SelectorConfig("large_vocab", 64, 16, 5376, 262144, 16, 512, "scaled_rows"),
}

_T_HIDDEN, _T_WVOCAB, _T_WSEL, _T_PRED, _T_SUCC, _T_ANCHOR, _T_PLANT = range(1, 8)
_CHUNK = 1 << 22


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(n_rows: int, n_cols: int, std: float, seed: int, tensor_id: int) -> np.ndarray:
    """[n_rows, n_cols] bf16 bits of N(0, std) float32 draws, chunked over independent streams."""
    n = n_rows * n_cols
    out = np.empty(n, dtype=np.uint16)
    std32 = np.float32(std)
    n_chunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, c])))
        x = g.standard_normal(hi - lo, dtype=np.float32)
        x *= std32
        out[lo:hi] = f32_to_bf16_bits(x)

    workers = min(n_chunks, max(1, os.cpu_count() or 1), 16)
    if workers <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with _cf.ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(n_rows, n_cols)


def _row_logits_f32(hidden_rows: np.ndarray, W: np.ndarray) -> np.ndarray:
    """float32 logits of a few hidden rows against all of W (both bf16 bits), chunked over V."""
    h = bf16_bits_to_f32(hidden_rows)
    out = np.empty((h.shape[0], W.shape[0]), dtype=np.float32)
    step = 1 << 15
    for v0 in range(0, W.shape[0], step):
        out[:, v0:v0 + step] = h @ bf16_bits_to_f32(W[v0:v0 + step]).T
    return out


def _rank_order(row: np.ndarray) -> np.ndarray:
    """Token ids of one float32 row ordered by value (desc), then id (asc)."""
    return np.lexsort((np.arange(row.shape[0]), -row.astype(np.float64)))


def make_inputs(cfg: SelectorConfig | str, seed: int = 0) -> dict:
    """Draw the seeded inputs of one config.

    Returns numpy arrays: hidden/W_vocab/W_sel/pred_cb/succ_cb as uint16 bf16
    bit patterns (row-major, shapes [R,H], [V,H], [D,H], [V,D], [V,D]) and
    anchor as int32 [B].  Also returns 'cfg' and a 'plant' record.
    """
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    B, T, H, V, k, D = cfg.B, cfg.T, cfg.H, cfg.V, cfg.k, cfg.D
    R = B * T
    w_std = 1.0 / np.sqrt(H)
    hidden = _normal_bf16(R, H, 1.0, seed, _T_HIDDEN)
    W_vocab = _normal_bf16(V, H, w_std, seed, _T_WVOCAB)
    W_sel = _normal_bf16(D, H, w_std, seed, _T_WSEL)
    pred_cb = _normal_bf16(V, D, 0.1, seed, _T_PRED)
    succ_cb = _normal_bf16(V, D, 0.1, seed, _T_SUCC)
    ga = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _T_ANCHOR])))
    anchor = ga.integers(0, V, size=B, dtype=np.int64).astype(np.int32)
    gp = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _T_PLANT])))
    plant: dict = {"kind": cfg.plant}

    if cfg.plant == "rank_boost":
        rows, toks = [], []
        for b in range(B):
            t = int(gp.integers(0, T))
            rho = int(gp.integers(2, 9))
            r = b * T + t
            lg = _row_logits_f32(hidden[r:r + 1], W_vocab)[0]
            v = int(_rank_order(lg)[rho - 1])
            sigma = float(lg.astype(np.float64).std())
            w = bf16_bits_to_f32(W_vocab[v]).astype(np.float64)
            h = bf16_bits_to_f32(hidden[r]).astype(np.float64)
            h = h + 2.0 * sigma * w / float(w @ w)
            hidden[r] = f32_to_bf16_bits(h.astype(np.float32))
            rows.append(r)
            toks.append(v)
        plant.update(rows=rows, tokens=toks)
    elif cfg.plant == "dup_logits":
        n_dup = int(round(0.05 * R))
        rows = np.sort(gp.choice(R, size=n_dup, replace=False))
        lg = _row_logits_f32(hidden[rows], W_vocab)
        pairs = []
        for q, r in enumerate(rows):
            rho = int(gp.integers(1, k // 2 + 1))
            v = int(_rank_order(lg[q])[rho - 1])
            u = int(gp.integers(v + 1, V)) if v < V - 1 else int(gp.integers(0, v))
            W_vocab[u] = W_vocab[v]
            pairs.append((int(r), v, u))
        plant.update(rows=[int(r) for r in rows], pairs=pairs)
    elif cfg.plant == "scaled_rows":
        n_sc = int(round(0.10 * R))
        rows = np.sort(gp.choice(R, size=n_sc, replace=False))
        x = bf16_bits_to_f32(hidden[rows]) * np.float32(4.0)
        hidden[rows] = f32_to_bf16_bits(x)
        plant.update(rows=[int(r) for r in rows])

    return {
        "cfg": cfg,
        "hidden": hidden,
        "W_vocab": W_vocab,
        "W_sel": W_sel,
        "pred_cb": pred_cb,
        "succ_cb": succ_cb,
        "anchor": anchor,
        "plant": plant,
    }


_T_CONV_X, _T_CONV_PREV, _T_CONV_BASE, _T_CONV_DYN, _T_CONV_GAMMA = range(21, 26)


def make_conv_inputs(B: int, T: int, C: int, G: int = 16, seed: int = 0) -> dict:
    """Seeded inputs of the dynamic local convolution of B blocks of T positions.

    x [B*T, C] and x_prev [B, C] ~ N(0, 1); base [2, C] ~ N(0, 0.5); gamma [C] ~ 1 + N(0, 0.1)
    (all bf16 bits); dyn [B*T, 2, C/G] ~ N(0, 0.1) float32 (already-projected corrections).
    """
    x = _normal_bf16(B * T, C, 1.0, seed, _T_CONV_X)
    x_prev = _normal_bf16(B, C, 1.0, seed, _T_CONV_PREV)
    base = _normal_bf16(2, C, 0.5, seed, _T_CONV_BASE)
    gg = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _T_CONV_GAMMA])))
    gamma = f32_to_bf16_bits((1.0 + 0.1 * gg.standard_normal(C)).astype(np.float32))
    gd = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, _T_CONV_DYN])))
    dyn = (0.1 * gd.standard_normal((B * T, 2, C // G), dtype=np.float32)).astype(np.float32)
    return {"x": x, "x_prev": x_prev, "base": base, "gamma": gamma, "dyn": dyn, "B": B, "T": T, "C": C, "G": G}
