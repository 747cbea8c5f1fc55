"""CPU oracle for the DFlash2 candidate-selector head -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product path (the CUDA library
and its binding) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, float32
where the method fixes it); this module only marshals numpy arrays.  Each
step cites the passage it follows in ``oracle.c``'s header:

* ``logits``  -- LM head, float32 logits from a double sum of exact products
  ("DFlash 2: Keep Drafting Parallel", section "A Lightweight Path Selector").
* ``topk``    -- full sort by (logit desc, id asc), first k ("DFlash2 Lands in
  llama.cpp", section "What llama.cpp Actually Builds for the Selector").
* ``gate``    -- linear selector projection of the current hidden state.
* ``lattice`` -- S_t(a,b) = U_t(b) + <A(a) (.) g_t, B(b)>, packed as
  [k ids | k*k scores, predecessor-major]; the anchor is the predecessor at
  position 0.
* ``walk``    -- greedy walk from the anchor, first maximum wins.
* ``walk_sample`` -- the walk with the chosen transition's softmax confidence,
  the p_min early stop ("DFlash2 Lands in llama.cpp", section "p_min Means
  Something Different Under DFlash2") and inverse-CDF sampling from the same
  scores with given uniforms (DFlash 2 page, "A Lightweight Path Selector").
* ``dynamic_conv`` -- grouped two-tap dynamic depthwise convolution ("DFlash 2:
  Keep Drafting Parallel", section "A Lightweight Local Convolution"; "DFlash2
  Lands in llama.cpp", section "Dynamic Local Convolution").
* ``select`` / ``select_from_logits`` -- the whole path for a set of
  sequences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no FMA contraction)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(
                ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                 "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"],
                check=True,
            )
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB names an alternative build of oracle.c; the mutation tests use it to
        # load deliberately broken copies and check that the pins catch them.
        path = os.environ.get("ORACLE_LIB")
        if not path:
            path = build()
        lib = ctypes.CDLL(path)
        i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.oracle_logits.argtypes = [p, p, i64, i64, i64, p, p]
        lib.oracle_topk.argtypes = [p, i64, i64, i32, p, p]
        lib.oracle_gate.argtypes = [p, p, i64, i64, i64, p]
        lib.oracle_lattice.argtypes = [i64, i64, i32, i64, i64, p, p, p, p, p, p, p, p]
        lib.oracle_walk.argtypes = [i64, i64, i32, p, p, p]
        lib.oracle_threads.argtypes = []
        lib.oracle_set_threads.argtypes = [i32]
        lib.oracle_walk_sample.argtypes = [i64, i64, i32, p, ctypes.c_double, ctypes.c_double, p, p, p, p]
        lib.oracle_dynamic_conv.argtypes = [i64, i64, i64, i64, p, p, p, p, p, ctypes.c_double, p]
        for f in (lib.oracle_logits, lib.oracle_topk, lib.oracle_gate, lib.oracle_lattice, lib.oracle_walk,
                  lib.oracle_threads, lib.oracle_walk_sample, lib.oracle_dynamic_conv, lib.oracle_set_threads):
            f.restype = ctypes.c_int
        _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle's loops use."""
    return int(_load().oracle_threads())


def set_threads(n: int) -> int:
    """Use n OpenMP threads from now on; returns the previous count."""
    return int(_load().oracle_set_threads(int(n)))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def logits(hidden, W_vocab, want64: bool = False):
    """float32 logits [R, V] (and the unrounded double sums if ``want64``)."""
    lib = _load()
    hidden, W_vocab = _c(hidden, np.uint16), _c(W_vocab, np.uint16)
    R, H = hidden.shape
    V = W_vocab.shape[0]
    assert W_vocab.shape[1] == H
    out = np.empty((R, V), np.float32)
    out64 = np.empty((R, V), np.float64) if want64 else None
    _check(lib.oracle_logits(_ptr(hidden), _ptr(W_vocab), R, H, V, _ptr(out), _ptr(out64)), "logits")
    return (out, out64) if want64 else out


def topk(logits_f32, k: int):
    """(ids int32 [R,k], values float32 [R,k]) by (value desc, id asc)."""
    lib = _load()
    lg = _c(logits_f32, np.float32)
    R, V = lg.shape
    ids = np.empty((R, k), np.int32)
    vals = np.empty((R, k), np.float32)
    _check(lib.oracle_topk(_ptr(lg), R, V, k, _ptr(ids), _ptr(vals)), "topk")
    return ids, vals


def gate(hidden, W_sel):
    """Gate g [R, D] in double."""
    lib = _load()
    hidden, W_sel = _c(hidden, np.uint16), _c(W_sel, np.uint16)
    R, H = hidden.shape
    D = W_sel.shape[0]
    assert W_sel.shape[1] == H
    g = np.empty((R, D), np.float64)
    _check(lib.oracle_gate(_ptr(hidden), _ptr(W_sel), R, H, D, _ptr(g)), "gate")
    return g


def lattice(cand_ids, unary, g, pred_cb, succ_cb, anchor, T: int, want64: bool = False):
    """Packed float32 lattice [B*T, k + k*k] (and double scores [B*T, k, k] if ``want64``)."""
    lib = _load()
    cand_ids, unary = _c(cand_ids, np.int32), _c(unary, np.float32)
    g = _c(g, np.float64)
    pred_cb, succ_cb = _c(pred_cb, np.uint16), _c(succ_cb, np.uint16)
    anchor = _c(anchor, np.int32)
    R, k = cand_ids.shape
    B = anchor.shape[0]
    assert R == B * T
    V, D = pred_cb.shape
    out = np.empty((R, k + k * k), np.float32)
    out64 = np.empty((R, k, k), np.float64) if want64 else None
    _check(lib.oracle_lattice(B, T, k, V, D, _ptr(cand_ids), _ptr(unary), _ptr(g), _ptr(pred_cb),
                              _ptr(succ_cb), _ptr(anchor), _ptr(out), _ptr(out64)), "lattice")
    return (out, out64) if want64 else out


def walk(lattice_f32, B: int, T: int, k: int):
    """(draft ids int32 [B, T], chosen candidate index int32 [B, T])."""
    lib = _load()
    lat = _c(lattice_f32, np.float32)
    assert lat.shape == (B * T, k + k * k)
    draft = np.empty((B, T), np.int32)
    choice = np.empty((B, T), np.int32)
    _check(lib.oracle_walk(B, T, k, _ptr(lat), _ptr(draft), _ptr(choice)), "walk")
    return draft, choice


def walk_sample(lattice_f32, B: int, T: int, k: int, temperature: float = 1.0, p_min: float = 0.0, uniforms=None):
    """Walk with confidence and p_min stop; sampling when ``uniforms`` [B, T] is given.

    Returns (draft int32 [B, T] with -1 after a stop, n_draft int32 [B], confidence float64 [B, T]).
    """
    lib = _load()
    lat = _c(lattice_f32, np.float32)
    assert lat.shape == (B * T, k + k * k)
    u = None if uniforms is None else _c(uniforms, np.float32).reshape(B * T)
    draft = np.empty((B, T), np.int32)
    n = np.empty(B, np.int32)
    conf = np.empty((B, T), np.float64)
    _check(lib.oracle_walk_sample(B, T, k, _ptr(lat), float(temperature), float(p_min), _ptr(u), _ptr(draft), _ptr(n),
                                  _ptr(conf)), "walk_sample")
    return draft, n, conf


def dynamic_conv(x, x_prev, base, dyn, T: int, G: int = 16, gamma=None, eps: float = 1e-6):
    """Two-tap dynamic depthwise conv over blocks of T rows, in double: y [B*T, C] float64.

    x bf16 bits [B*T, C]; x_prev bf16 bits [B, C] or None (zeros); base bf16 bits [2, C]
    (tap 0: the position itself, tap 1: its predecessor); dyn float32 [B*T, 2, C/G];
    gamma bf16 bits [C] or None (no RMS normalisation)."""
    lib = _load()
    x = _c(x, np.uint16)
    R, C = x.shape
    B = R // T
    assert B * T == R
    xp = None if x_prev is None else _c(x_prev, np.uint16)
    base = _c(base, np.uint16)
    dyn = _c(dyn, np.float32)
    gm = None if gamma is None else _c(gamma, np.uint16)
    assert base.shape == (2, C) and dyn.shape == (R, 2, C // G)
    y = np.empty((R, C), np.float64)
    _check(lib.oracle_dynamic_conv(B, T, C, G, _ptr(x), _ptr(xp), _ptr(base), _ptr(dyn), _ptr(gm), float(eps),
                                   _ptr(y)), "dynamic_conv")
    return y


def walk_margins(lattice64, choice):
    """Per step, best minus runner-up of the double scores on the row the walk read.

    lattice64 [B*T, k, k], choice [B, T] -> margins [B, T] (inf when k == 1).
    """
    B, T = choice.shape
    k = lattice64.shape[-1]
    m = np.full((B, T), np.inf)
    for b in range(B):
        jp = 0
        for t in range(T):
            row = lattice64[b * T + t, jp]
            if k > 1:
                srt = np.sort(row)[::-1]
                m[b, t] = srt[0] - srt[1]
            jp = int(choice[b, t])
    return m


def select_from_logits(logits_f32, hidden, W_sel, pred_cb, succ_cb, anchor, k: int, T: int):
    """The whole path given float32 logits [B*T, V]; returns a dict of numpy arrays."""
    ids, vals = topk(logits_f32, k)
    g = gate(hidden, W_sel)
    lat, lat64 = lattice(ids, vals, g, pred_cb, succ_cb, anchor, T, want64=True)
    B = np.asarray(anchor).shape[0]
    draft, choice = walk(lat, B, T, k)
    return {"topk_ids": ids, "topk_vals": vals, "gate": g, "lattice": lat, "lattice64": lat64,
            "draft": draft, "choice": choice, "margins": walk_margins(lat64, choice)}


def select(hidden, W_vocab, W_sel, pred_cb, succ_cb, anchor, k: int, T: int):
    """The whole path from hidden states; also returns the float32 logits."""
    lg = logits(hidden, W_vocab)
    out = select_from_logits(lg, hidden, W_sel, pred_cb, succ_cb, anchor, k, T)
    out["logits"] = lg
    return out
