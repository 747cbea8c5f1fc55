"""The C-ABI library builds, loads, exports every declared symbol and rejects bad
arguments on the host before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from speculative_decoding_drafter_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash2.h")

DF2_OK, DF2_ERR_INVALID_ARG, DF2_ERR_UNSUPPORTED, DF2_ERR_WORKSPACE = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    from speculative_decoding_drafter_gb300 import dflash2

    return dflash2.library()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DF2_API\s+[\w\s\*]*?\b(dflash2_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), f"{n} declared in dflash2.h but not exported"
    from speculative_decoding_drafter_gb300 import dflash2

    assert sorted(dflash2.EXPORTED_SYMBOLS) == names


def test_version_and_status_strings(lib):
    from speculative_decoding_drafter_gb300 import dflash2

    assert dflash2.dflash2_version() == 300
    for s in range(6):
        assert len(dflash2.dflash2_status_string(s)) >= 2
    assert dflash2.dflash2_status_string(99) == "unknown status"


def dims(B=1, T=16, H=4096, V=151936, k=8, D=256):
    from speculative_decoding_drafter_gb300.dflash2 import Dims

    return Dims(B, T, H, V, k, D)


def test_workspace_bytes_and_dimension_limits(lib):
    from speculative_decoding_drafter_gb300.dflash2 import dflash2_workspace_bytes

    n = dflash2_workspace_bytes(dims())
    R, kp = 16, 8
    assert n >= 256 + 256 + R * 256 * kp * 8 + R * 8 * 4 + R * 256 * 4
    assert n % 256 == 0
    for bad in (dims(k=0), dims(k=33), dims(V=4, k=8), dims(H=4100), dims(D=12), dims(D=2048), dims(B=0),
                dims(T=0), dims(V=1 << 24), dims(B=1 << 16, T=32)):
        assert dflash2_workspace_bytes(bad) == 0, bad


def _select(lib, d, ptrs, ws=0x100000, ws_bytes=1 << 40):
    names = ["hidden", "W_vocab", "W_sel", "pred_cb", "succ_cb", "anchor", "lattice", "draft"]
    p = {n: ptrs.get(n, 0x200000 + 0x1000 * i) for i, n in enumerate(names)}
    return lib.dflash2_select(ctypes.byref(d), p["hidden"], p["W_vocab"], p["W_sel"], p["pred_cb"], p["succ_cb"],
                              p["anchor"], p["lattice"], p["draft"], None, None, None, ws, ws_bytes, None)


def test_select_rejects_bad_arguments_before_any_cuda_call(lib):
    # Pointer values below are never dereferenced: every case fails validation first.
    assert _select(lib, dims(k=33), {}) == DF2_ERR_UNSUPPORTED
    assert _select(lib, dims(k=0), {}) == DF2_ERR_INVALID_ARG
    assert _select(lib, dims(V=4, k=8), {}) == DF2_ERR_INVALID_ARG
    assert _select(lib, dims(H=4100), {}) == DF2_ERR_UNSUPPORTED
    assert _select(lib, dims(), {"hidden": 0}) == DF2_ERR_INVALID_ARG
    assert _select(lib, dims(), {"W_vocab": 0x200008}) == DF2_ERR_INVALID_ARG  # not 16-byte aligned
    assert _select(lib, dims(), {"anchor": 0x200002}) == DF2_ERR_INVALID_ARG
    assert _select(lib, dims(), {}, ws=0) == DF2_ERR_WORKSPACE
    assert _select(lib, dims(), {}, ws=0x100010) == DF2_ERR_WORKSPACE  # not 256-byte aligned
    assert _select(lib, dims(), {}, ws_bytes=1024) == DF2_ERR_WORKSPACE
    assert lib.dflash2_select(None, 0, 0, 0, 0, 0, 0, 0, 0, None, None, None, 0, 0, None) == DF2_ERR_INVALID_ARG


def test_select_walk_rejects_bad_options_before_any_cuda_call(lib):
    # Pointer values below are never dereferenced: every case fails validation first.
    from speculative_decoding_drafter_gb300.dflash2 import WalkOpts

    names = ["hidden", "W_vocab", "W_sel", "pred_cb", "succ_cb", "anchor", "lattice", "draft"]
    p = [0x200000 + 0x1000 * i for i in range(len(names))]

    def call(opts, d=None, ws=0x100000):
        d = d or dims()
        return lib.dflash2_select_walk(ctypes.byref(d), None if opts is None else ctypes.byref(opts), *p, None, None,
                                       None, ws, 1 << 40, None)

    assert call(WalkOpts(0.0, 0.5, None, None, None)) == DF2_ERR_INVALID_ARG  # temperature must be > 0
    assert call(WalkOpts(float("inf"), 0.5, None, None, None)) == DF2_ERR_INVALID_ARG
    assert call(WalkOpts(1.0, float("nan"), None, None, None)) == DF2_ERR_INVALID_ARG
    assert call(WalkOpts(1.0, 0.5, 0x3002, None, None)) == DF2_ERR_INVALID_ARG  # uniforms not 4-byte aligned
    assert call(WalkOpts(1.0, 0.5, None, 0x3001, None)) == DF2_ERR_INVALID_ARG
    assert call(WalkOpts(1.0, 0.5, None, None, 0x3003)) == DF2_ERR_INVALID_ARG
    assert call(WalkOpts(1.0, 0.5, None, None, None), d=dims(k=33)) == DF2_ERR_UNSUPPORTED
    assert call(WalkOpts(1.0, 0.5, None, None, None), ws=0x100010) == DF2_ERR_WORKSPACE
    assert call(None, ws=0) == DF2_ERR_WORKSPACE  # NULL options: dflash2_select's checks


def test_stage_entry_points_reject_bad_arguments(lib):
    d = dims()
    assert lib.dflash2_walk(ctypes.byref(d), None, 0x1000, None) == DF2_ERR_INVALID_ARG
    assert lib.dflash2_lattice(ctypes.byref(d), 0x1000, 0x2000, 0x3004, 0x4000, 0x5000, 0x6000, 0x7000,
                               None) == DF2_ERR_INVALID_ARG  # gate not 16-byte aligned
    assert lib.dflash2_topk(ctypes.byref(dims(k=40)), 0x1000, 0x2000, 0x3000, 0x100000, 1 << 40,
                            None) == DF2_ERR_UNSUPPORTED
    assert lib.dflash2_gate(ctypes.byref(d), 0x1000, 0x2000, 0x3000, 0x100000, 16, None) == DF2_ERR_WORKSPACE
    assert lib.dflash2_lm_head_logits(ctypes.byref(d), 0x1008, 0x2000, 0x3000, 0x100000, 1 << 40,
                                      None) == DF2_ERR_INVALID_ARG
    assert lib.dflash2_check_device_status(None, 0, None) == DF2_ERR_WORKSPACE
    assert lib.dflash2_walk_sample(ctypes.byref(d), 0x1000, 0.0, 0.5, None, 0x2000, None, None,
                                   None) == DF2_ERR_INVALID_ARG  # temperature must be > 0
    assert lib.dflash2_walk_sample(ctypes.byref(d), 0x1000, float("inf"), 0.5, None, 0x2000, None, None,
                                   None) == DF2_ERR_INVALID_ARG
    assert lib.dflash2_walk_sample(ctypes.byref(d), 0x1000, 1.0, float("nan"), None, 0x2000, None, None,
                                   None) == DF2_ERR_INVALID_ARG
    assert lib.dflash2_walk_sample(ctypes.byref(d), None, 1.0, 0.5, None, 0x2000, None, None,
                                   None) == DF2_ERR_INVALID_ARG
    from speculative_decoding_drafter_gb300.dflash2 import ConvDims

    good = (0x1000, None, 0x2000, 0x3000, None, 1e-6, 0x4000, None)
    assert lib.dflash2_dynamic_conv(ctypes.byref(ConvDims(2, 4, 40, 16)), *good) == DF2_ERR_INVALID_ARG  # C % G
    assert lib.dflash2_dynamic_conv(ctypes.byref(ConvDims(2, 4, 48, 12)), *good) == DF2_ERR_UNSUPPORTED  # G % 8
    assert lib.dflash2_dynamic_conv(ctypes.byref(ConvDims(2, 4, 16384, 16)), *good) == DF2_ERR_UNSUPPORTED
    assert lib.dflash2_dynamic_conv(ctypes.byref(ConvDims(2, 4, 64, 16)), 0x1008, None, 0x2000, 0x3000, None, 1e-6,
                                    0x4000, None) == DF2_ERR_INVALID_ARG  # x not 16-byte aligned
    assert lib.dflash2_dynamic_conv(ctypes.byref(ConvDims(2, 4, 64, 16)), 0x1000, None, 0x2000, 0x3000, None, -1.0,
                                    0x4000, None) == DF2_ERR_INVALID_ARG  # eps < 0
    assert lib.dflash2_workspace_init(ctypes.byref(d), 0x100010, 1 << 40, None) == DF2_ERR_WORKSPACE
    assert lib.dflash2_workspace_init(ctypes.byref(d), 0x100000, 4096, None) == DF2_ERR_WORKSPACE
    assert lib.dflash2_workspace_init(ctypes.byref(dims(k=0)), 0x100000, 1 << 40, None) == DF2_ERR_INVALID_ARG


def test_select_host_workspace_and_rejections(lib):
    # Pointer values below are never dereferenced: every case fails validation first.
    from speculative_decoding_drafter_gb300.dflash2 import (dflash2_select_host_workspace_bytes,
                                                            dflash2_workspace_bytes)

    d = dims()
    R, H, B, k = d.B * d.T, d.H, d.B, d.k
    base = dflash2_workspace_bytes(d)
    n = dflash2_select_host_workspace_bytes(d)
    assert n % 256 == 0
    assert n >= base + R * H * 2 + B * 4 + R * (k + k * k) * 4 + R * 4
    assert dflash2_select_host_workspace_bytes(dims(k=0)) == 0
    h, w, a, lat, dr = 0x300000, 0x200000, 0x310000, 0x320000, 0x330000

    def call(dd=d, hidden=h, anchor=a, draft=dr, ws=0x100000, ws_bytes=n, W_vocab=w):
        return lib.dflash2_select_host(ctypes.byref(dd), hidden, W_vocab, w, w, w, anchor, lat, draft, None, ws,
                                       ws_bytes, None)

    assert call(hidden=None) == DF2_ERR_INVALID_ARG
    assert call(anchor=None) == DF2_ERR_INVALID_ARG
    assert call(draft=None) == DF2_ERR_INVALID_ARG
    assert call(W_vocab=0x200008) == DF2_ERR_INVALID_ARG
    assert call(dd=dims(k=0)) == DF2_ERR_INVALID_ARG
    assert call(ws_bytes=base) == DF2_ERR_WORKSPACE  # room for dflash2_select only, not the staging
    assert call(ws=0x100010) == DF2_ERR_WORKSPACE
    # device pointers are checked before any copy is enqueued (W_sel not 16-byte aligned)
    assert lib.dflash2_select_host(ctypes.byref(d), h, w, w + 8, w, w, a, lat, dr, None, 0x100000, n, None) == \
        DF2_ERR_INVALID_ARG


def test_selftest_wait_timeout_rejections(lib):
    assert lib.dflash2_selftest_wait_timeout(0, 0x100000, 4096, None) == DF2_ERR_INVALID_ARG
    assert lib.dflash2_selftest_wait_timeout(1000001, 0x100000, 4096, None) == DF2_ERR_INVALID_ARG
    assert lib.dflash2_selftest_wait_timeout(100, None, 4096, None) == DF2_ERR_WORKSPACE
    assert lib.dflash2_selftest_wait_timeout(100, 0x100010, 4096, None) == DF2_ERR_WORKSPACE


def test_header_is_usable_from_plain_c(lib, tmp_path):
    """include/dflash2.h compiles as C99 and the library links and answers from a C program."""
    import shutil
    import subprocess

    from speculative_decoding_drafter_gb300.build import LIB_PATH

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    exe = tmp_path / "abi_from_c"
    libdir = os.path.dirname(LIB_PATH)
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                    os.path.join(root, "tests", "c", "abi_from_c.c"), "-o", str(exe), "-L", libdir, "-ldflash2",
                    "-Wl,-rpath," + libdir], check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip() == "ok"
