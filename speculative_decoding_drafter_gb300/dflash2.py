"""Thin ctypes binding of libdflash2.so (the C ABI in include/dflash2.h).

Functions carry the C names and only marshal arguments: torch CUDA tensors are
checked for dtype, device, shape and contiguity, their data pointers and the
current CUDA stream are passed through, and a non-OK status raises
:class:`DFlash2Error`.  Every step of the selector head runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback, and a missing library is
an error.
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

import torch

from .build import LIB_PATH

__all__ = [
    "DFlash2Error", "Dims", "library", "dflash2_workspace_bytes", "dflash2_workspace_init", "dflash2_select",
    "dflash2_select_from_logits", "dflash2_lm_head_logits", "dflash2_topk", "dflash2_gate", "dflash2_lattice",
    "dflash2_walk", "dflash2_check_device_status", "dflash2_status_string", "dflash2_version", "Workspace",
    "dflash2_profile_events", "dflash2_topk_noalloc", "dflash2_walk_sample", "dflash2_dynamic_conv",
    "ConvDims", "EXPORTED_SYMBOLS", "dflash2_select_host", "dflash2_select_host_workspace_bytes", "HostWorkspace",
    "SelectHostPlan", "dflash2_selftest_wait_timeout", "WalkOpts", "dflash2_select_walk",
]

EXPORTED_SYMBOLS = (
    "dflash2_workspace_bytes", "dflash2_workspace_init", "dflash2_select", "dflash2_select_from_logits",
    "dflash2_lm_head_logits", "dflash2_topk", "dflash2_gate", "dflash2_lattice", "dflash2_walk",
    "dflash2_check_device_status", "dflash2_status_string", "dflash2_version", "dflash2_profile_events",
    "dflash2_topk_noalloc", "dflash2_walk_sample", "dflash2_dynamic_conv", "dflash2_select_host",
    "dflash2_select_host_workspace_bytes", "dflash2_selftest_wait_timeout", "dflash2_select_walk",
)


class DFlash2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({_status_string(status)})")


class ConvDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("C", ctypes.c_int32), ("G", ctypes.c_int32)]


class WalkOpts(ctypes.Structure):
    """df2_walk_opts: temperature, p_min, uniforms [B, T] (or NULL: greedy), n_draft [B], confidence [B, T]."""
    _fields_ = [("temperature", ctypes.c_float), ("p_min", ctypes.c_float), ("uniforms", ctypes.c_void_p),
                ("n_draft", ctypes.c_void_p), ("confidence", ctypes.c_void_p)]


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("V", ctypes.c_int32),
                ("k", ctypes.c_int32), ("D", ctypes.c_int32)]

    def __repr__(self):
        return f"Dims(B={self.B}, T={self.T}, H={self.H}, V={self.V}, k={self.k}, D={self.D})"


_lock = threading.Lock()
_lib = None


def library(path: str | None = None):
    """Load libdflash2.so (built by ``__graft_entry__.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = path or LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is not built; run speculative_decoding_drafter_gb300.build.build() "
                                   "(nvcc, sm_103a) first -- there is no fallback path")
            lib = ctypes.CDLL(path)
            P, S, I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
            D = ctypes.POINTER(Dims)
            sig = {
                "dflash2_workspace_bytes": (S, [D]),
                "dflash2_workspace_init": (I, [D, P, S, P]),
                "dflash2_select": (I, [D, P, P, P, P, P, P, P, P, P, P, P, P, S, P]),
                "dflash2_select_from_logits": (I, [D, P, P, P, P, P, P, P, P, P, P, P, P, S, P]),
                "dflash2_lm_head_logits": (I, [D, P, P, P, P, S, P]),
                "dflash2_topk": (I, [D, P, P, P, P, S, P]),
                "dflash2_gate": (I, [D, P, P, P, P, S, P]),
                "dflash2_lattice": (I, [D, P, P, P, P, P, P, P, P]),
                "dflash2_walk": (I, [D, P, P, P]),
                "dflash2_check_device_status": (I, [P, S, P]),
                "dflash2_status_string": (ctypes.c_char_p, [I]),
                "dflash2_version": (ctypes.c_int32, []),
                "dflash2_profile_events": (I, [P, P]),
                "dflash2_topk_noalloc": (I, [D, P, P, P, P]),
                "dflash2_walk_sample": (I, [D, P, ctypes.c_float, ctypes.c_float, P, P, P, P, P]),
                "dflash2_dynamic_conv": (I, [ctypes.POINTER(ConvDims), P, P, P, P, P, ctypes.c_float, P, P]),
                "dflash2_select_host": (I, [D, P, P, P, P, P, P, P, P, P, P, S, P]),
                "dflash2_select_host_workspace_bytes": (S, [D]),
                "dflash2_selftest_wait_timeout": (I, [ctypes.c_uint32, P, S, P]),
                "dflash2_select_walk": (I, [D, ctypes.POINTER(WalkOpts), P, P, P, P, P, P, P, P, P, P, P, P, S, P]),
            }
            for name, (res, args) in sig.items():
                f = getattr(lib, name)
                f.restype, f.argtypes = res, args
            _lib = lib
        return _lib


def _status_string(status: int) -> str:
    try:
        return library().dflash2_status_string(status).decode()
    except Exception:  # pragma: no cover - only when the library itself is missing
        return "unknown"


def dflash2_status_string(status: int) -> str:
    return library().dflash2_status_string(int(status)).decode()


def dflash2_version() -> int:
    return int(library().dflash2_version())


def _check(status: int, where: str) -> None:
    if status != 0:
        raise DFlash2Error(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _torch_stream(stream):
    """torch's object for a `stream` argument (a torch stream, or an int: a raw handle)."""
    if isinstance(stream, torch.cuda.Stream):
        return stream
    handle = int(stream)
    return torch.cuda.default_stream() if handle == 0 else torch.cuda.ExternalStream(handle)


def _on_stream(fn):
    """Runs a wrapper with its `stream` as torch's current stream, so that what it allocates
    (outputs, a workspace zeroed when allocated) is filled on, and reused in the order of, the
    stream the library launches on."""

    @functools.wraps(fn)
    def wrapper(*args, stream=None, **kwargs):
        if stream is None or not torch.cuda.is_available():
            # the current stream is the launch stream already (without a GPU the wrapper's
            # argument checks raise before any CUDA call)
            return fn(*args, stream=stream, **kwargs)
        ts = _torch_stream(stream)
        with torch.cuda.stream(ts):
            return fn(*args, stream=ts, **kwargs)

    return wrapper


def _ptr(t, dtype, shape, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.get_device() != torch.cuda.current_device():
        # the library launches on the current device (and takes that device's scratch): a
        # tensor on another device would be read across devices
        raise ValueError(f"{name} is on cuda:{t.get_device()}, not on the current device "
                         f"cuda:{torch.cuda.current_device()} (use torch.cuda.device(...))")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def make_dims(B, T, H, V, k, D) -> Dims:
    return Dims(int(B), int(T), int(H), int(V), int(k), int(D))


def dflash2_workspace_bytes(dims: Dims) -> int:
    return int(library().dflash2_workspace_bytes(ctypes.byref(dims)))


@_on_stream
def dflash2_workspace_init(workspace: "Workspace", stream=None) -> None:
    """Zero the workspace's control block (status word, counters, the LM head's bound slots) on the stream."""
    _check(library().dflash2_workspace_init(ctypes.byref(workspace.dims), workspace.ptr, workspace.nbytes,
                                            _stream(stream)), "dflash2_workspace_init")


class Workspace:
    """Device scratch for one problem size (uint8 tensor, 256-byte aligned, zeroed on the current stream
    when allocated)."""

    def __init__(self, dims: Dims, device=None):
        n = dflash2_workspace_bytes(dims)
        if n == 0:
            raise ValueError(f"invalid or unsupported dims {dims}")
        self.dims = dims
        self.tensor = torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.tensor.data_ptr()) % 256
        self.view = self.tensor[off:off + n]
        self.nbytes = n

    @property
    def ptr(self) -> int:
        return self.view.data_ptr()


class HostWorkspace(Workspace):
    """Workspace of dflash2_select_host: the select workspace plus device staging of the
    host-side inputs and results."""

    def __init__(self, dims: Dims, device=None):
        n = dflash2_select_host_workspace_bytes(dims)
        if n == 0:
            raise ValueError(f"invalid or unsupported dims {dims}")
        self.dims = dims
        self.tensor = torch.zeros(n + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.tensor.data_ptr()) % 256
        self.view = self.tensor[off:off + n]
        self.nbytes = n


def dflash2_select_host_workspace_bytes(dims: Dims) -> int:
    return int(library().dflash2_select_host_workspace_bytes(ctypes.byref(dims)))


def _host_ptr(t, dtype, shape, name):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or t.device.type != "cpu":
        raise TypeError(f"{name} must be a CPU tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _workspace(ws, dims, device):
    if ws is None:
        return Workspace(dims, device)
    if ws.nbytes < dflash2_workspace_bytes(dims):
        raise ValueError("workspace too small for these dims")
    return ws


def _dims_of(hidden, W_vocab_or_none, W_sel, pred_cb, k, T, V=None):
    R, H = hidden.shape
    if R % T:
        raise ValueError(f"hidden has {R} rows, not a multiple of T={T}")
    V = V if V is not None else W_vocab_or_none.shape[0]
    D = W_sel.shape[0]
    return make_dims(R // T, T, H, V, k, D)


@_on_stream
def dflash2_select(hidden, W_vocab, W_sel, pred_cb, succ_cb, anchor, k: int, T: int, *, lattice=None,
                   draft_ids=None, topk_ids=None, topk_logits=None, gate=None, workspace=None, stream=None):
    """Whole selector head on the GPU. Returns (lattice [B*T, k+k*k] float32, draft_ids [B, T] int32)."""
    d = _dims_of(hidden, W_vocab, W_sel, pred_cb, k, T)
    dev = hidden.device
    R = d.B * d.T
    lattice = lattice if lattice is not None else torch.empty((R, k + k * k), dtype=torch.float32, device=dev)
    draft_ids = draft_ids if draft_ids is not None else torch.empty((d.B, T), dtype=torch.int32, device=dev)
    ws = _workspace(workspace, d, dev)
    bf = torch.bfloat16
    st = library().dflash2_select(
        ctypes.byref(d), _ptr(hidden, bf, (R, d.H), "hidden"), _ptr(W_vocab, bf, (d.V, d.H), "W_vocab"),
        _ptr(W_sel, bf, (d.D, d.H), "W_sel"), _ptr(pred_cb, bf, (d.V, d.D), "pred_cb"),
        _ptr(succ_cb, bf, (d.V, d.D), "succ_cb"), _ptr(anchor, torch.int32, (d.B,), "anchor"),
        _ptr(lattice, torch.float32, (R, k + k * k), "lattice"), _ptr(draft_ids, torch.int32, (d.B, T), "draft_ids"),
        _ptr(topk_ids, torch.int32, (R, k), "topk_ids"), _ptr(topk_logits, torch.float32, (R, k), "topk_logits"),
        _ptr(gate, torch.float32, (R, d.D), "gate"), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "dflash2_select")
    return lattice, draft_ids


@_on_stream
def dflash2_select_walk(hidden, W_vocab, W_sel, pred_cb, succ_cb, anchor, k: int, T: int, *, temperature: float = 1.0,
                        p_min: float = 0.0, uniforms=None, lattice=None, draft_ids=None, n_draft=None,
                        confidence=None, topk_ids=None, topk_logits=None, gate=None, workspace=None, stream=None):
    """Whole selector head with the confidence / p_min / sampling walk in the same launches.

    Returns (lattice, draft_ids [B, T] with -1 from a stop on, n_draft int32 [B], confidence float32 [B, T])."""
    d = _dims_of(hidden, W_vocab, W_sel, pred_cb, k, T)
    dev = hidden.device
    R = d.B * d.T
    lattice = lattice if lattice is not None else torch.empty((R, k + k * k), dtype=torch.float32, device=dev)
    draft_ids = draft_ids if draft_ids is not None else torch.empty((d.B, T), dtype=torch.int32, device=dev)
    n_draft = n_draft if n_draft is not None else torch.empty((d.B,), dtype=torch.int32, device=dev)
    confidence = confidence if confidence is not None else torch.empty((d.B, T), dtype=torch.float32, device=dev)
    ws = _workspace(workspace, d, dev)
    opts = WalkOpts(float(temperature), float(p_min), _ptr(uniforms, torch.float32, (d.B, T), "uniforms"),
                    _ptr(n_draft, torch.int32, (d.B,), "n_draft"),
                    _ptr(confidence, torch.float32, (d.B, T), "confidence"))
    bf = torch.bfloat16
    st = library().dflash2_select_walk(
        ctypes.byref(d), ctypes.byref(opts), _ptr(hidden, bf, (R, d.H), "hidden"),
        _ptr(W_vocab, bf, (d.V, d.H), "W_vocab"), _ptr(W_sel, bf, (d.D, d.H), "W_sel"),
        _ptr(pred_cb, bf, (d.V, d.D), "pred_cb"), _ptr(succ_cb, bf, (d.V, d.D), "succ_cb"),
        _ptr(anchor, torch.int32, (d.B,), "anchor"), _ptr(lattice, torch.float32, (R, k + k * k), "lattice"),
        _ptr(draft_ids, torch.int32, (d.B, T), "draft_ids"), _ptr(topk_ids, torch.int32, (R, k), "topk_ids"),
        _ptr(topk_logits, torch.float32, (R, k), "topk_logits"), _ptr(gate, torch.float32, (R, d.D), "gate"),
        ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "dflash2_select_walk")
    return lattice, draft_ids, n_draft, confidence


def _select_host_args(hidden_host, W_vocab, W_sel, pred_cb, succ_cb, anchor_host, k, T, lattice_host,
                      draft_ids_host, workspace, stream, status_host=None):
    """Checks the arguments of dflash2_select_host once; returns (args tuple, tensors kept alive)."""
    d = _dims_of(hidden_host, W_vocab, W_sel, pred_cb, k, T)
    R = d.B * d.T
    if lattice_host is None:
        lattice_host = torch.empty((R, k + k * k), dtype=torch.float32).pin_memory()
    elif lattice_host is False:
        lattice_host = None
    if draft_ids_host is None:
        draft_ids_host = torch.empty((d.B, T), dtype=torch.int32).pin_memory()
    if workspace is None:
        workspace = HostWorkspace(d, W_vocab.device)
    elif workspace.nbytes < dflash2_select_host_workspace_bytes(d):
        raise ValueError("workspace too small for dflash2_select_host with these dims")
    bf = torch.bfloat16
    args = (ctypes.byref(d), _host_ptr(hidden_host, bf, (R, d.H), "hidden_host"),
            _ptr(W_vocab, bf, (d.V, d.H), "W_vocab"), _ptr(W_sel, bf, (d.D, d.H), "W_sel"),
            _ptr(pred_cb, bf, (d.V, d.D), "pred_cb"), _ptr(succ_cb, bf, (d.V, d.D), "succ_cb"),
            _host_ptr(anchor_host, torch.int32, (d.B,), "anchor_host"),
            _host_ptr(lattice_host, torch.float32, (R, k + k * k), "lattice_host"),
            _host_ptr(draft_ids_host, torch.int32, (d.B, T), "draft_ids_host"),
            _host_ptr(status_host, torch.int32, (1,), "status_host"), workspace.ptr, workspace.nbytes, _stream(stream))
    keep = (d, hidden_host, W_vocab, W_sel, pred_cb, succ_cb, anchor_host, workspace, status_host)
    return args, keep, lattice_host, draft_ids_host


@_on_stream
def dflash2_select_host(hidden_host, W_vocab, W_sel, pred_cb, succ_cb, anchor_host, k: int, T: int, *,
                        lattice_host=None, draft_ids_host=None, workspace: HostWorkspace | None = None, stream=None):
    """Selector head with host-memory inputs and results (pin them for asynchronous copies).

    hidden_host bf16 [B*T, H] and anchor_host int32 [B] are CPU tensors; the weights are CUDA
    tensors.  Returns (lattice_host or None, draft_ids_host [B, T] int32), filled when the call
    returns.  Pass lattice_host=False to skip the lattice copy.
    """
    args, _keep, lattice_host, draft_ids_host = _select_host_args(
        hidden_host, W_vocab, W_sel, pred_cb, succ_cb, anchor_host, k, T, lattice_host, draft_ids_host, workspace,
        stream)
    _check(library().dflash2_select_host(*args), "dflash2_select_host")
    return lattice_host, draft_ids_host


class SelectHostPlan:
    """dflash2_select_host with its buffers bound once, for a drafting loop that refills the
    same host buffers every step: the arguments are checked here, and each call is a single
    C call (the per-call checks of the function above cost as much as a kernel launch).
    The bound tensors are kept alive; write the next step's hidden states and anchors into
    them in place.  Calling returns (lattice_host or None, draft_ids_host)."""

    @_on_stream
    def __init__(self, hidden_host, W_vocab, W_sel, pred_cb, succ_cb, anchor_host, k: int, T: int, *,
                 lattice_host=None, draft_ids_host=None, workspace: HostWorkspace | None = None, stream=None,
                 pinned_status: bool = True):
        # a page-locked word for the device status (a pageable one costs a staged copy per call)
        self.status_host = torch.zeros(1, dtype=torch.int32).pin_memory() if pinned_status else None
        self._args, self._keep, self.lattice_host, self.draft_ids_host = _select_host_args(
            hidden_host, W_vocab, W_sel, pred_cb, succ_cb, anchor_host, k, T, lattice_host, draft_ids_host,
            workspace, stream, self.status_host)
        self._fn = library().dflash2_select_host

    def __call__(self):
        st = self._fn(*self._args)
        if st:
            raise DFlash2Error(st, "dflash2_select_host")
        return self.lattice_host, self.draft_ids_host


@_on_stream
def dflash2_select_from_logits(logits, hidden, W_sel, pred_cb, succ_cb, anchor, k: int, T: int, *, lattice=None,
                               draft_ids=None, topk_ids=None, topk_logits=None, gate=None, workspace=None,
                               stream=None):
    """Selector head from given float32 logits [B*T, V]. Returns (lattice, draft_ids)."""
    d = _dims_of(hidden, None, W_sel, pred_cb, k, T, V=logits.shape[1])
    dev = hidden.device
    R = d.B * d.T
    lattice = lattice if lattice is not None else torch.empty((R, k + k * k), dtype=torch.float32, device=dev)
    draft_ids = draft_ids if draft_ids is not None else torch.empty((d.B, T), dtype=torch.int32, device=dev)
    ws = _workspace(workspace, d, dev)
    bf = torch.bfloat16
    st = library().dflash2_select_from_logits(
        ctypes.byref(d), _ptr(logits, torch.float32, (R, d.V), "logits"), _ptr(hidden, bf, (R, d.H), "hidden"),
        _ptr(W_sel, bf, (d.D, d.H), "W_sel"), _ptr(pred_cb, bf, (d.V, d.D), "pred_cb"),
        _ptr(succ_cb, bf, (d.V, d.D), "succ_cb"), _ptr(anchor, torch.int32, (d.B,), "anchor"),
        _ptr(lattice, torch.float32, (R, k + k * k), "lattice"), _ptr(draft_ids, torch.int32, (d.B, T), "draft_ids"),
        _ptr(topk_ids, torch.int32, (R, k), "topk_ids"), _ptr(topk_logits, torch.float32, (R, k), "topk_logits"),
        _ptr(gate, torch.float32, (R, d.D), "gate"), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "dflash2_select_from_logits")
    return lattice, draft_ids


@_on_stream
def dflash2_lm_head_logits(hidden, W_vocab, *, out=None, workspace=None, stream=None):
    """float32 logits [R, V] from the tensor-core LM head (stage check / standalone use)."""
    R, H = hidden.shape
    V = W_vocab.shape[0]
    d = make_dims(R, 1, H, V, 1, 8)
    out = out if out is not None else torch.empty((R, V), dtype=torch.float32, device=hidden.device)
    ws = _workspace(workspace, d, hidden.device)
    bf = torch.bfloat16
    st = library().dflash2_lm_head_logits(ctypes.byref(d), _ptr(hidden, bf, (R, H), "hidden"),
                                          _ptr(W_vocab, bf, (V, H), "W_vocab"),
                                          _ptr(out, torch.float32, (R, V), "logits"), ws.ptr, ws.nbytes,
                                          _stream(stream))
    _check(st, "dflash2_lm_head_logits")
    return out


@_on_stream
def dflash2_topk(logits, k: int, *, ids=None, vals=None, workspace=None, stream=None):
    """Top-k of float32 logits [R, V] by (value desc, id asc). Returns (ids int32 [R,k], vals float32 [R,k])."""
    R, V = logits.shape
    d = make_dims(R, 1, 8, V, k, 8)
    ids = ids if ids is not None else torch.empty((R, k), dtype=torch.int32, device=logits.device)
    vals = vals if vals is not None else torch.empty((R, k), dtype=torch.float32, device=logits.device)
    ws = _workspace(workspace, d, logits.device)
    st = library().dflash2_topk(ctypes.byref(d), _ptr(logits, torch.float32, (R, V), "logits"),
                                _ptr(ids, torch.int32, (R, k), "topk_ids"),
                                _ptr(vals, torch.float32, (R, k), "topk_logits"), ws.ptr, ws.nbytes,
                                _stream(stream))
    _check(st, "dflash2_topk")
    return ids, vals


@_on_stream
def dflash2_topk_noalloc(logits, k: int, *, ids=None, vals=None, stream=None):
    """dflash2_topk without a workspace (the library's own fixed device array holds the
    scratch); for callers that cannot allocate.  Overlapping calls race."""
    R, V = logits.shape
    d = make_dims(R, 1, 8, V, k, 8)
    ids = ids if ids is not None else torch.empty((R, k), dtype=torch.int32, device=logits.device)
    vals = vals if vals is not None else torch.empty((R, k), dtype=torch.float32, device=logits.device)
    st = library().dflash2_topk_noalloc(ctypes.byref(d), _ptr(logits, torch.float32, (R, V), "logits"),
                                        _ptr(ids, torch.int32, (R, k), "topk_ids"),
                                        _ptr(vals, torch.float32, (R, k), "topk_logits"), _stream(stream))
    _check(st, "dflash2_topk_noalloc")
    return ids, vals


@_on_stream
def dflash2_gate(hidden, W_sel, *, out=None, workspace=None, stream=None):
    """Gate float32 [R, D] = hidden . W_sel^T on tensor cores."""
    R, H = hidden.shape
    D = W_sel.shape[0]
    d = make_dims(R, 1, H, max(1, D), 1, D)
    out = out if out is not None else torch.empty((R, D), dtype=torch.float32, device=hidden.device)
    ws = _workspace(workspace, d, hidden.device)
    bf = torch.bfloat16
    st = library().dflash2_gate(ctypes.byref(d), _ptr(hidden, bf, (R, H), "hidden"), _ptr(W_sel, bf, (D, H), "W_sel"),
                                _ptr(out, torch.float32, (R, D), "gate"), ws.ptr, ws.nbytes, _stream(stream))
    _check(st, "dflash2_gate")
    return out


@_on_stream
def dflash2_lattice(topk_ids, topk_logits, gate, pred_cb, succ_cb, anchor, T: int, *, out=None, stream=None):
    """Packed lattice [B*T, k+k*k] from candidates, unary scores and the gate."""
    R, k = topk_ids.shape
    V, D = pred_cb.shape
    B = anchor.shape[0]
    if R != B * T:
        raise ValueError("topk_ids rows must equal B*T")
    d = make_dims(B, T, 8, V, k, D)
    out = out if out is not None else torch.empty((R, k + k * k), dtype=torch.float32, device=topk_ids.device)
    bf = torch.bfloat16
    st = library().dflash2_lattice(ctypes.byref(d), _ptr(topk_ids, torch.int32, (R, k), "topk_ids"),
                                   _ptr(topk_logits, torch.float32, (R, k), "topk_logits"),
                                   _ptr(gate, torch.float32, (R, D), "gate"), _ptr(pred_cb, bf, (V, D), "pred_cb"),
                                   _ptr(succ_cb, bf, (V, D), "succ_cb"), _ptr(anchor, torch.int32, (B,), "anchor"),
                                   _ptr(out, torch.float32, (R, k + k * k), "lattice"), _stream(stream))
    _check(st, "dflash2_lattice")
    return out


@_on_stream
def dflash2_walk(lattice, B: int, T: int, k: int, *, out=None, stream=None):
    """Greedy walk over packed rows: draft ids int32 [B, T]."""
    d = make_dims(B, T, 8, max(k, 1), k, 8)
    out = out if out is not None else torch.empty((B, T), dtype=torch.int32, device=lattice.device)
    st = library().dflash2_walk(ctypes.byref(d), _ptr(lattice, torch.float32, (B * T, k + k * k), "lattice"),
                                _ptr(out, torch.int32, (B, T), "draft_ids"), _stream(stream))
    _check(st, "dflash2_walk")
    return out


@_on_stream
def dflash2_walk_sample(lattice, B: int, T: int, k: int, *, temperature: float = 1.0, p_min: float = 0.0,
                        uniforms=None, draft=None, n_draft=None, confidence=None, stream=None):
    """Walk with confidence and p_min stop; inverse-CDF sampling when ``uniforms`` [B, T] is given.

    Returns (draft int32 [B, T] with -1 from a stop on, n_draft int32 [B], confidence float32 [B, T])."""
    d = make_dims(B, T, 8, max(k, 1), k, 8)
    dev = lattice.device
    draft = draft if draft is not None else torch.empty((B, T), dtype=torch.int32, device=dev)
    n_draft = n_draft if n_draft is not None else torch.empty((B,), dtype=torch.int32, device=dev)
    confidence = confidence if confidence is not None else torch.empty((B, T), dtype=torch.float32, device=dev)
    st = library().dflash2_walk_sample(ctypes.byref(d), _ptr(lattice, torch.float32, (B * T, k + k * k), "lattice"),
                                       float(temperature), float(p_min),
                                       _ptr(uniforms, torch.float32, (B, T), "uniforms"),
                                       _ptr(draft, torch.int32, (B, T), "draft_ids"),
                                       _ptr(n_draft, torch.int32, (B,), "n_draft"),
                                       _ptr(confidence, torch.float32, (B, T), "confidence"), _stream(stream))
    _check(st, "dflash2_walk_sample")
    return draft, n_draft, confidence


@_on_stream
def dflash2_dynamic_conv(x, base, dyn, T: int, *, x_prev=None, gamma=None, eps: float = 1e-6, G: int = 16, out=None,
                         stream=None):
    """Two-tap dynamic depthwise conv of B blocks of T rows: bf16 [B*T, C] -> bf16 [B*T, C]."""
    R, C = x.shape
    if R % T:
        raise ValueError(f"x has {R} rows, not a multiple of T={T}")
    B = R // T
    d = ConvDims(B, T, C, G)
    out = out if out is not None else torch.empty_like(x)
    bf = torch.bfloat16
    st = library().dflash2_dynamic_conv(ctypes.byref(d), _ptr(x, bf, (R, C), "x"), _ptr(x_prev, bf, (B, C), "x_prev"),
                                        _ptr(base, bf, (2, C), "base"),
                                        _ptr(dyn, torch.float32, (R, 2, C // G), "dyn"), _ptr(gamma, bf, (C,), "gamma"),
                                        float(eps), _ptr(out, bf, (R, C), "y"), _stream(stream))
    _check(st, "dflash2_dynamic_conv")
    return out


@_on_stream
def dflash2_check_device_status(workspace: Workspace, stream=None) -> None:
    """Synchronises the stream; raises DFlash2Error(DF2_ERR_TIMEOUT) if a kernel wait gave up."""
    _check(library().dflash2_check_device_status(workspace.ptr, workspace.nbytes, _stream(stream)),
           "dflash2_check_device_status")


@_on_stream
def dflash2_selftest_wait_timeout(workspace: Workspace, limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test: a device wait that nothing satisfies gives up after
    limit_us and raises the workspace's status word (read it with dflash2_check_device_status)."""
    _check(library().dflash2_selftest_wait_timeout(int(limit_us), workspace.ptr, workspace.nbytes, _stream(stream)),
           "dflash2_selftest_wait_timeout")


def dflash2_profile_events(begin=None, end=None) -> None:
    """Record torch.cuda.Event pairs around the LM-head launch of following select calls (None, None stops)."""
    b = None if begin is None else begin.cuda_event
    e = None if end is None else end.cuda_event
    if (begin is not None and not b) or (end is not None and not e):
        raise ValueError("record each torch.cuda.Event once before passing it (torch creates it lazily)")
    _check(library().dflash2_profile_events(b, e), "dflash2_profile_events")
