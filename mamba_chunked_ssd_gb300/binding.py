"""Thin Python binding of libmamba2ssd.so (argument marshalling only).

Each function has the name of the C entry point it calls and takes torch
tensors that already live on the GPU; it passes their data pointers, the
shape and the current CUDA stream to the library and allocates any missing
output with ``torch.empty``.  No step of the forward pass runs in Python: if
the library is missing the import fails loudly, there is no fallback.

Layouts and semantics are those of include/mamba2_ssd.h ("Accelerating
Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile",
§Kernel 1-3).
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmamba2ssd.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "mamba2_ssd.h")

MAMBA2_F32, MAMBA2_BF16 = 0, 1
STATUS = {0: "MAMBA2_OK", 1: "MAMBA2_ERR_INVALID_ARG", 2: "MAMBA2_ERR_UNSUPPORTED",
          3: "MAMBA2_ERR_CUDA", 4: "MAMBA2_ERR_TIMEOUT"}


class Mamba2Error(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} failed: {text}")
        self.code = code


class mamba2_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("dstate", ctypes.c_int64), ("ngroups", ctypes.c_int64),
                ("chunk_size", ctypes.c_int64), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmamba2ssd.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m mamba_chunked_ssd_gb300.build_lib` (needs nvcc)")
    lib = ctypes.CDLL(path)
    P, S = ctypes.c_void_p, ctypes.POINTER(mamba2_shape)
    sig = {
        "mamba2_chunk_cumsum": (ctypes.c_int, [S, P, P, P, P]),
        "mamba2_state_pass": (ctypes.c_int, [S, P, P, P, P, P, P, P, P]),
        "mamba2_chunk_out": (ctypes.c_int, [S, P, P, P, P, P, P, P, P, P]),
        "mamba2_ssd_fwd_workspace_size": (ctypes.c_size_t, [S]),
        "mamba2_ssd_fwd_chunk_size": (ctypes.c_int64, [S]),
        "mamba2_ssd_fwd": (ctypes.c_int, [S, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P]),
        "mamba2_ssd_fwd_noalloc": (ctypes.c_int, [S, P, P, P, P, P, P, P, P, P, P]),
        "mamba2_ssd_step": (ctypes.c_int, [S, P, P, P, P, P, P, P, P, P, P]),
        "mamba2_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_int64, P]),
        "mamba2_check_device_status": (ctypes.c_int, [P]),
        "mamba2_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "mamba2_version": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype, f.argtypes = res, args
    _lib = lib
    return lib


def header_functions(path: str = HEADER):
    """Names of the functions include/mamba2_ssd.h declares."""
    text = open(path).read()
    return sorted(set(re.findall(r"MAMBA2_API\s+[\w\s\*]+?\b(mamba2_\w+)\s*\(", text)))


def _check(fn: str, rc: int):
    if rc != 0:
        text = load_library().mamba2_status_string(rc).decode()
        raise Mamba2Error(fn, rc, text)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MAMBA2_BF16
    if t.dtype == torch.float32:
        return MAMBA2_F32
    raise TypeError(f"unsupported dtype {t.dtype}: x, B, C must be bfloat16 or float32")


def make_shape(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, dtype_code) -> mamba2_shape:
    return mamba2_shape(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, dtype_code, 0)


def shape_of(x: torch.Tensor, B: torch.Tensor, chunk_size: int) -> mamba2_shape:
    b, L, nh, H = x.shape
    return make_shape(b, L, nh, H, B.shape[3], B.shape[2], int(chunk_size), _dtype_code(x))


def _need(t, name):
    if t is not None and not (t.is_cuda and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def mamba2_chunk_cumsum(dt, A, chunk_size, G=None, stream=None):
    """Stage 1: G [b, nh, L] fp32 (log2 units)."""
    _need(dt, "dt"), _need(A, "A")
    b, L, nh = dt.shape
    shape = make_shape(b, L, nh, 1, 1, 1, int(chunk_size), MAMBA2_F32)
    if G is None:
        G = torch.empty(b, nh, L, device=dt.device, dtype=torch.float32)
    _check("mamba2_chunk_cumsum", load_library().mamba2_chunk_cumsum(
        ctypes.byref(shape), _ptr(dt), _ptr(A), _ptr(G), _stream(stream)))
    return G


def mamba2_state_pass(x, dt, B, G, chunk_size, initial_state=None, chunk_states=None,
                      final_state=None, want_final_state=True, stream=None):
    """Stage 2: (chunk_states [b, nh, nc, S, H], final_state [b, nh, S, H] or None)."""
    for t, n in ((x, "x"), (dt, "dt"), (B, "B"), (G, "G"), (initial_state, "initial_state")):
        _need(t, n)
    shape = shape_of(x, B, chunk_size)
    nc = -(-shape.seqlen // shape.chunk_size)
    if chunk_states is None:
        chunk_states = torch.empty(shape.batch, shape.nheads, nc, shape.dstate, shape.headdim,
                                   device=x.device, dtype=x.dtype)
    if final_state is None and want_final_state:
        final_state = torch.empty(shape.batch, shape.nheads, shape.dstate, shape.headdim,
                                  device=x.device, dtype=torch.float32)
    _check("mamba2_state_pass", load_library().mamba2_state_pass(
        ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(B), _ptr(G), _ptr(initial_state),
        _ptr(chunk_states), _ptr(final_state), _stream(stream)))
    return chunk_states, final_state


def mamba2_chunk_out(x, dt, B, C, G, chunk_states, chunk_size, D=None, y=None, stream=None):
    """Stage 3: y [b, L, nh, H] in x's dtype."""
    for t, n in ((x, "x"), (dt, "dt"), (B, "B"), (C, "C"), (G, "G"), (chunk_states, "chunk_states"),
                 (D, "D")):
        _need(t, n)
    shape = shape_of(x, B, chunk_size)
    if y is None:
        y = torch.empty_like(x)
    _check("mamba2_chunk_out", load_library().mamba2_chunk_out(
        ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(B), _ptr(C), _ptr(D), _ptr(G),
        _ptr(chunk_states), _ptr(y), _stream(stream)))
    return y


def mamba2_ssd_fwd_workspace_size(shape: mamba2_shape) -> int:
    return int(load_library().mamba2_ssd_fwd_workspace_size(ctypes.byref(shape)))


def mamba2_ssd_fwd_chunk_size(shape: mamba2_shape) -> int:
    return int(load_library().mamba2_ssd_fwd_chunk_size(ctypes.byref(shape)))


def mamba2_ssd_fwd(x, dt, A, B, C, chunk_size, D=None, initial_state=None, y=None, final_state=None,
                   want_final_state=True, workspace=None, stream=None):
    """Whole forward pass: (y, final_state or None)."""
    for t, n in ((x, "x"), (dt, "dt"), (A, "A"), (B, "B"), (C, "C"), (D, "D"),
                 (initial_state, "initial_state")):
        _need(t, n)
    shape = shape_of(x, B, chunk_size)
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and want_final_state:
        final_state = torch.empty(shape.batch, shape.nheads, shape.dstate, shape.headdim,
                                  device=x.device, dtype=torch.float32)
    ws_bytes = mamba2_ssd_fwd_workspace_size(shape)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), device=x.device, dtype=torch.uint8)
    _check("mamba2_ssd_fwd", load_library().mamba2_ssd_fwd(
        ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(initial_state), _ptr(y), _ptr(final_state), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return y, final_state


def mamba2_ssd_fwd_noalloc(x, dt, A, B, C, chunk_size, D=None, initial_state=None, y=None,
                           final_state=None, want_final_state=True, stream=None):
    """Whole forward pass with the library's fixed internal scratch (no
    workspace argument; the C entry point allocates nothing).  Missing outputs
    are allocated here, by the caller side, with torch."""
    for t, n in ((x, "x"), (dt, "dt"), (A, "A"), (B, "B"), (C, "C"), (D, "D"),
                 (initial_state, "initial_state")):
        _need(t, n)
    shape = shape_of(x, B, chunk_size)
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and want_final_state:
        final_state = torch.empty(shape.batch, shape.nheads, shape.dstate, shape.headdim,
                                  device=x.device, dtype=torch.float32)
    _check("mamba2_ssd_fwd_noalloc", load_library().mamba2_ssd_fwd_noalloc(
        ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(initial_state), _ptr(y), _ptr(final_state), _stream(stream)))
    return y, final_state


def mamba2_ssd_step(x, dt, A, B, C, state_in=None, D=None, state_out=None, y=None, stream=None):
    """One decode step: x [b, nh, H], dt [b, nh], B, C [b, G, S], state
    [b, nh, S, H] fp32.  Returns (y [b, nh, H], state_out).  Pass
    state_out=state_in to update the state in place."""
    for t, n in ((x, "x"), (dt, "dt"), (A, "A"), (B, "B"), (C, "C"), (D, "D"),
                 (state_in, "state_in"), (state_out, "state_out")):
        _need(t, n)
    b, nh, H = x.shape
    shape = make_shape(b, 1, nh, H, B.shape[2], B.shape[1], 1, _dtype_code(x))
    if y is None:
        y = torch.empty_like(x)
    if state_out is None:
        state_out = torch.empty(b, nh, B.shape[2], H, device=x.device, dtype=torch.float32)
    _check("mamba2_ssd_step", load_library().mamba2_ssd_step(
        ctypes.byref(shape), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(state_in), _ptr(state_out), _ptr(y), _stream(stream)))
    return y, state_out


def mamba2_selftest_wait_timeout(limit_ns: int, stream=None):
    """Enqueue the bounded-wait self-test kernel (see the header); the next
    mamba2_check_device_status then raises with MAMBA2_ERR_TIMEOUT."""
    _check("mamba2_selftest_wait_timeout",
           load_library().mamba2_selftest_wait_timeout(int(limit_ns), _stream(stream)))


def mamba2_check_device_status(stream=None):
    """Synchronises the stream and raises if a kernel reported a timeout."""
    _check("mamba2_check_device_status", load_library().mamba2_check_device_status(_stream(stream)))


def mamba2_version() -> int:
    return int(load_library().mamba2_version())
