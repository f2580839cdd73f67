"""fp64 CPU oracle for the Mamba-2 chunked SSD forward pass.

TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the product path (the
CUDA library and its binding) never does, and the two share no code.

Source: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
NVIDIA CUDA Tile" (NVIDIA technical blog).  The arithmetic lives in
``ssd_oracle.c`` (compiled here with gcc, no fast-math, no FMA contraction);
this module only marshals numpy/torch arrays into fp64 buffers and back.

Functions (all arrays in the library's layouts, returned as float64 numpy):
  ssd_recurrence  token-by-token recurrence  [blog §Mamba-2 architecture]
  chunk_cumsum    stage 1, G in log2 units   [blog §Kernel 1]
  state_pass      stage 2, chunk-start states and final state  [blog §Kernel 2]
  chunk_out       stage 3, outputs from chunk-start states     [blog §Kernel 3]
  ssd_chunked     stages 1 -> 2 -> 3 chained
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_LIB = os.path.join(_HERE, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in
                ("batch", "seqlen", "nheads", "headdim", "dstate", "ngroups", "chunk_size")]


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle shared library (gcc, -O2, strict IEEE fp64)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) and return the ctypes library."""
    global _lib
    with _lock:
        if path is not None:
            return _bind(ctypes.CDLL(path))
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    D = ctypes.POINTER(_Dims)
    lib.oracle_ssd_recurrence.argtypes = [D, P, P, P, P, P, P, P, P, P, P, P, I64, ctypes.c_int]
    lib.oracle_chunk_cumsum.argtypes = [D, P, P, P, P, I64, ctypes.c_int]
    lib.oracle_state_pass.argtypes = [D, P, P, P, P, P, P, P, P, I64, ctypes.c_int]
    lib.oracle_chunk_out.argtypes = [D, P, P, P, P, P, P, P, P, P, I64, ctypes.c_int]
    for f in (lib.oracle_ssd_recurrence, lib.oracle_chunk_cumsum, lib.oracle_state_pass,
              lib.oracle_chunk_out):
        f.restype = ctypes.c_int
    return lib


def _f64(a):
    """Any torch tensor / numpy array -> C-contiguous float64 numpy (exact widening)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor: widen on the CPU without numpy bf16
        import torch
        a = a.detach().to("cpu", torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dims(x, B, chunk_size):
    b, L, nh, H = x.shape
    S = B.shape[3]
    G = B.shape[2]
    if B.shape[:2] != (b, L) or nh % G:
        raise ValueError("inconsistent shapes")
    return _Dims(b, L, nh, H, S, G, int(chunk_size or 0))


def _pairs(pairs):
    if pairs is None:
        return None, 0
    arr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int64).reshape(-1, 2))
    return arr, arr.shape[0]


def _threads(nthreads):
    return int(nthreads or os.cpu_count() or 1)


def ssd_recurrence(x, dt, A, B, C, D=None, init=None, chunk_size=None, pairs=None, nthreads=None):
    """Token-by-token recurrence.  Returns dict(y, final_state[, chunk_states]).

    Only the listed (batch, head) ``pairs`` are computed when given; other
    entries of the outputs are left at zero."""
    x, dt, A, B, C, D, init = map(_f64, (x, dt, A, B, C, D, init))
    d = _dims(x, B, chunk_size)
    y = np.zeros_like(x)
    fin = np.zeros((d.batch, d.nheads, d.dstate, d.headdim))
    cs = None
    if chunk_size:
        nc = -(-d.seqlen // chunk_size)
        cs = np.zeros((d.batch, d.nheads, nc, d.dstate, d.headdim))
    pr, npr = _pairs(pairs)
    rc = load().oracle_ssd_recurrence(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                                      _ptr(D), _ptr(init), _ptr(y), _ptr(fin), _ptr(cs), _ptr(pr),
                                      npr, _threads(nthreads))
    if rc:
        raise ValueError("oracle_ssd_recurrence rejected its arguments")
    out = {"y": y, "final_state": fin}
    if cs is not None:
        out["chunk_states"] = cs
    return out


def ssd_step(x, dt, A, B, C, state=None, D=None):
    """One decode step: the recurrence advanced by one token from ``state``
    ("Accelerating Mamba-2 ...", §Mamba-2 architecture, core recurrence; the
    carried state of §Kernel 2).  x [b, nh, H], dt [b, nh], B, C [b, G, S],
    state [b, nh, S, H] or None (zeros).  It is the token-by-token recurrence
    on a one-token sequence.  Returns (y [b, nh, H], new state [b, nh, S, H])."""
    x, dt, B, C = (_f64(t)[:, None] for t in (x, dt, B, C))
    r = ssd_recurrence(x, dt, A, B, C, D=D, init=state)
    return r["y"][:, 0], r["final_state"]


def chunk_cumsum(dt, A, chunk_size, pairs=None, nthreads=None):
    """Stage 1: G [batch, nheads, L] (log2 units), fp64."""
    dt, A = _f64(dt), _f64(A)
    b, L, nh = dt.shape
    d = _Dims(b, L, nh, 1, 1, 1, int(chunk_size))
    G = np.zeros((b, nh, L))
    pr, npr = _pairs(pairs)
    if load().oracle_chunk_cumsum(ctypes.byref(d), _ptr(dt), _ptr(A), _ptr(G), _ptr(pr), npr,
                                  _threads(nthreads)):
        raise ValueError("oracle_chunk_cumsum rejected its arguments")
    return G


def state_pass(x, dt, B, G, chunk_size, init=None, pairs=None, nthreads=None):
    """Stage 2: (chunk_states [b, nh, nc, S, H], final_state [b, nh, S, H])."""
    x, dt, B, G, init = map(_f64, (x, dt, B, G, init))
    d = _dims(x, B, chunk_size)
    nc = -(-d.seqlen // chunk_size)
    cs = np.zeros((d.batch, d.nheads, nc, d.dstate, d.headdim))
    fin = np.zeros((d.batch, d.nheads, d.dstate, d.headdim))
    pr, npr = _pairs(pairs)
    if load().oracle_state_pass(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(B), _ptr(G), _ptr(init),
                                _ptr(cs), _ptr(fin), _ptr(pr), npr, _threads(nthreads)):
        raise ValueError("oracle_state_pass rejected its arguments")
    return cs, fin


def chunk_out(x, dt, B, C, G, chunk_states, chunk_size, D=None, pairs=None, nthreads=None):
    """Stage 3: y [b, L, nh, H] from G and the chunk-start states."""
    x, dt, B, C, D, G, cs = map(_f64, (x, dt, B, C, D, G, chunk_states))
    d = _dims(x, B, chunk_size)
    y = np.zeros_like(x)
    pr, npr = _pairs(pairs)
    if load().oracle_chunk_out(ctypes.byref(d), _ptr(x), _ptr(dt), _ptr(B), _ptr(C), _ptr(D), _ptr(G),
                               _ptr(cs), _ptr(y), _ptr(pr), npr, _threads(nthreads)):
        raise ValueError("oracle_chunk_out rejected its arguments")
    return y


def ssd_chunked(x, dt, A, B, C, chunk_size, D=None, init=None, pairs=None, nthreads=None):
    """Stages 1 -> 2 -> 3 chained.  Returns dict(y, final_state, chunk_states, G)."""
    G = chunk_cumsum(dt, A, chunk_size, pairs=pairs, nthreads=nthreads)
    cs, fin = state_pass(x, dt, B, G, chunk_size, init=init, pairs=pairs, nthreads=nthreads)
    y = chunk_out(x, dt, B, C, G, cs, chunk_size, D=D, pairs=pairs, nthreads=nthreads)
    return {"y": y, "final_state": fin, "chunk_states": cs, "G": G}
