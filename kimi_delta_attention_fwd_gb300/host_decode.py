"""The host decode tool: one KDA decode step on the CPU cores (host/kda_host_decode.c).

A separate tool beside the GPU library: it is built into its own shared library,
takes host (CPU) tensors, and the GPU path neither imports nor calls it.  The
recurrence per (sequence, head), in fp32, with the state updated in place:

  alpha = exp(g),  S~ = Diag(alpha) S,  e = beta (v - S~^T k),  S <- S~ + k e^T,
  o = scale * S^T q
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_PKG, "host", "kda_host_decode.c")
_BUILD_DIR = os.path.join(_PKG, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "libkda_host_decode.so")
GATE_CHANNEL, GATE_SCALAR, GATE_NONE = 0, 1, 2
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the tool with gcc (portable flags: the same code on x86 and Arm hosts)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    deps = [_SRC, os.path.join(_PKG, "host", "kda_host_decode.h")]
    if (not force and os.path.exists(LIB_PATH)
            and all(os.path.getmtime(LIB_PATH) >= os.path.getmtime(d) for d in deps)):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp,
                    "-lm"], check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            fp = ctypes.POINTER(ctypes.c_float)
            lib.kda_host_decode_step.restype = ctypes.c_int
            lib.kda_host_decode_step.argtypes = [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int] + \
                [fp] * 7 + [ctypes.c_int]
            lib.kda_host_decode_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(x, name, shape):
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if a.shape != tuple(shape):
        raise ValueError(f"{name}: shape {a.shape}, expected {tuple(shape)}")
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def decode_step(q, k, v, g, beta, state, scale=None, threads=None):
    """One decode step for N sequences on the CPU.

    q, k: [N, H, d_k]; v: [N, H, d_v]; beta: [N, H]; g: [N, H, d_k] (per key channel),
    [N, H] (one per token and head) or None (alpha = 1); state: float32 numpy array
    [N, H, d_k, d_v], updated in place.  Returns out [N, H, d_v] (float32 numpy)."""
    if not (isinstance(state, np.ndarray) and state.dtype == np.float32 and state.flags.c_contiguous):
        raise TypeError("state must be a C-contiguous float32 numpy array (updated in place)")
    N, H, dk, dv = state.shape
    q = _f32(q, "q", (N, H, dk))
    k = _f32(k, "k", (N, H, dk))
    v = _f32(v, "v", (N, H, dv))
    beta = _f32(beta, "beta", (N, H))
    if g is None:
        gate = GATE_NONE
    elif np.ndim(g) == 2 or (hasattr(g, "dim") and g.dim() == 2):
        gate, g = GATE_SCALAR, _f32(g, "g", (N, H))
    else:
        gate, g = GATE_CHANNEL, _f32(g, "g", (N, H, dk))
    out = np.empty((N, H, dv), dtype=np.float32)
    rc = _load().kda_host_decode_step(N, H, dk, dv, float(scale or 0.0), gate, _p(q), _p(k), _p(v),
                                      _p(g), _p(beta), _p(state), _p(out), int(threads or 0))
    if rc != 0:
        raise RuntimeError(f"kda_host_decode_step failed with status {rc}")
    return out


def default_threads() -> int:
    return int(_load().kda_host_decode_default_threads())
