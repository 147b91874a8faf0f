"""fp64 CPU oracle for the Kimi Delta Attention (KDA) forward recurrence.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use this package; the library path never does.
It shares no code with the CUDA library.

The arithmetic lives in ``kda_oracle.c`` (a plain sequential loop over tokens,
one (sequence, head) pair per thread).  It follows the recurrence of
"Kimi Delta Attention (KDA)" (brain.bigb.es): the opening equation and the
five-line reference recurrence written in the d_k x d_v state layout, with
forget -> predict -> correct -> write -> read after write.  This module only
compiles that file, widens inputs exactly to float64 and calls it.

Every function here is pinned by ``tests/test_oracle_pins.py`` (invariants stated
on that page, the worked example of "K3 架构图解" Ch.08, an exact rational
brute force over the DPLR transition product, and an independent chunkwise
schedule).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into a shared library with gcc (no -march flags,
    no FP contraction, so x86 and Arm hosts agree bit for bit)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_fwd.restype = ctypes.c_int
            lib.kda_oracle_fwd.argtypes = [
                ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, dp, dp, dp, dp, dp,
                dp, dp, dp, ctypes.c_int]
            lib.kda_oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    """Host threads the oracle uses by default (one per online core)."""
    return int(_load().kda_oracle_default_threads())


def _f64(x):
    """Exact widening of a CPU tensor / array (fp32, bf16, fp64) to float64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: bf16 has no numpy dtype
        x = x.detach().to("cpu")
        import torch  # local: the oracle itself needs only numpy
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def kda_fwd(q, k, v, g, beta, cu_seqlens, init_state=None, scale=None,
            threads: int | None = None, want_state: bool = True):
    """Run the recurrence over packed variable-length sequences.

    q, k, g: [T, H, d_k]; v: [T, H, d_v]; beta: [T, H]; cu_seqlens: [N+1];
    init_state: [N, H, d_k, d_v] or None (zeros); scale None -> d_k ** -0.5.
    Returns (out [T, H, d_v] float64, final_state [N, H, d_k, d_v] float64 or None).
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    init = _f64(init_state)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu.shape[0] - 1
    assert k.shape == (T, H, dk) and g.shape == (T, H, dk)
    assert v.shape == (T, H, dv) and beta.shape == (T, H)
    assert N >= 0 and (N == 0 or cu[-1] <= T)
    if init is not None:
        assert init.shape == (N, H, dk, dv)
    if scale is None:
        scale = dk ** -0.5
    out = np.zeros((T, H, dv), dtype=np.float64)
    fin = np.zeros((N, H, dk, dv), dtype=np.float64) if want_state else None
    rc = _load().kda_oracle_fwd(
        N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), H, dk, dv,
        float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init),
        _ptr(out), _ptr(fin), int(threads or 0))
    if rc < 0:
        raise ValueError("kda_oracle_fwd rejected its arguments")
    return out, fin


def preprocess(q, k, beta, qk_silu=False, qk_l2norm=False, beta_sigmoid=False):
    """The weight-free input steps of the module around the recurrence, in fp64.

    "22580: от GPT-2 до Kimi K3" (temp07.ru), section "DeltaNet, или Fast Weight
    Programmers", the forward with a per-token write strength: q and k go through
    SiLU and are then L2-normalised over the key dimension of each (token, head)
    (F.normalize: x / max(||x||_2, 1e-12)), and beta is the sigmoid of a logit.
    "K3 架构图解" Ch.08 notes that the real KDA module also has these
    normalisations.  Each step is optional, in that order: silu, then the norm.

    q, k: [..., d_k]; beta: any shape.  Returns float64 (q, k, beta).
    """
    q, k, beta = map(_f64, (q, k, beta))
    with np.errstate(over="ignore"):
        if qk_silu:  # silu(x) = x * sigmoid(x) = x / (1 + e^-x)
            q = q / (1.0 + np.exp(-q))
            k = k / (1.0 + np.exp(-k))
        if beta_sigmoid:
            beta = 1.0 / (1.0 + np.exp(-beta))
    if qk_l2norm:
        q = q / np.maximum(np.sqrt(np.sum(q * q, axis=-1, keepdims=True)), 1e-12)
        k = k / np.maximum(np.sqrt(np.sum(k * k, axis=-1, keepdims=True)), 1e-12)
    return q, k, beta


def gate_from_logits(x, gate_scale=1.0):
    """log alpha from gate logits, in fp64: -c * softplus(x), softplus(x) = log(1 + e^x),
    taken in the overflow-free form max(x, 0) + log1p(e^-|x|).

    The pages give the decay only as alpha_t in [0, 1] per key channel ("Kimi Delta
    Attention (KDA)", Gated DeltaNet and KDA sections: alpha = 1 keeps, alpha = 0
    clears memory); the workloads draw it as exp(-c * softplus(x)) of a normal x, a
    positive decay rate made so by softplus.  This is that map, for the kernels'
    optional gate step (KDA_PREP_G_SOFTPLUS).  x: any shape.  Returns float64.
    """
    x = _f64(x)
    return -float(gate_scale) * (np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x))))


def kda_decode_steps(q, k, v, g, beta, state, scale=None, threads=None):
    """Consecutive single-token steps for N independent sequences.

    q, k, g: [steps, N, H, d_k]; v: [steps, N, H, d_v]; beta: [steps, N, H];
    state: [N, H, d_k, d_v] (the state before the first step).
    A run of decode steps is the recurrence over a sequence of `steps` tokens,
    so this packs each sequence's tokens contiguously and calls kda_fwd.
    Returns (out [steps, N, H, d_v], state after the last step [N, H, d_k, d_v]).
    """
    q, k, v, g, beta = map(_f64, (q, k, v, g, beta))
    steps, N, H, dk = q.shape
    dv = v.shape[3]

    def pack(x):  # [steps, N, ...] -> [N * steps, ...], sequence-major
        return np.ascontiguousarray(np.swapaxes(x, 0, 1).reshape((N * steps,) + x.shape[2:]))

    cu = np.arange(N + 1, dtype=np.int64) * steps
    out, fin = kda_fwd(pack(q), pack(k), pack(v), pack(g), pack(beta), cu,
                       init_state=state, scale=scale, threads=threads)
    out = np.ascontiguousarray(np.swapaxes(out.reshape(N, steps, H, dv), 0, 1))
    return out, fin
