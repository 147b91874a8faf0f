"""Thin Python binding of the C ABI in include/kda.h (argument marshalling only).

Every step of the computation runs in the CUDA kernels of libkda_gb300.so;
this module checks tensor metadata, allocates outputs with PyTorch when the
caller did not pass them, and forwards raw device pointers and the CUDA stream.
There is no CPU path: without the built library every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

KDA_OK = 0
KDA_ERR_GATE_RANGE, KDA_ERR_SEQLENS = -8, -11
KDA_F32, KDA_BF16 = 0, 1
KDA_GATE_CHANNEL, KDA_GATE_SCALAR, KDA_GATE_NONE = 0, 1, 2
KDA_PREP_QK_SILU, KDA_PREP_QK_L2NORM, KDA_PREP_BETA_SIGMOID, KDA_PREP_G_SOFTPLUS = 1, 2, 4, 8
_ALGOS = {"auto": 0, "tensor": 1, "simt": 2}
_DTYPES = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16}


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {kda_status_string(code)} (status {code})")


class kda_shape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("num_heads", ctypes.c_int32), ("d_k", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("chunk_size", ctypes.c_int32), ("scale", ctypes.c_float),
                ("io_dtype", ctypes.c_int32), ("algo", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("prep", ctypes.c_int32), ("gate_scale", ctypes.c_float)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library():
    """Load libkda_gb300.so (built by __graft_entry__.build() or build.py)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"KDA CUDA library not built ({path} missing); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(path)
        vp, sp = ctypes.c_void_p, ctypes.POINTER(kda_shape)
        lib.kda_chunk_fwd.restype = ctypes.c_int
        lib.kda_chunk_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.kda_chunk_fwd_workspace_bytes.restype = ctypes.c_size_t
        lib.kda_chunk_fwd_workspace_bytes.argtypes = [sp]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.kda_recurrent_fwd.restype = ctypes.c_int
        lib.kda_recurrent_fwd.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.kda_workspace_status.restype = ctypes.c_int
        lib.kda_workspace_status.argtypes = [vp, vp]
        lib.kda_last_device_status.restype = ctypes.c_int
        lib.kda_last_device_status.argtypes = [vp]
        lib.kda_chunk_fwd_noalloc.restype = ctypes.c_int
        lib.kda_chunk_fwd_noalloc.argtypes = [sp] + [vp] * 10
        lib.kda_noalloc_status.restype = ctypes.c_int
        lib.kda_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), vp]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_status_string.argtypes = [ctypes.c_int]
        lib.kda_version.restype = ctypes.c_int
        lib.kda_chunk_fwd_selected_algo.restype = ctypes.c_int
        lib.kda_chunk_fwd_selected_algo.argtypes = [sp]
        _lib = lib
        return lib


def kda_status_string(code: int) -> str:
    return load_library().kda_status_string(int(code)).decode()


def kda_version() -> int:
    return int(load_library().kda_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _make_shape(num_seqs, total_tokens, H, dk, dv, scale, io, algo="auto", gate=0, prep=0,
                gate_scale=None):
    return kda_shape(int(num_seqs), int(total_tokens), int(H), int(dk), int(dv), 64,
                     float(scale) if scale is not None else 0.0, io, _ALGOS[algo], int(gate),
                     int(prep), float(gate_scale) if gate_scale is not None else 0.0)


def _prep_bits(qk_silu, qk_l2norm, beta_sigmoid, g_softplus=False):
    """KDA_PREP_* bits of the optional input steps (see include/kda.h)."""
    return ((KDA_PREP_QK_SILU if qk_silu else 0) | (KDA_PREP_QK_L2NORM if qk_l2norm else 0)
            | (KDA_PREP_BETA_SIGMOID if beta_sigmoid else 0)
            | (KDA_PREP_G_SOFTPLUS if g_softplus else 0))


def _gate_of(g, lead, H, dk):
    """kda_gate of g: None -> no gate (DeltaNet), [lead, H] -> one log alpha per
    (token, head) (Gated DeltaNet), [lead, H, d_k] -> one per key channel (KDA)."""
    if g is None:
        return KDA_GATE_NONE, None
    if g.dim() == 2:
        return KDA_GATE_SCALAR, (lead, H)
    return KDA_GATE_CHANNEL, (lead, H, dk)


def _check_io(name, t, shape, dtype, device):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _check_workspace(ws, device):
    """The caller's prefill workspace: device memory on the tensors' device, contiguous."""
    if ws.device != device:
        raise ValueError(f"workspace is on {ws.device}, expected {device}")
    if not ws.is_contiguous():
        raise ValueError("workspace must be contiguous")


def _check_ranks(where, **tensors):
    """Each named tensor (None allowed where the entry point allows it) has the rank
    given with it, checked before any shape is unpacked."""
    for name, (t, ranks) in tensors.items():
        if t is not None and t.dim() not in ranks:
            want = " or ".join(str(r) for r in ranks)
            raise ValueError(f"{where}: {name} has {t.dim()} dimensions, expected {want}")


def _check_cu_seqlens(cu, total_tokens):
    """Host check of packed-sequence offsets (a CPU int32 [N + 1] tensor): they start at
    0, never decrease and stay within the token count, so that no kernel indexes past
    the buffers (the library itself reads them on the device only, unchecked)."""
    c = [int(x) for x in cu.tolist()]
    if not c or c[0] != 0:
        raise ValueError("cu_seqlens must start at 0")
    if any(b < a for a, b in zip(c, c[1:])):
        raise ValueError("cu_seqlens must be nondecreasing")
    if c[-1] > total_tokens:
        raise ValueError(f"cu_seqlens ends at {c[-1]}, beyond the {total_tokens} tokens")


def kda_chunk_fwd_workspace_bytes(num_seqs, total_tokens, num_heads, d_k, d_v, io_dtype=torch.bfloat16,
                                  algo="auto") -> int:
    shape = _make_shape(num_seqs, total_tokens, num_heads, d_k, d_v, None, _DTYPES[io_dtype], algo)
    n = int(load_library().kda_chunk_fwd_workspace_bytes(ctypes.byref(shape)))
    if n == 0:
        raise KdaError(-2, "kda_chunk_fwd_workspace_bytes")
    return n


def kda_chunk_fwd_selected_algo(num_seqs, total_tokens, num_heads, d_k, d_v, io_dtype=torch.bfloat16,
                                algo="auto") -> str:
    """Which prefill kernel a call with these sizes runs: "tensor" or "simt"."""
    shape = _make_shape(num_seqs, total_tokens, num_heads, d_k, d_v, None, _DTYPES[io_dtype], algo)
    r = int(load_library().kda_chunk_fwd_selected_algo(ctypes.byref(shape)))
    if r < 0:
        raise KdaError(r, "kda_chunk_fwd_selected_algo")
    return {1: "tensor", 2: "simt"}[r]


def kda_chunk_fwd(q, k, v, g, beta, cu_seqlens, init_state=None, *, out=None, final_state=None,
                  output_final_state=True, workspace=None, scale=None, algo="auto", stream=None,
                  check=False, qk_silu=False, qk_l2norm=False, beta_sigmoid=False,
                  g_softplus=False, gate_scale=None):
    """Chunkwise prefill over packed sequences (see include/kda.h).

    q, k: [T, H, d_k]; v: [T, H, d_v]; beta: [T, H] (one dtype: bf16 or fp32, CUDA);
    g: [T, H, d_k] (one log alpha per key channel), [T, H] (one per token and head,
    Gated DeltaNet) or None (alpha = 1, DeltaNet);
    cu_seqlens: int32 [N+1] (CUDA); init_state: fp32 [N, H, d_k, d_v] or None.
    final_state may be the init_state tensor itself (in-place update).
    qk_silu, qk_l2norm, beta_sigmoid: the kernels apply silu and then the L2 norm
    to each (token, head) row of q and k, and read beta as logits (KDA_PREP_*).
    g_softplus: g holds gate logits x and log alpha = -gate_scale * softplus(x)
    (gate_scale None or <= 0: 1).
    Returns (out, final_state or None).  With check=True the call first reads
    cu_seqlens back and checks it on the host, then synchronises after the launch and
    raises if a kernel recorded a device-side error in the workspace.
    """
    _check_ranks("kda_chunk_fwd", q=(q, (3,)), k=(k, (3,)), v=(v, (3,)), g=(g, (2, 3)),
                 beta=(beta, (2,)), cu_seqlens=(cu_seqlens, (1,)))
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.shape[0] - 1
    dev = q.device
    if dev.type != "cuda":
        raise ValueError("kda_chunk_fwd runs on CUDA tensors only")
    dt = q.dtype
    if dt not in _DTYPES:
        raise TypeError(f"unsupported I/O dtype {dt}")
    gate, gshape = _gate_of(g, T, H, dk)
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("g", g, gshape),
                         ("v", v, (T, H, dv)), ("beta", beta, (T, H))):
        if t is not None:
            _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    if check:
        _check_cu_seqlens(cu_seqlens.cpu(), T)
    if init_state is not None:
        _check_io("init_state", init_state, (N, H, dk, dv), torch.float32, dev)
    shape = _make_shape(N, T, H, dk, dv, scale, _DTYPES[dt], algo, gate,
                        _prep_bits(qk_silu, qk_l2norm, beta_sigmoid, g_softplus), gate_scale)
    lib = load_library()
    need = int(lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(shape)))
    # what is allocated here belongs to the stream the kernels run on, so that the
    # caching allocator does not hand it to other work before they are done with it
    with torch.cuda.stream(stream):
        if out is None:
            out = torch.empty((T, H, dv), dtype=dt, device=dev)
        if final_state is None and output_final_state:
            final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        else:
            _check_workspace(workspace, dev)
    _check_io("out", out, (T, H, dv), dt, dev)
    if final_state is not None:
        _check_io("final_state", final_state, (N, H, dk, dv), torch.float32, dev)
    rc = lib.kda_chunk_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(init_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd")
    if check:
        st = kda_workspace_status(workspace, stream)
        if st != KDA_OK:
            raise KdaError(st, "kda_chunk_fwd (device status)")
    return out, final_state


def kda_workspace_status(workspace, stream=None) -> int:
    """Synchronises the stream and returns the device status of the last
    kda_chunk_fwd that used this workspace."""
    if workspace.device.type != "cuda":
        raise ValueError("kda_workspace_status reads a CUDA workspace only")
    return int(load_library().kda_workspace_status(_ptr(workspace), _stream(stream)))


def workspace_status_words(workspace, stream=None):
    """Synchronises the stream and returns the four status words of a prefill
    workspace: (first error, detail, tensor-core schedule that ran (1 plain, 2 solve
    helpers, 3 segment-parallel scan, 0 CUDA-core path), sequence-heads recomputed
    token by token)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    s.synchronize()
    w = workspace[:16].cpu().view(torch.int32).tolist()
    return tuple(int(x) for x in w)


def kda_last_device_status(stream=None) -> int:
    """Synchronises the stream, then returns and clears the first error the
    kda_recurrent_fwd kernels recorded on the current device (0 or -11)."""
    return int(load_library().kda_last_device_status(_stream(stream)))


def kda_decode_step(q, k, v, g, beta, state, *, out=None, scale=None, stream=None, qk_silu=False,
                    qk_l2norm=False, beta_sigmoid=False, g_softplus=False, gate_scale=None):
    """One single-token step for N sequences: q, k [N, H, d_k]; v [N, H, d_v];
    g [N, H, d_k], [N, H] or None (as for kda_chunk_fwd); beta [N, H];
    state fp32 [N, H, d_k, d_v] updated in place.  The input steps as for
    kda_chunk_fwd.  Returns out [N, H, d_v]."""
    _check_ranks("kda_decode_step", q=(q, (3,)), k=(k, (3,)), v=(v, (3,)), g=(g, (2, 3)),
                 beta=(beta, (2,)), state=(state, (4,)))
    N, H, dk = q.shape
    dv = v.shape[2]
    dev, dt = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("kda_decode_step runs on CUDA tensors only")
    if dt not in _DTYPES:
        raise TypeError(f"unsupported I/O dtype {dt}")
    gate, gshape = _gate_of(g, N, H, dk)
    for name, t, shp in (("q", q, (N, H, dk)), ("k", k, (N, H, dk)), ("g", g, gshape),
                         ("v", v, (N, H, dv)), ("beta", beta, (N, H))):
        if t is not None:
            _check_io(name, t, shp, dt, dev)
    _check_io("state", state, (N, H, dk, dv), torch.float32, dev)
    if out is None:
        with torch.cuda.stream(stream):  # allocated on the stream the kernel runs on
            out = torch.empty((N, H, dv), dtype=dt, device=dev)
    _check_io("out", out, (N, H, dv), dt, dev)
    shape = _make_shape(N, N, H, dk, dv, scale, _DTYPES[dt], gate=gate,
                        prep=_prep_bits(qk_silu, qk_l2norm, beta_sigmoid, g_softplus),
                        gate_scale=gate_scale)
    rc = load_library().kda_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                        _ptr(beta), _ptr(state), _ptr(out), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step")
    return out


def kda_recurrent_fwd(q, k, v, g, beta, cu_seqlens, init_state=None, *, accepted=None, out=None,
                      final_state=None, output=True, output_final_state=True, scale=None,
                      stream=None, qk_silu=False, qk_l2norm=False, beta_sigmoid=False,
                      g_softplus=False, gate_scale=None):
    """The recurrence token by token over short packed sequences (see include/kda.h):
    the same tensors as kda_chunk_fwd, plus accepted (int32 [N], CUDA, or None): the
    state returned for sequence n is the one after its first accepted[n] tokens.
    output=False skips the outputs (the commit of a speculative step);
    output_final_state=False leaves every state untouched (the verify).
    final_state may be the init_state tensor itself.  The input steps as for
    kda_chunk_fwd.  Returns (out or None, final_state or None)."""
    _check_ranks("kda_recurrent_fwd", q=(q, (3,)), k=(k, (3,)), v=(v, (3,)), g=(g, (2, 3)),
                 beta=(beta, (2,)), cu_seqlens=(cu_seqlens, (1,)))
    T, H, dk = q.shape
    dv = v.shape[2]
    N = cu_seqlens.shape[0] - 1
    dev, dt = q.device, q.dtype
    if dev.type != "cuda":
        raise ValueError("kda_recurrent_fwd runs on CUDA tensors only")
    if dt not in _DTYPES:
        raise TypeError(f"unsupported I/O dtype {dt}")
    gate, gshape = _gate_of(g, T, H, dk)
    for name, t, shp in (("q", q, (T, H, dk)), ("k", k, (T, H, dk)), ("g", g, gshape),
                         ("v", v, (T, H, dv)), ("beta", beta, (T, H))):
        if t is not None:
            _check_io(name, t, shp, dt, dev)
    _check_io("cu_seqlens", cu_seqlens, (N + 1,), torch.int32, dev)
    if accepted is not None:
        _check_io("accepted", accepted, (N,), torch.int32, dev)
    if init_state is not None:
        _check_io("init_state", init_state, (N, H, dk, dv), torch.float32, dev)
    with torch.cuda.stream(stream):  # allocated on the stream the kernel runs on
        if output:
            if out is None:
                out = torch.empty((T, H, dv), dtype=dt, device=dev)
            _check_io("out", out, (T, H, dv), dt, dev)
        else:
            out = None
        if output_final_state:
            if final_state is None:
                final_state = torch.empty((N, H, dk, dv), dtype=torch.float32, device=dev)
            _check_io("final_state", final_state, (N, H, dk, dv), torch.float32, dev)
        else:
            final_state = None
    shape = _make_shape(N, T, H, dk, dv, scale, _DTYPES[dt], gate=gate,
                        prep=_prep_bits(qk_silu, qk_l2norm, beta_sigmoid, g_softplus),
                        gate_scale=gate_scale)
    rc = load_library().kda_recurrent_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                          _ptr(beta), _ptr(init_state), _ptr(cu_seqlens),
                                          _ptr(accepted), _ptr(out), _ptr(final_state),
                                          _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_recurrent_fwd")
    return out, final_state
