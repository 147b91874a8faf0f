"""Host-side checks of the C ABI: the library builds for sm_103a, loads without a
GPU, exports every function include/kda.h declares, and rejects bad arguments
before touching the device.  No call here reaches a kernel: every call either
fails validation or has nothing to do."""
import ctypes
import os
import re
import subprocess

import pytest

from kimi_delta_attention_fwd_gb300 import build as kbuild
from kimi_delta_attention_fwd_gb300 import kda as K

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return K.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kda_chunk_fwd", "kda_decode_step", "kda_chunk_fwd_workspace_bytes",
                 "kda_workspace_status", "kda_status_string", "kda_version"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", kbuild.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (kda_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_library_is_sm103a_only():
    src = open(os.path.join(kbuild.PKG, "build.py")).read()
    assert "arch=compute_103a,code=sm_103a" in src


def _shape(**kw):
    d = dict(num_seqs=2, total_tokens=128, num_heads=4, d_k=128, d_v=128, chunk_size=64, scale=0.0,
             io_dtype=1, algo=0)
    d.update(kw)
    return K.kda_shape(**d)


FAKE = 0x10000  # aligned fake device address: never dereferenced (validation fails first)


def _chunk(lib, shape, ptr=FAKE, ws=FAKE, ws_bytes=None, init=None):
    if ws_bytes is None:
        ws_bytes = lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(shape))
    p = ctypes.c_void_p(ptr)
    return lib.kda_chunk_fwd(ctypes.byref(shape), p, p, p, p, p, init, p, p, p,
                             ctypes.c_void_p(ws) if ws else None, ws_bytes, None)


def test_workspace_size(lib):
    n = lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(_shape()))
    assert n >= 256 and n % 16 == 0
    assert lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(_shape(d_k=96))) == 0
    assert lib.kda_chunk_fwd_workspace_bytes(None) == 0


def test_workspace_holds_the_solve_helper_ring_for_few_sequence_heads(lib):
    """Tensor-core path: the status block, one recomputation flag word per
    sequence-head (rounded up to 256 bytes; none without a gate), and with at most 76
    sequence-heads a ring of 4 x 16 KiB and 32 bytes per sequence-head; with more, for 2 to
    2048 sequences, the launch order (4 bytes per sequence, rounded up to 256)."""
    ws = lambda **kw: lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(_shape(**kw)))
    assert ws(num_seqs=1, num_heads=1) == 256 + 256 + 65568
    assert ws(num_seqs=19, num_heads=2) == 256 + 256 + 38 * 65568
    assert ws(num_seqs=13, num_heads=3) == 256 + 256 + 39 * 65568
    assert ws(num_seqs=38, num_heads=2) == 256 + 512 + 76 * 65568   # the most with a ring
    assert ws(num_seqs=11, num_heads=7) == 256 + 512 + 256           # 77 sequence-heads: no ring
    assert ws(num_seqs=1, num_heads=32) == 256 + 256 + 32 * 65568
    assert ws(num_seqs=64, num_heads=32) == 256 + 2048 * 4 + 256  # flags, launch order
    assert ws(num_seqs=2048, num_heads=1) == 256 + 2048 * 4 + 2048 * 4  # the most sequences ordered
    assert ws(num_seqs=2049, num_heads=1) == 256 + 8448  # flags only: too many to order
    assert ws(num_seqs=1, num_heads=1, gate=K.KDA_GATE_NONE) == 256 + 65568  # no decay, no flag
    assert ws(num_seqs=1, num_heads=1, algo=K._ALGOS["simt"]) == 256
    assert ws(num_seqs=1, num_heads=1, io_dtype=K.KDA_F32) == 256  # CUDA-core path


def test_workspace_holds_the_segments_of_one_long_sequence(lib):
    """Sequences of at least 3 x 32 chunks on average with at most 50 sequence-heads: for
    P = min((SMs / (N H) + 3) / 2, average chunks / 32) >= 3 segments per sequence, the run
    tables and the pairs to skip (16 bytes per run slot, 3 slots per segment and sequence,
    4 bytes per sequence-head, rounded up to 256), 4P - 5 fp32 states per sequence-head, and
    a solve-helper ring for the larger of the two passes (2P - 3 and P - 1 runs per
    sequence-head) that has at most 76 pairs.  Without a device the size is taken for 152
    SMs."""
    ws = lambda **kw: lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(_shape(num_seqs=1, **kw)))
    st, ring = 128 * 128 * 4, 65568
    assert ws(num_heads=4, total_tokens=65536) == 512 + 1024 + 75 * 4 * st + 76 * ring    # P = 20
    assert ws(num_heads=32, total_tokens=65536) == 512 + 512 + 7 * 32 * st + 64 * ring   # P = 3
    assert ws(num_heads=2, total_tokens=64 * 96) == 512 + 256 + 7 * 2 * st + 6 * ring    # 96 chunks
    assert ws(num_heads=2, total_tokens=64 * 95) == 512 + 2 * ring                       # the ring only
    assert ws(num_heads=1, total_tokens=1 << 20) == 512 + 3840 + 303 * st + 76 * ring    # P = 77
    assert ws(num_heads=51, total_tokens=1 << 20) == 512 + 51 * ring                     # no segments
    assert ws(num_heads=4, total_tokens=65536, gate=K.KDA_GATE_NONE) == 256 + 1024 + 75 * 4 * st + 76 * ring
    # several sequences: P from the average length, N H (2P - 3) runs in the first pass
    ws2 = lambda **kw: lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(_shape(**kw)))
    assert ws2(num_seqs=2, num_heads=2, total_tokens=20014) == 512 + 512 + 11 * 4 * st + 20 * ring   # P = 4
    assert ws2(num_seqs=3, num_heads=1, total_tokens=18500) == 512 + 512 + 7 * 3 * st + 9 * ring    # P = 3
    assert ws2(num_seqs=2, num_heads=26, total_tokens=1 << 20) == 512 + 52 * ring                   # 52 pairs: no
    assert ws2(num_seqs=64, num_heads=32, total_tokens=1 << 20) == 256 + 8192 + 256                 # varlen: order
    # 2^30 tokens or more: no segments (their zero V tiles are read below token 0)
    assert ws2(num_seqs=1, num_heads=1, total_tokens=(1 << 30) - 64) == 512 + 3840 + 303 * st + 76 * ring
    assert ws2(num_seqs=1, num_heads=1, total_tokens=1 << 30) == 512 + ring
    assert lib.kda_version() >= 1005  # 1.5 added the segments


def test_status_block_alone_is_an_accepted_workspace(lib):
    """256 bytes select the plain schedule; fewer are rejected before any device call."""
    s = _shape(num_seqs=1, num_heads=1)
    assert _chunk(lib, s, ws_bytes=255) == -4


@pytest.mark.parametrize("bad", [dict(d_k=96), dict(d_v=32), dict(num_heads=0), dict(num_seqs=-1),
                                 dict(chunk_size=128), dict(io_dtype=5), dict(algo=9),
                                 dict(total_tokens=-3), dict(gate=3), dict(gate=-1)])
def test_rejects_bad_shapes(lib, bad):
    assert _chunk(lib, _shape(**bad)) == -2


def test_rejects_null_and_small_workspace_and_misalignment(lib):
    s = _shape()
    assert lib.kda_chunk_fwd(None, None, None, None, None, None, None, None, None, None, None, 0,
                             None) == -1
    assert _chunk(lib, s, ptr=0) == -1                     # q == NULL with tokens > 0
    assert _chunk(lib, s, ws=0) == -4                      # no workspace
    assert _chunk(lib, s, ws_bytes=8) == -4                # too small
    assert _chunk(lib, s, ptr=FAKE + 4) == -3              # misaligned tensors
    assert _chunk(lib, s, ws=FAKE + 8) == -3               # misaligned workspace


def test_recurrent_validation(lib):
    """kda_recurrent_fwd rejects bad arguments before touching the device, and with
    neither outputs nor a final state there is nothing to do."""
    s = _shape()
    p = ctypes.c_void_p(FAKE)

    def rec(shape, q=p, init=None, cu=p, acc=None, out=p, fin=p):
        return lib.kda_recurrent_fwd(ctypes.byref(shape) if shape is not None else None, q, q, q, q,
                                     q, init, cu, acc, out, fin, None)
    assert rec(None) == -1
    assert rec(_shape(d_k=96)) == -2
    assert rec(_shape(gate=5)) == -2
    assert rec(s, out=None, fin=None) == 0                      # nothing to produce: no launch
    assert rec(s, q=None) == -1
    assert rec(s, cu=None) == -1
    assert rec(s, q=ctypes.c_void_p(FAKE + 1)) == -3           # q not on its element size
    assert rec(s, fin=ctypes.c_void_p(FAKE + 8)) == -3         # states on 16 bytes
    assert rec(s, acc=ctypes.c_void_p(FAKE + 2)) == -3         # accepted on 4 bytes
    assert rec(s, out=ctypes.c_void_p(FAKE + 2)) == -3         # outputs on 4 elements


def test_decode_validation(lib):
    s = _shape(total_tokens=2)
    p = ctypes.c_void_p(FAKE)
    assert lib.kda_decode_step(ctypes.byref(_shape(total_tokens=3)), p, p, p, p, p, p, p, None) == -2
    assert lib.kda_decode_step(ctypes.byref(s), None, p, p, p, p, p, p, None) == -1
    odd = ctypes.c_void_p(FAKE + 1)
    assert lib.kda_decode_step(ctypes.byref(s), odd, p, p, p, p, p, p, None) == -3  # q not 2-aligned
    two = ctypes.c_void_p(FAKE + 2)
    assert lib.kda_decode_step(ctypes.byref(s), p, p, p, p, p, two, p, None) == -3  # state not 16-aligned
    assert lib.kda_decode_step(ctypes.byref(s), p, p, p, p, p, p, two, None) == -3  # out not 8-aligned
    # no sequences: nothing to do, nothing touched
    assert lib.kda_decode_step(ctypes.byref(_shape(num_seqs=0, total_tokens=0)), None, None, None,
                               None, None, None, None, None) == 0


def test_status_strings(lib):
    seen = set()
    for code in range(0, -12, -1):
        s = lib.kda_status_string(code).decode()
        assert s and s != "unknown status"
        seen.add(s)
    assert len(seen) == 12
    assert lib.kda_status_string(-99).decode() == "unknown status"
    assert lib.kda_workspace_status(None, None) == -1
    assert lib.kda_version() >= 1003  # 1.3 added the device check of the offsets


def test_gate_modes_validation(lib):
    """g is required (and 16-byte aligned for the prefill) with one log alpha per key
    channel, required on its element size with one per token, and not read at all
    without a gate (DeltaNet): NULL and odd addresses then pass validation, which
    reaches the device check (-6, no GPU here)."""
    p = ctypes.c_void_p(FAKE)
    s_chan, s_tok, s_none = _shape(gate=0), _shape(gate=1), _shape(gate=2)

    def chunk_g(shape, g):
        ws = lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(shape))
        return lib.kda_chunk_fwd(ctypes.byref(shape), p, p, p, g, p, None, p, p, p, p, ws, None)

    assert chunk_g(s_chan, None) == -1
    assert chunk_g(s_tok, None) == -1
    assert chunk_g(s_chan, ctypes.c_void_p(FAKE + 2)) == -3   # per channel: 16-byte aligned
    assert chunk_g(s_tok, ctypes.c_void_p(FAKE + 2)) == -6    # per token: element aligned
    assert chunk_g(s_tok, ctypes.c_void_p(FAKE + 1)) == -3
    assert chunk_g(s_none, None) == -6
    assert chunk_g(s_none, ctypes.c_void_p(FAKE + 1)) == -6   # not read
    d = _shape(total_tokens=2, gate=2)
    assert lib.kda_decode_step(ctypes.byref(d), p, p, p, None, p, p, p, None) == -6
    d = _shape(total_tokens=2, gate=1)
    assert lib.kda_decode_step(ctypes.byref(d), p, p, p, None, p, p, p, None) == -1


def test_prep_bits_validation(lib):
    """kda_shape.prep takes the four KDA_PREP_* bits in any combination; any other
    bit, or a gate scale that is not finite, is a shape error on every entry point
    (before the device check, -6 here)."""
    assert lib.kda_version() >= 1004  # 1.4 added KDA_PREP_G_SOFTPLUS and kda_shape.gate_scale
    assert ctypes.sizeof(K.kda_shape) == 48
    p = ctypes.c_void_p(FAKE)
    for bits in range(16):
        s = _shape(prep=bits)
        ws = lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(s))
        assert ws >= 256
        assert lib.kda_chunk_fwd(ctypes.byref(s), p, p, p, p, p, None, p, p, p, p, ws, None) == -6
        d = _shape(total_tokens=2, prep=bits)
        assert lib.kda_decode_step(ctypes.byref(d), p, p, p, p, p, p, p, None) == -6
    for bad in (dict(prep=16), dict(prep=-1), dict(gate_scale=float("inf")),
                dict(gate_scale=float("nan"))):
        s = _shape(**bad)
        bits = bad.get("prep", 0)
        assert lib.kda_chunk_fwd_workspace_bytes(ctypes.byref(s)) == 0
        assert lib.kda_chunk_fwd(ctypes.byref(s), p, p, p, p, p, None, p, p, p, p, 256, None) == -2
        d = _shape(total_tokens=2, **bad)
        assert lib.kda_decode_step(ctypes.byref(d), p, p, p, p, p, p, p, None) == -2
        assert lib.kda_recurrent_fwd(ctypes.byref(s), p, p, p, p, p, None, p, None, p, None,
                                     None) == -2
    assert K._prep_bits(True, True, True) == 7 and K._prep_bits(False, True, False) == 2
    assert K._prep_bits(False, False, False, True) == 8
