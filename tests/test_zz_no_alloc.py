"""kda_chunk_fwd_noalloc: the prefill entry point for callers that cannot
allocate device memory (they own only their inputs and outputs, e.g. a
framework whose device memory is all reserved by its own allocator).  It takes
its scratch from a buffer built into the library instead of a caller workspace.

Called through the C ABI and compared with kda_chunk_fwd on the same inputs,
twice in a row (the built-in buffer keeps the previous call's contents, so the
second call checks that each call starts from a clean status block).  This file
sorts last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import build as kbuild
from kimi_delta_attention_fwd_gb300 import kda as K
from kimi_delta_attention_fwd_gb300 import kda_chunk_fwd
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, rel_l2_per_head, rel_l2_states, to_dev

pytestmark = pytest.mark.gpu


def _noalloc(lib, d, out, fin):
    T, H, dk = d["q"].shape
    dv = d["v"].shape[2]
    N = d["cu_seqlens"].shape[0] - 1
    gate = K.KDA_GATE_SCALAR if d["g"].dim() == 2 else K.KDA_GATE_CHANNEL
    shape = K.kda_shape(N, T, H, dk, dv, 64, 0.0, K.KDA_BF16, 0, gate)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    rc = lib.kda_chunk_fwd_noalloc(ctypes.byref(shape), p(d["q"]), p(d["k"]), p(d["v"]), p(d["g"]),
                                   p(d["beta"]), p(d["init_state"]), p(d["cu_seqlens"]), p(out),
                                   p(fin), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc


def test_noalloc_matches_kda_chunk_fwd_on_two_calls():
    kbuild.build()
    lib = K.load_library()
    for seed, lens in ((51, [300, 1, 129]), (52, [64, 1000])):
        x = W.prefill_inputs(W.custom_prefill(lens, num_heads=3, d=128, seed=seed))
        d = to_dev(x)
        ref_o, ref_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                     d["init_state"], check=True)
        out = torch.full_like(ref_o, float("nan"))
        fin = torch.full_like(ref_f, float("nan"))
        assert _noalloc(lib, d, out, fin) == 0
        torch.cuda.synchronize()
        cu = x["cu_seqlens"].numpy()
        assert rel_l2_per_head(out.float().cpu().numpy(), ref_o.float().cpu().numpy(), cu) <= TOL_BF16
        assert rel_l2_states(fin.cpu().numpy(), ref_f.cpu().numpy()) <= TOL_BF16
        assert np.isfinite(out.float().cpu().numpy()).all()


def _noalloc_words(lib):
    """Status of the last no-allocation call: (rc, the block's first four words)."""
    words = (ctypes.c_uint32 * 4)()
    rc = lib.kda_noalloc_status(words, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, tuple(words)


def test_noalloc_runs_the_schedule_that_fits_its_buffer():
    """Up to 3 sequence-heads the solve helpers' ring fits the 256 KiB buffer and the
    helper schedule runs; with more the plain one does (the status block records which,
    read back through kda_noalloc_status).  Both give the results of kda_chunk_fwd's
    plain schedule (a 256-byte workspace) bit for bit."""
    kbuild.build()
    lib = K.load_library()
    assert K.kda_chunk_fwd_workspace_bytes(1, 700, 3, 128, 128) <= 256 * 1024  # ring fits: helpers
    assert K.kda_chunk_fwd_workspace_bytes(1, 700, 4, 128, 128) > 256 * 1024   # plain
    for H in (3, 4):
        x = W.prefill_inputs(W.custom_prefill([700], num_heads=H, d=128, gate="mixed", seed=53 + H))
        d = to_dev(x)
        ws = torch.empty(256, dtype=torch.uint8, device="cuda")
        ref_o, ref_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                     d["init_state"], workspace=ws, check=True)
        out = torch.full_like(ref_o, float("nan"))
        fin = torch.full_like(ref_f, float("nan"))
        assert _noalloc(lib, d, out, fin) == 0
        rc, words = _noalloc_words(lib)
        assert rc == 0 and words[0] == 0
        assert words[2] == (2 if H == 3 else 1), words  # 2: solve helpers, 1: plain
        assert torch.equal(out, ref_o) and torch.equal(fin, ref_f)


def test_noalloc_long_sequence_keeps_one_chain():
    """One sequence long enough for the segment-parallel scan: the built-in buffer has no
    room for the segments, so the call runs one chain (with the helpers' ring, which fits)
    and gives kda_chunk_fwd's plain results bit for bit."""
    kbuild.build()
    lib = K.load_library()
    T, H = 10007, 2
    assert K.kda_chunk_fwd_workspace_bytes(1, T, H, 128, 128) > 256 * 1024  # segments: no room
    x = W.prefill_inputs(W.custom_prefill([T], num_heads=H, d=128, gate="mixed", seed=58))
    d = to_dev(x)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    ref_o, ref_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 d["init_state"], workspace=ws, check=True)
    out = torch.full_like(ref_o, float("nan"))
    fin = torch.full_like(ref_f, float("nan"))
    assert _noalloc(lib, d, out, fin) == 0
    rc, words = _noalloc_words(lib)
    assert rc == 0 and words[0] == 0 and words[2] == 2, words  # solve helpers
    assert torch.equal(out, ref_o) and torch.equal(fin, ref_f)


def test_noalloc_reports_device_status_and_recomputes_beyond_the_decay_range():
    """A sequence-head whose chunk decay passes the tensor-core range (g = -2 per token:
    -128 per chunk) is recomputed token by token through the built-in buffer too: the
    status is clear, word 3 counts the one recomputed sequence-head, and the results
    match kda_chunk_fwd with its full workspace."""
    kbuild.build()
    lib = K.load_library()
    x = W.prefill_inputs(W.custom_prefill([130, 64], num_heads=2, d=128, seed=57))
    g = x["g"].float()
    g[:130, 1] = -2.0  # sequence 0, head 1
    x["g"] = g.to(x["g"].dtype)
    d = to_dev(x)
    ref_o, ref_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 d["init_state"], check=True)
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        fin = torch.full_like(ref_f, float("nan"))
        assert _noalloc(lib, d, out, fin) == 0
        rc, words = _noalloc_words(lib)
        assert rc == 0 and words[0] == 0 and words[3] == 1, words
        assert torch.equal(out, ref_o) and torch.equal(fin, ref_f)


def test_noalloc_rejects_bad_shapes_without_launching():
    kbuild.build()
    lib = K.load_library()
    bad = K.kda_shape(1, 64, 1, 96, 128, 64, 0.0, K.KDA_BF16, 0)
    assert lib.kda_chunk_fwd_noalloc(ctypes.byref(bad), *([None] * 10)) == -2
    assert lib.kda_chunk_fwd_noalloc(None, *([None] * 10)) == -1
    # the status block and one flag word per sequence-head must fit the 256 KiB buffer
    big = K.kda_shape(65473, 65473, 1, 128, 128, 64, 0.0, K.KDA_BF16, 0)
    assert lib.kda_chunk_fwd_noalloc(ctypes.byref(big), *([None] * 10)) == -10
    fits = K.kda_shape(65472, 65472, 1, 128, 128, 64, 0.0, K.KDA_BF16, 0)
    assert lib.kda_chunk_fwd_noalloc(ctypes.byref(fits), *([None] * 10)) == -1  # then the pointers
