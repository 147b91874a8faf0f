"""The segment-parallel scan of a few long sequences with few heads.

The state recurrence of "Kimi Delta Attention (KDA)" is affine in the start state: over
any stretch of tokens S_end = M S_start + B, with M the product of the per-token
transitions (I - beta k k^T) Diag(alpha) and B the end state from a zero start.  With one
sequence, at most 50 heads and at least 3 x 32 chunks, kda_chunk_fwd_workspace_bytes()
includes room for cutting the sequence into P segments: a first launch runs segment 0
from the true start and every middle segment from zero (B) and from the identity with
V = 0 (M), a small kernel chains S_{p+1} = M_p S_p + B_p, and a second launch runs
segments 1 .. P - 1 from those states; a pass with at most 76 (run, head) pairs runs
with solve helpers (every case here has one such pass; the P = 20 and P = 39 cases run
their first pass without).  The rounding differs from the one-chain
schedules, so the results are compared with the oracle at the bf16 tolerance (and with
the one-chain schedule at twice it), and word 2 of the status block (3) shows that the
segments ran.
"""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_fwd_gb300 import (kda_chunk_fwd, kda_chunk_fwd_workspace_bytes,
                                            workspace_status_words)
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, rel_l2_per_head, rel_l2_states, run_oracle_prefill, to_dev

pytestmark = pytest.mark.gpu

STATUS_BYTES, SCHED_SEGMENTS = 256, 3


def _segments(T, H, sms, N=1):
    """Segments per sequence: from the average sequence's chunks, while the first pass's
    N H (2P - 3) runs fit one wave."""
    if N * H > sms:
        return 0
    nch = (T // N + 63) // 64
    P = min((sms // (N * H) + 3) // 2, nch // 32)
    return P if P >= 3 else 0


def _seg_start(T, P, q):
    """First token of segment q (q = P: the end): chunks q n / P .. of the n chunks."""
    n = (T + 63) // 64
    return min(T, q * n // P * 64)


def _seg_bytes(P, H, N=1):
    """Run tables and skip marks, 4P - 5 states per sequence-head, the ring of the larger
    pass that takes solve helpers (at most 76 pairs)."""
    pairs = [r * N * H for r in (2 * P - 3, P - 1) if r * N * H <= 76]
    return ((3 * P * 16 * N + 4 * N * H + 255) // 256 * 256 + (4 * P - 5) * N * H * 128 * 128 * 4
            + max(pairs, default=0) * 4 * (16384 + 8))


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _gates(x, mode):
    """(g for the GPU call, per-channel g for the oracle).  "slow" and "scalar": the
    recipe's gate over 100, so that a segment's start state still shows at its end (with
    the recipe's decay it has fallen below the fp32 range after about 1,500 tokens, and
    the segments would agree with one chain without their combine being right)."""
    if mode == "slow":
        g = (x["g"].float() / 100).to(x["g"].dtype).contiguous()
        return g, g
    if mode == "channel":
        return x["g"], x["g"]
    if mode == "scalar":  # one log alpha per token and head, slow as well
        g_tok = (x["g"][..., 0].float() / 100).to(x["g"].dtype).contiguous()
        return g_tok, g_tok.unsqueeze(-1).expand_as(x["g"]).contiguous()
    return None, torch.zeros_like(x["g"])


def _call(d, g, ws, **kw):
    return kda_chunk_fwd(d["q"], d["k"], d["v"], g, d["beta"], d["cu_seqlens"], d["init_state"],
                         workspace=ws, algo="tensor", **kw)


CASES = [
    # T, H, gate, init: P = 4 with a ragged last segment; P = 3 ending on a chunk
    # boundary; P = 9 over four heads; P = 20 (the most a 152-SM part gives 4 heads);
    # P = 39 over 2 heads; the recipe's decay
    (10007, 2, "slow", "normal"),
    (6144, 1, "slow", "normal"),
    (20000, 4, "scalar", "zeros"),
    (41000, 4, "none", "normal"),
    (80000, 2, "slow", "zeros"),
    (10007, 2, "channel", "normal"),
]


@pytest.mark.parametrize("T,H,mode,init", CASES)
def test_segments_match_the_oracle(T, H, mode, init):
    P = _segments(T, H, _sms())
    assert P >= 3
    gate = "std" if mode in ("slow", "scalar") else "mixed"
    x = W.prefill_inputs(W.custom_prefill([T], num_heads=H, d=128, gate=gate, init=init, seed=101 + H))
    g_gpu, g_ref = _gates(x, mode)
    d = to_dev(x)
    need = kda_chunk_fwd_workspace_bytes(1, T, H, 128, 128)
    assert need == STATUS_BYTES + 256 + _seg_bytes(P, H)  # status, flags, segments
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    out, fin = _call(d, None if g_gpu is None else g_gpu.cuda(), ws, check=True)
    words = workspace_status_words(ws)
    assert words[0] == 0 and words[2] == SCHED_SEGMENTS and words[3] == 0, words
    xo = dict(x)
    xo["g"] = g_ref
    ro, rs = run_oracle_prefill(xo)
    o, s = out.float().cpu().numpy(), fin.cpu().numpy()
    assert np.isfinite(o).all() and np.isfinite(s).all()
    assert rel_l2_per_head(o, ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(s, rs) <= TOL_BF16
    # every segment's outputs, not only the norm over the sequence: the worst segment
    for p in range(P):
        lo, hi = _seg_start(T, P, p), _seg_start(T, P, p + 1)
        cu = np.array([0, hi - lo])
        assert rel_l2_per_head(o[lo:hi], ro[lo:hi], cu) <= TOL_BF16, p
    if mode in ("slow", "scalar", "none"):
        # the last segment's start state still matters: from zero its outputs are far off
        lo = _seg_start(T, P, P - 1)
        xs = {kk: xo[kk][lo:] for kk in ("q", "k", "v", "g", "beta")}
        xs.update(cu_seqlens=torch.tensor([0, T - lo], dtype=torch.int32), init_state=None)
        rz, _ = run_oracle_prefill(xs)
        assert rel_l2_per_head(rz, ro[lo:], np.array([0, T - lo])) > 10 * TOL_BF16
    # the one-chain schedule (a workspace without room for the segments) agrees
    small = torch.zeros(need - _seg_bytes(P, H), dtype=torch.uint8, device="cuda")
    o1, s1 = _call(d, None if g_gpu is None else g_gpu.cuda(), small, check=True)
    assert workspace_status_words(small)[2] in (1, 2)
    assert rel_l2_per_head(o, o1.float().cpu().numpy(), x["cu_seqlens"].numpy()) <= 2 * TOL_BF16
    assert rel_l2_states(s, s1.cpu().numpy()) <= 2 * TOL_BF16


def test_segments_with_input_steps():
    """The instantiation with the input steps (silu, L2 norm, sigmoid, softplus gate)
    runs the segments too."""
    T, H = 9000, 2
    x = W.prefill_inputs(W.custom_prefill([T], num_heads=H, d=128, gate="mixed", seed=111),
                         raw=True, raw_gate=True)
    d = to_dev(x)
    ws = torch.zeros(kda_chunk_fwd_workspace_bytes(1, T, H, 128, 128), dtype=torch.uint8, device="cuda")
    out, fin = _call(d, d["g"], ws, check=True, qk_silu=True, qk_l2norm=True, beta_sigmoid=True,
                     g_softplus=True, gate_scale=1.0)
    assert workspace_status_words(ws)[2] == SCHED_SEGMENTS
    q, k, b = oracle.preprocess(x["q"], x["k"], x["beta"], qk_silu=True, qk_l2norm=True,
                                beta_sigmoid=True)
    g_ref = oracle.gate_from_logits(x["g"], gate_scale=1.0)
    ro, rs = oracle.kda_fwd(q, k, x["v"], g_ref, b, x["cu_seqlens"], x["init_state"])
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16


@pytest.mark.parametrize("where", ["first", "middle", "last"])
@pytest.mark.parametrize("in_place", [False, True])
def test_segments_gate_beyond_range(where, in_place):
    """A head whose decay leaves the tensor-core range in segment 0, a middle segment or
    the last one is marked, skipped by the second pass and recomputed token by token
    from the untouched initial state (also when final_state aliases it); the other head
    keeps the segment results."""
    T, H = 10007, 2
    P = _segments(T, H, _sms())
    lo = {"first": 100, "middle": _seg_start(T, P, 1) + 300, "last": _seg_start(T, P, P - 1) + 50}[where]
    x = W.prefill_inputs(W.custom_prefill([T], num_heads=H, d=128, seed=112))
    g = x["g"].float()
    g[lo:lo + 200, 1] = -2.0
    x["g"] = g.to(x["g"].dtype).contiguous()
    d = to_dev(x)
    ws = torch.zeros(kda_chunk_fwd_workspace_bytes(1, T, H, 128, 128), dtype=torch.uint8, device="cuda")
    st = d["init_state"].clone()
    out, fin = _call(d | {"init_state": st}, d["g"], ws, check=True,
                     **({"final_state": st} if in_place else {}))
    words = workspace_status_words(ws)
    assert words[0] == 0 and words[2] == SCHED_SEGMENTS and words[3] == 1, words
    if in_place:
        assert fin.data_ptr() == st.data_ptr()
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16


@pytest.mark.parametrize("cu", [[0, 10007 + 64], [5, 3], [-64, 10007]])
def test_segments_skip_bad_offsets(cu):
    """Offsets the device finds out of order or out of range: every segment run is
    skipped, nothing is written, and KDA_ERR_SEQLENS is recorded.  The tensors hold 128
    rows beyond the declared 10,007 (the largest offset here is 10,071), so even a missed
    check stays inside them."""
    T, H = 10007, 2
    x = W.prefill_inputs(W.custom_prefill([T + 128], num_heads=H, d=128, seed=113))
    d = to_dev(x)
    rows = {kk: (vv[:T] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in d.items()}
    ws = torch.zeros(kda_chunk_fwd_workspace_bytes(1, T, H, 128, 128), dtype=torch.uint8, device="cuda")
    out = torch.full((T + 128, H, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    fin = torch.full_like(d["init_state"], 7.0)
    kda_chunk_fwd(rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"],
                  torch.tensor(cu, dtype=torch.int32, device="cuda"), d["init_state"], out=out[:T],
                  final_state=fin, workspace=ws, algo="tensor")
    words = workspace_status_words(ws)
    assert words[0] == 11 and words[2] == SCHED_SEGMENTS, words  # KDA_ERR_SEQLENS
    assert torch.equal(out, torch.full_like(out, 5.0))
    assert torch.equal(fin, torch.full_like(fin, 7.0))


def test_many_heads_or_short_sequences_keep_one_chain():
    """51 sequence-heads (fewer than three runs each fit in one wave) and sequences of 95
    chunks on average: no room for segments is asked for."""
    sms = _sms()
    assert _segments(65536, 51, sms) == 0 and _segments(64 * 95, 2, sms) == 0
    assert _segments(2 * 65536, 26, sms, N=2) == 0 and _segments(2 * 64 * 95, 2, sms, N=2) == 0
    for N, T, H in ((1, 64 * 95, 2), (2, 2 * 64 * 95, 2), (2, 2 * 65536, 26)):
        assert kda_chunk_fwd_workspace_bytes(N, T, H, 128, 128) < _seg_bytes(3, H, N)


def _slow(x):
    x["g"] = (x["g"].float() / 100).to(x["g"].dtype).contiguous()
    return x


@pytest.mark.parametrize("lens,H", [([7000, 12000], 2), ([9000, 0, 9500], 1), ([6500, 6200, 7000, 6400], 2)])
def test_several_sequences_match_the_oracle(lens, H):
    """Several long sequences (one empty among them): each cut into the same number of
    segments from its own length, the runs of all of them in the same two passes."""
    N, T = len(lens), sum(lens)
    P = _segments(T, H, _sms(), N)
    assert P >= 3
    x = _slow(W.prefill_inputs(W.custom_prefill(lens, num_heads=H, d=128, gate="std", seed=121)))
    d = to_dev(x)
    need = kda_chunk_fwd_workspace_bytes(N, T, H, 128, 128)
    assert need == STATUS_BYTES + (4 * N * H + 255) // 256 * 256 + _seg_bytes(P, H, N)
    ws = torch.full((need,), 0x5A, dtype=torch.uint8, device="cuda")
    out, fin = _call(d, d["g"], ws, check=True)
    words = workspace_status_words(ws)
    assert words[0] == 0 and words[2] == SCHED_SEGMENTS and words[3] == 0, words
    ro, rs = run_oracle_prefill(x)
    o, s = out.float().cpu().numpy(), fin.cpu().numpy()
    cu = x["cu_seqlens"].numpy()
    assert rel_l2_per_head(o, ro, cu) <= TOL_BF16
    nonempty = [n for n, L in enumerate(lens) if L > 0]
    assert rel_l2_states(s[nonempty], rs[nonempty]) <= TOL_BF16
    for n, L in enumerate(lens):
        if L == 0:  # an empty sequence passes its initial state through
            assert torch.equal(fin[n], d["init_state"][n])
            continue
        for p in range(P):  # every segment of every sequence
            lo, hi = cu[n] + _seg_start(L, P, p), cu[n] + _seg_start(L, P, p + 1)
            assert rel_l2_per_head(o[lo:hi], ro[lo:hi], np.array([0, hi - lo])) <= TOL_BF16, (n, p)


def test_several_sequences_gate_beyond_range_and_bad_offsets():
    """Two of three sequences' offsets are valid: the third (out of order) is skipped and
    reported, and one head of the second, whose decay leaves the tensor-core range, is
    recomputed token by token; everything else keeps the segment results."""
    lens, H = [8000, 9000, 8000], 2
    x = _slow(W.prefill_inputs(W.custom_prefill(lens + [128], num_heads=H, d=128, gate="std", seed=122)))
    g = x["g"].float()
    g[8000 + 3000:8000 + 3200, 0] = -2.0
    x["g"] = g.to(x["g"].dtype).contiguous()
    T = sum(lens)
    d = to_dev(x)
    rows = {kk: (vv[:T] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in d.items()}
    cu = torch.tensor([0, 8000, 17000, 16000], dtype=torch.int32, device="cuda")  # sequence 2 = [17000, 16000)
    init = d["init_state"][:3].contiguous()
    ws = torch.zeros(kda_chunk_fwd_workspace_bytes(3, T, H, 128, 128), dtype=torch.uint8, device="cuda")
    out = torch.full((T + 128, H, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    fin = torch.full_like(init, 7.0)
    kda_chunk_fwd(rows["q"], rows["k"], rows["v"], rows["g"], rows["beta"], cu, init, out=out[:T],
                  final_state=fin, workspace=ws, algo="tensor")
    words = workspace_status_words(ws)
    assert words[0] == 11 and words[2] == SCHED_SEGMENTS and words[3] == 1, words  # KDA_ERR_SEQLENS
    assert torch.equal(fin[2], torch.full_like(fin[2], 7.0))  # the skipped sequence
    assert torch.equal(out[17000:], torch.full_like(out[17000:], 5.0))
    xs = {kk: x[kk][:17000] for kk in ("q", "k", "v", "g", "beta")}
    xs.update(cu_seqlens=torch.tensor([0, 8000, 17000], dtype=torch.int32), init_state=x["init_state"][:2])
    ro, rs = run_oracle_prefill(xs)
    assert rel_l2_per_head(out[:17000].float().cpu().numpy(), ro, xs["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin[:2].cpu().numpy(), rs) <= TOL_BF16


def _random_case(seed):
    import random
    r = random.Random(seed)
    n = r.randint(1, 3)
    short = n > 1 and r.random() < 0.5
    lens = [r.randint(12300 if short else 6200, 16000) for _ in range(n)]  # 96 chunks on average
    if short:
        lens[r.randrange(n)] = r.choice([0, 1, 63, 64, 65, 700])  # a short one among them
    return dict(lens=lens, H=r.randint(1, 4), gate=r.choice(["channel", "scalar", "none"]),
                decay=r.choice([1.0, 0.05, 0.01]), init=r.choice(["normal", "zeros"]),
                beta_scale=r.choice([1.0, 0.3]), state_scale=r.choice([1.0, 50.0]))


@pytest.mark.parametrize("seed", range(2000, 2008))
def test_random_long_sequences(seed):
    """Seeded random calls that take the segments: one to three sequences (a short or empty
    one among them at times), one to four heads, every gate form, decays from the recipe's
    down to a hundredth of it, with and without an initial state (of standard deviation
    0.02 or 1), write strengths at the recipe's or 0.3 of it."""
    c = _random_case(seed)
    lens, H = c["lens"], c["H"]
    N, T = len(lens), sum(lens)
    P = _segments(T, H, _sms(), N)
    if P < 3:
        pytest.skip(f"average length too short for segments: {lens}")
    x = W.prefill_inputs(W.custom_prefill(lens, num_heads=H, d=128, gate="std", init=c["init"], seed=seed))
    x["g"] = (x["g"].float() * c["decay"]).to(x["g"].dtype)
    x["beta"] = (x["beta"].float() * c["beta_scale"]).to(x["beta"].dtype)
    if x["init_state"] is not None:
        x["init_state"] = x["init_state"] * c["state_scale"]
    if c["gate"] == "channel":
        g_gpu = g_ref = x["g"]
    elif c["gate"] == "scalar":
        g_gpu = x["g"][..., 0].contiguous()
        g_ref = g_gpu.unsqueeze(-1).expand_as(x["g"]).contiguous()
    else:
        g_gpu, g_ref = None, torch.zeros_like(x["g"])
    d = to_dev(x)
    ws = torch.zeros(kda_chunk_fwd_workspace_bytes(N, T, H, 128, 128), dtype=torch.uint8, device="cuda")
    out, fin = _call(d, None if g_gpu is None else g_gpu.cuda(), ws, check=True)
    assert workspace_status_words(ws)[2] == SCHED_SEGMENTS
    xo = dict(x)
    xo["g"] = g_ref
    ro, rs = run_oracle_prefill(xo)
    o, s = out.float().cpu().numpy(), fin.cpu().numpy()
    cu = x["cu_seqlens"].numpy()
    assert np.isfinite(o).all() and np.isfinite(s).all()
    assert rel_l2_per_head(o, ro, cu) <= TOL_BF16, c
    nonempty = [n for n, L in enumerate(lens) if L > 0]
    assert rel_l2_states(s[nonempty], rs[nonempty]) <= TOL_BF16, c
