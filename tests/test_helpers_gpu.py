"""The few-sequence-head schedule of the tensor-core prefill.

With at most 76 (sequence, head) pairs and a workspace of
kda_chunk_fwd_workspace_bytes(), one (up to 76 pairs) or two (up to 50) solve-helper
CTAs per pair compute each chunk's [T - I; A^qk] ("Kimi Delta Attention (KDA)", the
chunkwise algorithm's WY / UT-transform step) and hand it to the pair's tile CTA through
a ring in the workspace (after the status block and, with a gate, one flag word per
pair rounded up to 256 bytes).  A 256-byte workspace selects the plain schedule,
where the tile solves every chunk itself.  Both run the same arithmetic on the
same operands, so their results must agree bit for bit; the helper schedule is
also checked against the oracle, and the ring's hand-over counters are read
back to show that the helpers ran."""
import numpy as np
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import (kda_chunk_fwd, kda_chunk_fwd_workspace_bytes,
                                            kda_workspace_status, workspace_status_words)
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, rel_l2_per_head, rel_l2_states, run_oracle_prefill, to_dev

pytestmark = pytest.mark.gpu

STATUS_BYTES = 256
FLAG_BYTES = 256  # one flag word per pair (at most 64 here), rounded up to 256 bytes
SLOTS, SLOT_BYTES = 4, 16384
MAX_PAIRS = 64


def _run(dv, g, workspace):
    return kda_chunk_fwd(dv["q"], dv["k"], dv["v"], g, dv["beta"], dv["cu_seqlens"],
                         dv["init_state"], workspace=workspace, algo="tensor", check=True)


def _full_workspace(x, H):
    T = x["q"].shape[0]
    n = len(x["cu_seqlens"]) - 1
    need = kda_chunk_fwd_workspace_bytes(n, T, H, 128, 128)
    # garbage in the workspace must not matter: the call clears what it reads
    return torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda"), need


def _expected_ring_words(lens, H):
    """Per pair and slot: (last chunk published + 1, consumptions) after the call."""
    words = []
    for L in lens:
        nch = (L + 63) // 64
        for _ in range(H):
            for slot in range(SLOTS):
                cs = [c for c in range(nch) if c % SLOTS == slot]
                words += [cs[-1] + 1 if cs else 0, len(cs)]  # one read per chunk
    return np.array(words, dtype=np.uint32)


def _gate_for(x, mode):
    if mode == "channel":
        return x["g"], x["g"]
    if mode == "scalar":
        g_tok = x["g"][..., 0].contiguous()
        return g_tok, g_tok.unsqueeze(-1).expand_as(x["g"]).contiguous()
    return None, torch.zeros_like(x["g"])


CASES = [
    # lengths, heads: single and partial chunks, ragged tails, an empty sequence,
    # a sequence spanning many ring cycles, and the largest pair count with helpers
    ([1, 63, 65, 300, 200], 2),
    ([0, 130, 0, 64], 3),
    ([64 * 13 + 7], 4),
    ([5 + 37 * i for i in range(19)], 2),
    # 60 pairs: one helper per pair (two fit up to 50 pairs on 152 SMs)
    ([40 + 23 * i for i in range(30)], 2),
]


@pytest.mark.parametrize("lens,H", CASES)
@pytest.mark.parametrize("mode", ["channel", "scalar", "none"])
def test_helper_schedule_matches_plain_schedule_and_oracle(lens, H, mode):
    spec = W.custom_prefill(lens, num_heads=H, d=128, gate="mixed", seed=61 + len(lens))
    x = W.prefill_inputs(spec)
    g_gpu, g_ref = _gate_for(x, mode)
    pairs = len(lens) * H
    assert pairs <= MAX_PAIRS
    dv = to_dev(x)
    gd = None if g_gpu is None else g_gpu.cuda()
    ws, need = _full_workspace(x, H)
    assert need == STATUS_BYTES + FLAG_BYTES + pairs * SLOTS * (SLOT_BYTES + 8)
    o_h, s_h = _run(dv, gd, ws)
    assert workspace_status_words(ws)[2] == 2  # the solve-helper schedule ran
    o_p, s_p = _run(dv, gd, torch.empty(STATUS_BYTES, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_p)
    assert torch.equal(s_h, s_p)
    ring = STATUS_BYTES + (FLAG_BYTES if mode != "none" else 0)  # no decay, no flags
    words = ws[ring + pairs * SLOTS * SLOT_BYTES:][:pairs * SLOTS * 8].cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(words, _expected_ring_words(lens, H))
    ro, rs = run_oracle_prefill(dict(x, g=g_ref))
    cu = x["cu_seqlens"].numpy()
    assert rel_l2_per_head(o_h.float().cpu().numpy(), ro, cu) <= TOL_BF16
    assert rel_l2_states(s_h.cpu().numpy(), rs) <= TOL_BF16


def test_helper_schedule_is_repeatable_on_one_workspace():
    """Back-to-back calls reuse the ring: each clears its counters first."""
    spec = W.custom_prefill([700, 129], num_heads=3, d=128, gate="mixed", seed=67)
    x = W.prefill_inputs(spec)
    dv = to_dev(x)
    ws, _ = _full_workspace(x, 3)
    first = _run(dv, dv["g"], ws)
    for _ in range(3):
        again = _run(dv, dv["g"], ws)
        assert torch.equal(first[0], again[0]) and torch.equal(first[1], again[1])


def test_helper_schedule_on_concurrent_streams():
    """Calls on two streams, each with its own workspace, may run at the same time
    (each cooperative grid is resident as a whole); every result and status is
    that of a lone call."""
    spec = W.custom_prefill([900, 300, 65], num_heads=2, d=128, gate="mixed", seed=69)
    x = W.prefill_inputs(spec)
    dv = to_dev(x)
    ref = _run(dv, dv["g"], _full_workspace(x, 2)[0])
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [_full_workspace(x, 2)[0] for _ in streams]
    outs = []
    torch.cuda.synchronize()
    for _ in range(4):
        for st, ws in zip(streams, wss):
            with torch.cuda.stream(st):
                outs.append(kda_chunk_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"],
                                          dv["cu_seqlens"], dv["init_state"], workspace=ws,
                                          algo="tensor", stream=st))
    torch.cuda.synchronize()
    for o, f in outs:
        assert torch.equal(o, ref[0]) and torch.equal(f, ref[1])
    for ws in wss:
        assert kda_workspace_status(ws) == 0


def test_more_pairs_than_helpers_use_the_plain_schedule():
    lens = [100] * 11
    assert kda_chunk_fwd_workspace_bytes(11, 1100, 7, 128, 128) == STATUS_BYTES + 512 + 256  # 77: order
    assert kda_chunk_fwd_workspace_bytes(38, 3800, 2, 128, 128) > STATUS_BYTES + 512  # 76
    spec = W.custom_prefill(lens, num_heads=7, d=128, gate="mixed", seed=68)
    x = W.prefill_inputs(spec)
    dv = to_dev(x)
    ws = torch.empty(STATUS_BYTES + 512, dtype=torch.uint8, device="cuda")
    o, s = _run(dv, dv["g"], ws)
    assert workspace_status_words(ws)[2] == 1  # plain
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(o.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(s.cpu().numpy(), rs) <= TOL_BF16
