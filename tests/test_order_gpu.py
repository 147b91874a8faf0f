"""Launch order of the tensor-core prefill's plain schedule.

When a call takes more than one wave of CTAs (more sequence-heads than SMs) and the
workspace has room (kda_chunk_fwd_workspace_bytes() includes it for 2 to 2048
sequences), a small kernel sorts the sequences longest first and the CTAs take their
sequence-head from that order, so that the longest chains start first.  Each CTA still
computes one (sequence, head) on its own, so the results must be bit-identical to the
given order, and they must match the oracle.
"""
import numpy as np
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import (kda_chunk_fwd, kda_chunk_fwd_workspace_bytes,
                                            kda_workspace_status, workspace_status_words)
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, rel_l2_per_head, rel_l2_states, run_oracle_prefill, to_dev

pytestmark = pytest.mark.gpu


def _run(dv, ws):
    return kda_chunk_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"],
                         dv["init_state"], workspace=ws, algo="tensor")


@pytest.mark.parametrize("gate", ["std", "mixed"])
def test_longest_first_order_is_bit_identical_and_matches_the_oracle(gate):
    # 14 sequences x 16 heads = 224 sequence-heads, more than the 152 SMs hold at once;
    # lengths out of order, with an empty and a one-token sequence and ragged tails
    lens = [70, 400, 0, 129, 1, 333, 64, 257, 190, 65, 511, 3, 128, 300]
    H = 16
    x = W.prefill_inputs(W.custom_prefill(lens, num_heads=H, d=128, gate=gate, seed=91))
    dv = to_dev(x)
    T, N = x["q"].shape[0], len(lens)
    full = kda_chunk_fwd_workspace_bytes(N, T, H, 128, 128)
    flags = (4 * N * H + 255) // 256 * 256
    assert full == 256 + flags + 256  # the status block, the flags, the launch order
    ws_ordered = torch.full((full,), 0xAB, dtype=torch.uint8, device="cuda")
    ws_given = torch.full((256 + flags,), 0xAB, dtype=torch.uint8, device="cuda")
    o1, s1 = _run(dv, ws_ordered)
    o2, s2 = _run(dv, ws_given)
    torch.cuda.synchronize()
    assert kda_workspace_status(ws_ordered) == 0 and kda_workspace_status(ws_given) == 0
    assert workspace_status_words(ws_ordered)[2] == 1  # the plain schedule ran
    # the order the kernel used, read back: every sequence once, longest first
    order = ws_ordered[256 + flags:256 + flags + 4 * N].cpu().numpy().view(np.int32)
    assert sorted(order.tolist()) == list(range(N))
    assert [lens[i] for i in order] == sorted(lens, reverse=True)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(o1.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    nonempty = [n for n, L in enumerate(lens) if L > 0]
    assert rel_l2_states(s1.cpu().numpy()[nonempty], rs[nonempty]) <= TOL_BF16
    # an empty sequence passes its initial state through
    assert torch.equal(s1[2], dv["init_state"][2])


def test_one_wave_or_one_sequence_keeps_the_given_order():
    # 150 sequence-heads fit in one wave, and a single sequence has nothing to order:
    # the launch order is not computed, and the words after the flags stay as they were
    for lens, H in (([90, 40, 200], 50), ([300], 200)):
        x = W.prefill_inputs(W.custom_prefill(lens, num_heads=H, d=128, seed=92))
        dv = to_dev(x)
        T, N = x["q"].shape[0], len(lens)
        full = kda_chunk_fwd_workspace_bytes(N, T, H, 128, 128)
        flags = (4 * N * H + 255) // 256 * 256
        ws = torch.full((full,), 0xAB, dtype=torch.uint8, device="cuda")
        o, s = _run(dv, ws)
        torch.cuda.synchronize()
        assert kda_workspace_status(ws) == 0
        tail = ws[256 + flags:].cpu().numpy()
        assert np.all(tail == 0xAB)
        ro, rs = run_oracle_prefill(x)
        assert rel_l2_per_head(o.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
        assert rel_l2_states(s.cpu().numpy(), rs) <= TOL_BF16
