"""kda_recurrent_fwd: the recurrence token by token over short packed sequences
("Kimi Delta Attention (KDA)", the fused recurrent schedule), with the state
after a chosen number of tokens per sequence for the rollback of speculative
decoding ("K3 架构图解", the section on speculative decoding).

Outputs and states are checked against the oracle run on the same sequences
(all tokens for the outputs, the first accepted[n] tokens for the state), and
the verify-then-commit pattern against a single run over the accepted tokens."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_fwd_gb300 import kda_chunk_fwd, kda_decode_step, kda_recurrent_fwd
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, TOL_F32, rel_l2_per_head, rel_l2_states, to_dev

pytestmark = pytest.mark.gpu

LENS = [0, 1, 3, 7, 16, 33]


def _gates(x, mode):
    """(g for the GPU call, per-channel g for the oracle)."""
    if mode == "channel":
        return x["g"], x["g"]
    if mode == "scalar":
        g_tok = x["g"][..., 0].contiguous()
        return g_tok, g_tok.unsqueeze(-1).expand_as(x["g"]).contiguous()
    return None, torch.zeros_like(x["g"])


def _truncate(x, g_ref, acc):
    """The first acc[n] tokens of every sequence, packed (oracle inputs)."""
    cu = x["cu_seqlens"].numpy()
    rows = np.concatenate([np.arange(cu[n], cu[n] + a) for n, a in enumerate(acc)]).astype(np.int64)
    idx = torch.from_numpy(rows)
    cu2 = torch.from_numpy(np.concatenate([[0], np.cumsum(acc)]).astype(np.int32))
    return {kk: x[kk][idx] for kk in ("q", "k", "v", "beta")} | {"g": g_ref[idx], "cu_seqlens": cu2,
                                                                  "init_state": x["init_state"]}


@pytest.mark.parametrize("mode", ["channel", "scalar", "none"])
@pytest.mark.parametrize("io,d,tol", [("bf16", 128, TOL_BF16), ("f32", 128, TOL_F32),
                                      ("bf16", 64, TOL_BF16), ("f32", 64, TOL_F32)])
def test_recurrent_matches_oracle_with_accepted_counts(mode, io, d, tol):
    spec = W.custom_prefill(LENS, num_heads=3, d=d, io=io, gate="mixed", seed=81)
    x = W.prefill_inputs(spec)
    g_gpu, g_ref = _gates(x, mode)
    dv = to_dev(x)
    acc = [0, 1, 2, 7, 20, 5]  # per sequence; above the length means all of it
    acc_t = torch.tensor(acc, dtype=torch.int32, device="cuda")
    out, fin = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], None if g_gpu is None else g_gpu.cuda(),
                                 dv["beta"], dv["cu_seqlens"], dv["init_state"], accepted=acc_t)
    torch.cuda.synchronize()
    ro, _ = oracle.kda_fwd(x["q"], x["k"], x["v"], g_ref, x["beta"], x["cu_seqlens"], x["init_state"])
    cu = x["cu_seqlens"].numpy()
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, cu) <= tol
    kept = [min(a, L) for a, L in zip(acc, LENS)]
    t = _truncate(x, g_ref, kept)
    _, rs = oracle.kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], t["init_state"])
    assert rel_l2_states(fin.cpu().numpy(), rs) <= tol


def test_verify_then_commit_equals_one_run_over_the_accepted_tokens():
    spec = W.custom_prefill([4] * 6, num_heads=2, d=128, gate="mixed", seed=82)
    x = W.prefill_inputs(spec)
    dv = to_dev(x)
    state = dv["init_state"].clone()
    before = state.clone()
    # verify: every draft's output, the state untouched
    out, none = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"],
                                  state, output_final_state=False)
    assert none is None
    torch.cuda.synchronize()
    assert torch.equal(state, before)
    # commit in place: the state advances over the accepted drafts only
    acc = torch.tensor([0, 1, 2, 3, 4, 2], dtype=torch.int32, device="cuda")
    o2, fin = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"],
                                state, accepted=acc, output=False, final_state=state)
    assert o2 is None and fin is state
    torch.cuda.synchronize()
    # the same in one call gives the same outputs and state, bit for bit
    out1, fin1 = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"],
                                   before, accepted=acc)
    torch.cuda.synchronize()
    assert torch.equal(out1, out) and torch.equal(fin1, state)
    # and the oracle over the accepted tokens
    t = _truncate(x, x["g"], acc.cpu().tolist())
    _, rs = oracle.kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], t["init_state"])
    assert rel_l2_states(state.cpu().numpy(), rs) <= TOL_BF16


def test_recurrent_agrees_with_decode_step_and_chunk_prefill():
    # one token per sequence: the decode step
    y = W.decode_inputs(W.DecodeSpec(5, 3, 128, 128, 1, "bf16", "std", 83))
    st = y["state"].clone().cuda()
    o_dec = kda_decode_step(y["q"][0].cuda(), y["k"][0].cuda(), y["v"][0].cuda(), y["g"][0].cuda(),
                            y["beta"][0].cuda(), st)
    cu = torch.arange(6, dtype=torch.int32, device="cuda")
    o_rec, s_rec = kda_recurrent_fwd(y["q"][0].cuda(), y["k"][0].cuda(), y["v"][0].cuda(),
                                     y["g"][0].cuda(), y["beta"][0].cuda(), cu, y["state"].cuda())
    torch.cuda.synchronize()
    assert rel_l2_states(s_rec.cpu().numpy(), st.cpu().numpy()) <= 1e-6
    assert rel_l2_per_head(o_rec.float().cpu().numpy(), o_dec.float().cpu().numpy(),
                           np.arange(6)) <= 1e-2
    # longer sequences: the chunkwise prefill
    spec = W.custom_prefill([70, 5, 129], num_heads=2, d=128, gate="mixed", seed=84)
    x = W.prefill_inputs(spec)
    dv = to_dev(x)
    o1, s1 = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"],
                               dv["init_state"])
    o2, s2 = kda_chunk_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"],
                           dv["init_state"], check=True)
    torch.cuda.synchronize()
    cuh = x["cu_seqlens"].numpy()
    assert rel_l2_per_head(o1.float().cpu().numpy(), o2.float().cpu().numpy(), cuh) <= TOL_BF16
    assert rel_l2_states(s1.cpu().numpy(), s2.cpu().numpy()) <= TOL_BF16


def test_recurrent_zero_init_and_empty_inputs():
    spec = W.custom_prefill([2, 0, 5], num_heads=1, d=64, io="f32", init="zeros", seed=85)
    x = W.prefill_inputs(spec)
    dv = to_dev(x)
    out, fin = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], dv["g"], dv["beta"], dv["cu_seqlens"])
    torch.cuda.synchronize()
    ro, rs = oracle.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"], None)
    assert rel_l2_per_head(out.cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_F32
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_F32
    # no sequences at all
    e = torch.zeros((0, 1, 64), device="cuda")
    o, f = kda_recurrent_fwd(e, e, e, e, torch.zeros((0, 1), device="cuda"),
                             torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert o.shape == (0, 1, 64) and f.shape == (0, 1, 64, 64)


@pytest.mark.parametrize("mode", ["channel", "scalar", "none"])
@pytest.mark.parametrize("io,d,tol", [("bf16", 128, TOL_BF16), ("f32", 64, TOL_F32)])
def test_persistent_launch_matches_oracle(mode, io, d, tol):
    """More sequence-heads than two CTAs per SM, with two or more tokens per sequence on
    average: the launch takes persistent CTAs that stage each next sequence-head's state
    in shared memory while they run the current one.  Ragged lengths (0 to 9 tokens),
    accepted counts, the state updated in place, against the oracle."""
    n = 2 * torch.cuda.get_device_properties(0).multi_processor_count + 37  # > 2 CTAs per SM
    gen = torch.Generator().manual_seed(86)
    lens = [int(x) for x in torch.randint(0, 10, (n,), generator=gen)]
    lens[0] = 9
    assert sum(lens) >= 2 * n
    spec = W.custom_prefill(lens, num_heads=1, d=d, io=io, gate="mixed", seed=86)
    x = W.prefill_inputs(spec)
    g_gpu, g_ref = _gates(x, mode)
    dv = to_dev(x)
    acc = [int(a) for a in torch.randint(0, 11, (n,), generator=gen)]
    acc_t = torch.tensor(acc, dtype=torch.int32, device="cuda")
    st = dv["init_state"].clone()
    gd = None if g_gpu is None else g_gpu.cuda()
    out, fin = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], gd, dv["beta"], dv["cu_seqlens"], st,
                                 accepted=acc_t, final_state=st)
    # the commit alone (no outputs: each sequence-head runs only its accepted tokens)
    st2 = dv["init_state"].clone()
    _, fin2 = kda_recurrent_fwd(dv["q"], dv["k"], dv["v"], gd, dv["beta"], dv["cu_seqlens"], st2,
                                accepted=acc_t, output=False, final_state=st2)
    torch.cuda.synchronize()
    assert torch.equal(fin2, fin)
    ro, _ = oracle.kda_fwd(x["q"], x["k"], x["v"], g_ref, x["beta"], x["cu_seqlens"], x["init_state"])
    cu = x["cu_seqlens"].numpy()
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, cu) <= tol
    kept = [min(a, L) for a, L in zip(acc, lens)]
    t = _truncate(x, g_ref, kept)
    _, rs = oracle.kda_fwd(t["q"], t["k"], t["v"], t["g"], t["beta"], t["cu_seqlens"], t["init_state"])
    assert rel_l2_states(fin.cpu().numpy(), rs) <= tol
