"""Bitwise repeatability of the tensor-core prefill and of the persistent recurrent pass
under repeated calls.

The schedules (plain, the solve helpers with their ring in the workspace, and the
segments of one long sequence) are deterministic: the same inputs must give the same bits on every call.  A race in
the hand-over between the K-side groups, the state side and the producers would
show up as an occasional call that differs, most likely with many short
sequences (38 sequence-heads with two helpers each, 60 with one) and a gate without
per-channel decay (the shortest K-side chain).  A change withdrawn during
development failed this check in about one call in twenty."""
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import (kda_chunk_fwd, kda_chunk_fwd_workspace_bytes,
                                            kda_recurrent_fwd, workspace_status_words)
from kimi_delta_attention_fwd_gb300 import workloads as W

pytestmark = pytest.mark.gpu

LENS = [5 + 37 * i for i in range(19)]       # 38 sequence-heads: two helpers each
LENS60 = [40 + 23 * i for i in range(30)]    # 60 sequence-heads: one helper each
H = 2
REPS = 30


@pytest.mark.parametrize("mode", ["none", "scalar", "channel"])
@pytest.mark.parametrize("schedule", ["plain", "helper", "helper1"])
def test_repeated_calls_are_bitwise_identical(mode, schedule):
    lens = LENS60 if schedule == "helper1" else LENS
    x = W.prefill_inputs(W.custom_prefill(lens, num_heads=H, d=128, gate="mixed", seed=90),
                         device="cuda")
    g = None if mode == "none" else (x["g"][..., 0].contiguous() if mode == "scalar" else x["g"])
    need = kda_chunk_fwd_workspace_bytes(len(lens), x["q"].shape[0], H, 128, 128)
    ws = torch.zeros(need if schedule != "plain" else 256, dtype=torch.uint8, device="cuda")
    args = (x["q"], x["k"], x["v"], g, x["beta"], x["cu_seqlens"], x["init_state"])
    o0, f0 = kda_chunk_fwd(*args, workspace=ws, algo="tensor", check=True)
    o0, f0 = o0.clone(), f0.clone()
    differing = 0
    for _ in range(REPS):
        o, f = kda_chunk_fwd(*args, workspace=ws, algo="tensor")
        differing += not (torch.equal(o, o0) and torch.equal(f, f0))
    torch.cuda.synchronize()
    assert differing == 0, f"{differing} of {REPS} calls differ from the first"


@pytest.mark.parametrize("T,Hs,reps", [(10007, 2, REPS), (41000, 4, 10)])
@pytest.mark.parametrize("mode", ["none", "channel"])
def test_segment_schedule_is_bitwise_repeatable(T, Hs, reps, mode):
    """One long sequence cut into segments (P = 4: both passes with two solve helpers per
    pair; P = 20: a plain first pass, one helper per pair in the second) and chained
    through the combine: the same bits on every call."""
    x = W.prefill_inputs(W.custom_prefill([T], num_heads=Hs, d=128, gate="mixed", seed=93),
                         device="cuda")
    g = None if mode == "none" else x["g"]
    ws = torch.zeros(kda_chunk_fwd_workspace_bytes(1, T, Hs, 128, 128), dtype=torch.uint8, device="cuda")
    args = (x["q"], x["k"], x["v"], g, x["beta"], x["cu_seqlens"], x["init_state"])
    o0, f0 = kda_chunk_fwd(*args, workspace=ws, algo="tensor", check=True)
    assert workspace_status_words(ws)[2] == 3  # the segments ran
    o0, f0 = o0.clone(), f0.clone()
    differing = 0
    for _ in range(reps):
        o, f = kda_chunk_fwd(*args, workspace=ws, algo="tensor")
        differing += not (torch.equal(o, o0) and torch.equal(f, f0))
    torch.cuda.synchronize()
    assert differing == 0, f"{differing} of {reps} calls differ from the first"


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
def test_persistent_recurrent_pass_is_bitwise_repeatable(gate):
    """The multi-token recurrent pass on 256 x 32 sequence-heads (persistent CTAs staging
    each next sequence-head's state and first token block through cp.async): repeated
    calls give the same bits."""
    drafts, N, H = 4, 256, 32
    y = W.decode_inputs(W.DecodeSpec(N, H, 128, 128, drafts, "bf16", "std", 3), device="cuda")
    pack = lambda t: t.transpose(0, 1).reshape(N * drafts, *t.shape[2:]).contiguous()
    q, k, v, g, beta = (pack(y[n]) for n in ("q", "k", "v", "g", "beta"))
    g = g if gate == "channel" else (g[..., 0].contiguous() if gate == "scalar" else None)
    cu = torch.arange(N + 1, dtype=torch.int32, device="cuda") * drafts
    acc = torch.randint(0, drafts + 1, (N,), dtype=torch.int32, device="cuda",
                        generator=torch.Generator(device="cuda").manual_seed(5))

    def run():
        st = y["state"].clone()
        o, f = kda_recurrent_fwd(q, k, v, g, beta, cu, st, accepted=acc, final_state=st)
        return o.clone(), f.clone()

    o0, f0 = run()
    differing = 0
    for _ in range(REPS):
        o, f = run()
        differing += not (torch.equal(o, o0) and torch.equal(f, f0))
    torch.cuda.synchronize()
    assert differing == 0, f"{differing} of {REPS} calls differ from the first"
