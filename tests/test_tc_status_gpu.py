"""Tensor-core prefill path: selection, and the device status it reports.

The bounded-wait error path is exercised without faulting or hanging the GPU:
the KDA_TEST_FORCE_WAIT_TIMEOUT hook makes the kernel wait once on an mbarrier
that nothing arrives on; the wait gives up after ~1 ms, the kernel records
KDA_ERR_DEVICE_TIMEOUT and runs to completion, and the next call works.
"""
import os

import pytest
import torch

from kimi_delta_attention_fwd_gb300 import (KdaError, kda_chunk_fwd, kda_chunk_fwd_selected_algo,
                                            kda_chunk_fwd_workspace_bytes, kda_workspace_status,
                                            workspace_status_words)
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, rel_l2_per_head, rel_l2_states, run_oracle_prefill, to_dev

pytestmark = pytest.mark.gpu


def test_auto_selects_tensor_cores_for_bf16_d128():
    assert kda_chunk_fwd_selected_algo(4, 16384, 16, 128, 128, torch.bfloat16) == "tensor"
    assert kda_chunk_fwd_selected_algo(1, 256, 2, 64, 64, torch.float32) == "simt"
    assert kda_chunk_fwd_selected_algo(4, 16384, 16, 128, 128, torch.bfloat16, "simt") == "simt"


def test_forced_wait_timeout_is_reported_and_context_survives():
    spec = W.custom_prefill([300, 100], num_heads=2, d=128, seed=41)
    x = W.prefill_inputs(spec)
    d = to_dev(x)
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    os.environ["KDA_TEST_FORCE_WAIT_TIMEOUT"] = "1"
    try:
        kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"],
                      workspace=ws, algo="tensor")
        assert kda_workspace_status(ws) == -7
    finally:
        del os.environ["KDA_TEST_FORCE_WAIT_TIMEOUT"]
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], workspace=ws, algo="tensor", check=True)
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16


def test_gate_beyond_range_is_reported_without_room_for_flags():
    """A chunk whose total log decay is below -80 in some channel is outside the
    tensor-core factors' range.  With only the 256-byte status block as workspace there
    is no room for the recomputation flags, and the call reports KDA_ERR_GATE_RANGE
    (the CUDA-core path, which forms every decay pairwise, has no such limit)."""
    spec = W.custom_prefill([128], num_heads=1, d=128, seed=42)
    x = W.prefill_inputs(spec)
    x["g"] = torch.full_like(x["g"], -2.0)  # 64 tokens x -2 = -128 per chunk
    d = to_dev(x)
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(KdaError) as ei:
        kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"],
                      algo="tensor", workspace=ws, check=True)
    assert ei.value.code == -8
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], algo="simt", check=True)
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16


@pytest.mark.parametrize("algo", ["auto", "tensor"])
@pytest.mark.parametrize("case", ["g-2", "g-30-channels", "scalar-g-3"])
def test_gate_beyond_range_is_recomputed_exactly(algo, case):
    """With the workspace kda_chunk_fwd_workspace_bytes() asks for, the sequence-heads
    whose decay leaves the tensor-core range (alpha -> 0: "alpha = 0 clears memory")
    are recomputed token by token in the same call and match the oracle; the others
    keep their tensor-core results, and the status word counts the recomputed ones.
      g-2           g = -2 per token on head 0 (chunk decay -128), the recipe on head 1
      g-30-channels g = -30 on 8 of the 128 key channels of every head, tokens 100-399
      scalar-g-3    one log alpha of -3 per (token, head) on head 1 (Gated DeltaNet form)"""
    spec = W.custom_prefill([300, 1, 129, 64], num_heads=2, d=128, seed=45)
    x = W.prefill_inputs(spec)
    g = x["g"].float()
    if case == "g-2":
        g[:, 0] = -2.0
        want = 3  # sequences 0, 2 and 3 of head 0 reach -128 in a chunk (1 token does not)
    elif case == "g-30-channels":
        g[100:400, :, 8:16] = -30.0
        want = 2 * 2  # tokens 100-399: sequences 0 and 2 (sequence 1 is the one token 300)
    else:
        g = g[..., 0].clone()
        g[:, 1] = -3.0
        want = 3
    x["g"] = g.to(x["g"].dtype).contiguous()
    d = to_dev(x)
    ws = torch.zeros(kda_chunk_fwd_workspace_bytes(4, 494, 2, 128, 128), dtype=torch.uint8, device="cuda")
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], algo=algo, workspace=ws, check=True)
    words = workspace_status_words(ws)
    assert words[0] == 0 and words[3] == want, words
    xo = dict(x)
    if case == "scalar-g-3":  # the oracle takes one log alpha per key channel
        xo["g"] = x["g"].unsqueeze(-1).expand(-1, -1, 128).contiguous()
    ro, rs = run_oracle_prefill(xo)
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16


def test_gate_beyond_range_recomputed_in_place():
    """The recomputation reads the initial state, so a call with final_state aliasing
    init_state must leave a marked pair's initial state untouched until then."""
    spec = W.custom_prefill([200, 130], num_heads=2, d=128, seed=46)
    x = W.prefill_inputs(spec)
    g = x["g"].float()
    g[:, 1] = -2.5
    x["g"] = g.to(x["g"].dtype)
    d = to_dev(x)
    st = d["init_state"].clone()
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], st,
                             final_state=st, check=True)
    assert fin.data_ptr() == st.data_ptr()
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(st.cpu().numpy(), rs) <= TOL_BF16


def test_strong_decay_inside_range():
    """Per-token g = -1.2 (chunk decay -76.8, just inside the range) still matches."""
    spec = W.custom_prefill([200, 64], num_heads=2, d=128, seed=43)
    x = W.prefill_inputs(spec)
    x["g"] = torch.full_like(x["g"], -1.2)
    d = to_dev(x)
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], algo="tensor", check=True)
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16


@pytest.mark.parametrize("algo", ["tensor", "simt"])
def test_strong_decay_after_a_partial_chunk_stays_finite(algo):
    """A sequence's partial last chunk shares its tile with the next sequence's
    first tokens.  Here both decay at g = -2.4 for 32 tokens (each chunk's own
    total, -76.8, is inside the range), so the rows past the first sequence's end
    reach a cumulative decay of -153.6, where exp(-G) overflows fp32.  Those rows
    must contribute nothing: outputs and states stay finite and match."""
    spec = W.custom_prefill([96, 64], num_heads=2, d=128, seed=44)
    x = W.prefill_inputs(spec)
    g = torch.zeros_like(x["g"])
    g[64:128] = -2.4  # the last 32 tokens of sequence 0 and the first 32 of sequence 1
    x["g"] = g.to(x["g"].dtype)
    d = to_dev(x)
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], algo=algo, check=True)
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16
