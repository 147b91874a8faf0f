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
                                            kda_workspace_status)
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


def test_gate_beyond_range_is_reported():
    """A chunk whose total log decay is below -80 in some channel is outside the
    tensor-core path's range: the call reports KDA_ERR_GATE_RANGE (the CUDA-core
    path, which forms every decay pairwise, has no such limit)."""
    spec = W.custom_prefill([128], num_heads=1, d=128, seed=42)
    x = W.prefill_inputs(spec)
    x["g"] = torch.full_like(x["g"], -2.0)  # 64 tokens x -2 = -128 per chunk
    d = to_dev(x)
    with pytest.raises(KdaError) as ei:
        kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"],
                      algo="tensor", check=True)
    assert ei.value.code == -8
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], algo="simt", check=True)
    ro, rs = run_oracle_prefill(x)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin.cpu().numpy(), rs) <= TOL_BF16


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
