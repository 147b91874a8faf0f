"""Gated DeltaNet (one log alpha per token and head, applied to every key
channel) and DeltaNet (alpha = 1) through the same kernels ("Kimi Delta
Attention (KDA)", sections on DeltaNet and on Gated DeltaNet's retention gate).

The oracle computes the per-channel recurrence; it is given the per-channel g
that repeats the per-token value on every channel (or g = 0), which is the same
recurrence, so each mode is checked element by element against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_fwd_gb300 import kda_chunk_fwd, kda_decode_step
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, TOL_F32, rel_l2_per_head, rel_l2_states, run_oracle_prefill, to_dev

pytestmark = pytest.mark.gpu


def _gates(g, mode):
    """(g for the GPU call, per-channel g for the oracle) for a gate mode."""
    if mode == "scalar":
        g_tok = g[..., 0].contiguous()
        return g_tok, g_tok.unsqueeze(-1).expand_as(g).contiguous()
    return None, torch.zeros_like(g)


@pytest.mark.parametrize("mode", ["scalar", "none"])
@pytest.mark.parametrize("algo,io,d,tol", [("tensor", "bf16", 128, TOL_BF16),
                                            ("simt", "bf16", 128, TOL_BF16),
                                            ("simt", "f32", 64, TOL_F32)])
def test_prefill_gate_modes(mode, algo, io, d, tol):
    spec = W.custom_prefill([1, 63, 65, 300, 200], num_heads=2, d=d, io=io, gate="mixed", seed=51)
    x = W.prefill_inputs(spec)
    g_gpu, g_ref = _gates(x["g"], mode)
    dv = to_dev(x)
    out, fin = kda_chunk_fwd(dv["q"], dv["k"], dv["v"], None if g_gpu is None else g_gpu.cuda(),
                             dv["beta"], dv["cu_seqlens"], dv["init_state"], algo=algo, check=True)
    ref = dict(x, g=g_ref)
    ro, rs = run_oracle_prefill(ref)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= tol
    assert rel_l2_states(fin.cpu().numpy(), rs) <= tol


def test_scalar_gate_equals_broadcast_channel_gate_on_the_gpu():
    """The per-token mode and the per-channel mode given the repeated value run the
    same recurrence, so on the tensor-core path their results agree to rounding."""
    spec = W.custom_prefill([300, 128], num_heads=2, d=128, gate="mixed", seed=53)
    x = W.prefill_inputs(spec)
    g_tok, g_chan = _gates(x["g"], "scalar")
    dv = to_dev(x)
    a = kda_chunk_fwd(dv["q"], dv["k"], dv["v"], g_tok.cuda(), dv["beta"], dv["cu_seqlens"],
                      dv["init_state"], algo="tensor", check=True)
    b = kda_chunk_fwd(dv["q"], dv["k"], dv["v"], g_chan.cuda(), dv["beta"], dv["cu_seqlens"],
                      dv["init_state"], algo="tensor", check=True)
    assert rel_l2_per_head(a[0].float().cpu().numpy(), b[0].float().cpu().numpy(),
                           x["cu_seqlens"].numpy()) <= 1e-2
    assert rel_l2_states(a[1].cpu().numpy(), b[1].cpu().numpy()) <= 1e-2


@pytest.mark.parametrize("mode", ["scalar", "none"])
@pytest.mark.parametrize("io,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
def test_decode_gate_modes(mode, io, tol):
    spec = W.DecodeSpec(5, 3, 128, 128, 12, io, "mixed", 52)
    y = W.decode_inputs(spec)
    g_gpu, g_ref = _gates(y["g"], mode)
    st = y["state"].clone().cuda()
    outs = []
    for t in range(spec.steps):
        gt = None if g_gpu is None else g_gpu[t].cuda()
        outs.append(kda_decode_step(y["q"][t].cuda(), y["k"][t].cuda(), y["v"][t].cuda(), gt,
                                    y["beta"][t].cuda(), st).float().cpu())
    ro, rs = oracle.kda_decode_steps(y["q"], y["k"], y["v"], g_ref, y["beta"], y["state"])
    got = torch.stack(outs).numpy()
    g2 = np.swapaxes(got, 0, 1).reshape(-1, spec.num_heads, spec.d_v)
    r2 = np.swapaxes(ro, 0, 1).reshape(-1, spec.num_heads, spec.d_v)
    cu = np.arange(spec.num_seqs + 1) * spec.steps
    assert rel_l2_per_head(g2, r2, cu) <= tol
    assert rel_l2_states(st.cpu().numpy(), rs) <= tol
