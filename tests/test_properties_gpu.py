"""Properties of the recurrence that hold at any size, checked on the full-size
workloads where the oracle would take too long ("Kimi Delta Attention (KDA)",
the delta rule's predict-and-correct step and its forget gate):

- With a unit key, q_t = k_t and beta_t = 1 the write replaces what the key
  reads: S_t^T k_t = S~_t^T k_t + (v_t - S~_t^T k_t) = v_t whatever the decay and
  the earlier state, so every output is scale * v_t.
- With beta = 0 nothing is written: the state only decays, S_T = Diag(exp(sum_t g_t)) S_0
  per key channel, and o_t = scale * (Diag(exp(sum_{u<=t} g_u)) S_0)^T q_t.

Every kernel is checked: the tensor-core prefill in both schedules, the CUDA-core
prefill, the decode step and the multi-token recurrent pass."""
import numpy as np
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import kda_chunk_fwd, kda_decode_step, kda_recurrent_fwd
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, rel_l2_per_head, rel_l2_states

pytestmark = pytest.mark.gpu


def _full_write_inputs(name="prefill_bf16"):
    x = W.prefill_inputs(W.named(name), device="cuda")
    x["q"] = x["k"].clone()                    # unit keys (the recipe normalises k)
    x["beta"] = torch.ones_like(x["beta"])
    return x


def _prefill(x, **kw):
    return kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                         x["init_state"], check=True, **kw)


@pytest.mark.parametrize("how", ["tensor", "tensor-plain", "simt", "recurrent"])
def test_full_write_reads_back_v_at_full_size(how):
    x = _full_write_inputs()
    scale = 1.0 / np.sqrt(x["q"].shape[2])
    if how == "recurrent":
        out, _ = kda_recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                                   x["init_state"], output_final_state=False)
    elif how == "tensor-plain":
        out, _ = _prefill(x, algo="tensor", workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    else:
        out, _ = _prefill(x, algo=how)
    torch.cuda.synchronize()
    want = (scale * x["v"].float()).cpu().numpy()
    assert rel_l2_per_head(out.float().cpu().numpy(), want, x["cu_seqlens"].cpu().numpy()) <= TOL_BF16


def test_full_write_reads_back_v_in_decode():
    spec = W.named("decode_bf16")
    y = W.decode_inputs(W.DecodeSpec(spec.num_seqs, spec.num_heads, spec.d_k, spec.d_v, 2,
                                     spec.io_dtype, spec.gate, spec.seed), device="cuda")
    st = y["state"].clone()
    scale = 1.0 / np.sqrt(spec.d_k)
    for t in range(2):
        o = kda_decode_step(y["k"][t], y["k"][t], y["v"][t], y["g"][t], torch.ones_like(y["beta"][t]), st)
        torch.cuda.synchronize()
        got = o.float().cpu().numpy()
        want = (scale * y["v"][t].float()).cpu().numpy()
        cu = np.arange(spec.num_seqs + 1)
        assert rel_l2_per_head(got, want, cu) <= TOL_BF16


def _slow_gate(x, factor):
    """g scaled towards 0 (then rounded to the I/O dtype), so that the total decay
    of a long sequence stays well inside fp32 and the check is not trivially 0."""
    x["g"] = (x["g"].float() * factor).to(x["g"].dtype)


@pytest.mark.parametrize("how", ["tensor", "tensor-plain", "simt"])
def test_zero_write_only_decays_at_full_size(how):
    x = W.prefill_inputs(W.named("long_prefill_bf16"), device="cuda")
    x["beta"] = torch.zeros_like(x["beta"])
    _slow_gate(x, 1e-4)  # sum of g over 65536 tokens: about -1
    kw = {"algo": "tensor" if how.startswith("tensor") else how}
    if how == "tensor-plain":
        kw["workspace"] = torch.empty(256, dtype=torch.uint8, device="cuda")
    _, fin = _prefill(x, **kw)
    torch.cuda.synchronize()
    # S_T = Diag(exp(sum_t g_t)) S_0: one factor per (sequence, head, key channel)
    cu = x["cu_seqlens"].cpu().numpy()
    gsum = torch.stack([x["g"][cu[n]:cu[n + 1]].double().sum(0) for n in range(len(cu) - 1)])
    want = (torch.exp(gsum).unsqueeze(-1) * x["init_state"].double()).cpu().numpy()
    # The tensor-core state update forms Kc^T E as Kc^T (E - V) + Kc^T V in fp32: with
    # nothing written the two V terms cancel only to fp32 rounding, an absolute error
    # per chunk of about 2^-24 |Kc^T V|; the bf16 tolerance covers it while the state
    # keeps its scale.  The CUDA-core path takes the fp32 tolerance.
    tol = TOL_BF16 if how.startswith("tensor") else 1e-4
    assert rel_l2_states(fin.cpu().numpy(), want) <= tol


def test_zero_write_outputs_follow_the_decayed_state():
    spec = W.custom_prefill([1000, 333], num_heads=4, d=128, gate="mixed", seed=91)
    x = W.prefill_inputs(spec, device="cuda")
    x["beta"] = torch.zeros_like(x["beta"])
    _slow_gate(x, 1e-2)
    out, _ = _prefill(x, algo="tensor")
    torch.cuda.synchronize()
    scale = 1.0 / np.sqrt(128)
    cu = x["cu_seqlens"].cpu().numpy()
    want = torch.empty_like(out, dtype=torch.float64)
    for n in range(len(cu) - 1):
        gc = torch.cumsum(x["g"][cu[n]:cu[n + 1]].double(), 0)                 # [L, H, d_k]
        decayed = torch.exp(gc).unsqueeze(-1) * x["init_state"][n].double()    # [L, H, d_k, d_v]
        want[cu[n]:cu[n + 1]] = scale * torch.einsum("thk,thkv->thv", x["q"][cu[n]:cu[n + 1]].double(),
                                                     decayed)
    assert rel_l2_per_head(out.float().cpu().numpy(), want.cpu().numpy(), cu) <= TOL_BF16
