"""GPU parity: the CUDA path (through the Python binding and the C ABI) against
the fp64 oracle on the same seeded inputs.

Tolerances (max over (sequence, head) of the relative L2 error, for outputs
and for final states): 1e-4 with fp32 I/O, 2e-2 with bf16 I/O and fp32 state.
"""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_fwd_gb300 import (KdaError, kda_chunk_fwd, kda_decode_step,
                                            kda_workspace_status)
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import (TOL_BF16, TOL_F32, rel_l2_per_head, rel_l2_states, run_gpu_prefill,
                    run_oracle_prefill, to_dev)

pytestmark = pytest.mark.gpu

ALGOS_BF16 = ["auto", "simt"]


def _check_prefill(x, tol, algo="auto"):
    out, fin = run_gpu_prefill(x, algo=algo)
    ro, rs = run_oracle_prefill(x)
    cu = x["cu_seqlens"].numpy()
    eo, es = rel_l2_per_head(out, ro, cu), rel_l2_states(fin, rs)
    assert eo <= tol and es <= tol, (eo, es)
    assert np.isfinite(out).all() and np.isfinite(fin).all()
    return eo, es


def test_tiny_fp32_workload():
    """1 sequence x 256 tokens, H=2, d=64, fp32 I/O, zero initial state."""
    _check_prefill(W.prefill_inputs(W.named("tiny_fp32")), TOL_F32)


@pytest.mark.parametrize("d", [64, 128])
def test_fp32_ragged_varlen(d):
    spec = W.custom_prefill([1, 63, 64, 65, 200, 0, 129], num_heads=3, d=d, io="f32", seed=21)
    _check_prefill(W.prefill_inputs(spec), TOL_F32)


@pytest.mark.parametrize("algo", ALGOS_BF16)
def test_bf16_ragged_varlen(algo):
    spec = W.custom_prefill([1, 63, 64, 65, 300, 0, 129, 1000], num_heads=4, d=128, seed=22)
    _check_prefill(W.prefill_inputs(spec), TOL_BF16, algo)


@pytest.mark.parametrize("algo", ALGOS_BF16)
def test_bf16_mixed_decay(algo):
    """Slow and fast decay per channel (g = -softplus(N(-2, 1)))."""
    spec = W.custom_prefill([777, 2048], num_heads=4, d=128, gate="mixed", seed=23)
    _check_prefill(W.prefill_inputs(spec), TOL_BF16, algo)


@pytest.mark.parametrize("dk,dv", [(64, 128), (128, 64), (64, 64)])
def test_bf16_other_head_dims(dk, dv):
    spec = W.custom_prefill([130, 64], num_heads=2, d=dk, d_v=dv, seed=24)
    _check_prefill(W.prefill_inputs(spec), TOL_BF16)


def test_zero_state_default_and_aliasing_and_no_final_state():
    spec = W.custom_prefill([90, 190], num_heads=2, d=128, seed=25)
    x = W.prefill_inputs(spec)
    d = to_dev(x)
    # init_state=None means zeros
    o1, f1 = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], None)
    zeros = torch.zeros_like(d["init_state"])
    o2, f2 = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], zeros)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)
    # final_state aliasing init_state: in-place update
    ref_o, ref_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 d["init_state"])
    st = d["init_state"].clone()
    o3, f3 = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], st,
                           final_state=st)
    assert f3.data_ptr() == st.data_ptr()
    assert torch.equal(o3, ref_o) and torch.equal(st, ref_f)
    # no final state requested
    o4, f4 = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                           d["init_state"], output_final_state=False)
    assert f4 is None and torch.equal(o4, ref_o)


@pytest.mark.parametrize("algo", ["tensor", "simt"])
def test_small_write_strengths(algo):
    """beta about ten times smaller than the recipe's (0.005 .. 0.1): the new values
    E are then far smaller than v, which is where a bf16 operand formed as E - v
    would lose the output and state to rounding (it measured 3 % / 4.5 % on
    4 x 4096); the tensor-core path folds beta into k and v instead."""
    spec = W.custom_prefill([700, 300, 129], num_heads=4, d=128, gate="mixed", seed=24)
    x = W.prefill_inputs(spec)
    x["beta"] = (x["beta"].float() * 0.1).to(x["beta"].dtype)
    _check_prefill(x, TOL_BF16, algo=algo)


def test_empty_inputs():
    dev = "cuda"
    H, dk = 2, 128
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device=dev)
    # no sequences at all
    out, fin = kda_chunk_fwd(e(0, H, dk), e(0, H, dk), e(0, H, dk), e(0, H, dk), e(0, H),
                             torch.zeros(1, dtype=torch.int32, device=dev))
    assert out.shape == (0, H, dk) and fin.shape == (0, H, dk, dk)
    # sequences that are all empty keep their initial state
    init = torch.randn(3, H, dk, dk, device=dev)
    out, fin = kda_chunk_fwd(e(0, H, dk), e(0, H, dk), e(0, H, dk), e(0, H, dk), e(0, H),
                             torch.zeros(4, dtype=torch.int32, device=dev), init)
    torch.cuda.synchronize()
    assert torch.equal(fin, init)


def test_checkpoint_resume_and_prefill_then_decode():
    """prefill(T1) -> prefill(T2 from state) and prefill(T) -> decode steps both
    equal a single prefill over all tokens (up to the bf16 tolerance)."""
    spec = W.custom_prefill([400], num_heads=4, d=128, seed=26)
    x = W.prefill_inputs(spec)
    d = to_dev(x)
    T1, T = 250, 400
    full_o, full_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                   d["init_state"])
    cu1 = torch.tensor([0, T1], dtype=torch.int32, device="cuda")
    sl = lambda t, a, b: t[a:b].contiguous()
    o1, f1 = kda_chunk_fwd(*(sl(d[n], 0, T1) for n in ("q", "k", "v", "g", "beta")), cu1,
                           d["init_state"])
    cu2 = torch.tensor([0, T - T1 - 5], dtype=torch.int32, device="cuda")
    o2, f2 = kda_chunk_fwd(*(sl(d[n], T1, T - 5) for n in ("q", "k", "v", "g", "beta")), cu2, f1)
    outs = [o1, o2]
    st = f2.clone()
    for t in range(T - 5, T):
        outs.append(kda_decode_step(*(d[n][t:t + 1].contiguous() for n in ("q", "k", "v", "g", "beta")),
                                    st))
    got = torch.cat(outs).float().cpu().numpy()
    cu = np.array([0, T])
    assert rel_l2_per_head(got, full_o.float().cpu().numpy(), cu) <= TOL_BF16
    assert rel_l2_states(st.cpu().numpy(), full_f.cpu().numpy()) <= TOL_BF16


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("io,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_decode_steps_small(io, tol, dk, dv):
    spec = W.DecodeSpec(5, 3, dk, dv, 12, io, "std", 31)
    y = W.decode_inputs(spec)
    st = y["state"].clone().cuda()
    outs = []
    for t in range(spec.steps):
        outs.append(kda_decode_step(y["q"][t].cuda(), y["k"][t].cuda(), y["v"][t].cuda(),
                                    y["g"][t].cuda(), y["beta"][t].cuda(), st).float().cpu())
    ro, rs = oracle.kda_decode_steps(y["q"], y["k"], y["v"], y["g"], y["beta"], y["state"])
    got = torch.stack(outs).numpy()  # [steps, N, H, dv]
    # per (seq, head) over its steps
    g2 = np.swapaxes(got, 0, 1).reshape(-1, spec.num_heads, dv)
    r2 = np.swapaxes(ro, 0, 1).reshape(-1, spec.num_heads, dv)
    cu = np.arange(spec.num_seqs + 1) * spec.steps
    assert rel_l2_per_head(g2, r2, cu) <= tol
    assert rel_l2_states(st.cpu().numpy(), rs) <= tol


def test_decode_workload_full_size_sampled():
    """256 sequences x 32 heads, 128 consecutive steps, state updated in place;
    all outputs of 48 sampled (sequence, head) pairs and their final states
    against the oracle, every output finite."""
    spec = W.named("decode_bf16")
    y = W.decode_inputs(spec, device="cuda")
    st = y["state"].clone()
    outs = torch.empty((spec.steps, spec.num_seqs, spec.num_heads, spec.d_v), dtype=torch.bfloat16,
                       device="cuda")
    for t in range(spec.steps):
        kda_decode_step(y["q"][t], y["k"][t], y["v"][t], y["g"][t], y["beta"][t], st, out=outs[t])
    torch.cuda.synchronize()
    assert torch.isfinite(outs.float()).all() and torch.isfinite(st).all()
    gen = torch.Generator().manual_seed(0)
    ns = torch.randint(0, spec.num_seqs, (48,), generator=gen).tolist()
    hs = torch.randint(0, spec.num_heads, (48,), generator=gen).tolist()
    ns[0], hs[0], ns[1], hs[1] = 0, 0, spec.num_seqs - 1, spec.num_heads - 1
    sel = lambda t: torch.stack([t[:, n, h] for n, h in zip(ns, hs)], 1).unsqueeze(2).cpu()
    ro, rs = oracle.kda_decode_steps(sel(y["q"]), sel(y["k"]), sel(y["v"]), sel(y["g"]),
                                     sel(y["beta"]),
                                     torch.stack([y["state"][n, h] for n, h in zip(ns, hs)]).unsqueeze(1).cpu())
    got = sel(outs).float().numpy()
    cu = np.arange(49) * spec.steps
    g2 = np.swapaxes(got, 0, 1).reshape(-1, 1, spec.d_v)
    r2 = np.swapaxes(ro, 0, 1).reshape(-1, 1, spec.d_v)
    assert rel_l2_per_head(g2, r2, cu) <= TOL_BF16
    fin = torch.stack([st[n, h] for n, h in zip(ns, hs)]).unsqueeze(1).cpu().numpy()
    assert rel_l2_states(fin, rs) <= TOL_BF16


# ------------------------------------------------------- full-size prefill
def test_prefill_workload_full_size():
    """4 x 4096 tokens, H=16, d=128, bf16: every (sequence, head) against the oracle."""
    x = W.prefill_inputs(W.named("prefill_bf16"))
    _check_prefill(x, TOL_BF16)


def _sampled_full_size(spec, pairs, device="cuda"):
    x = W.prefill_inputs(spec, device=device)
    out, fin = kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                             x["init_state"], check=True)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    cu = x["cu_seqlens"].cpu().tolist()
    worst_o = worst_s = 0.0
    for n, h in pairs:
        a, b = cu[n], cu[n + 1]
        sl = lambda t: t[a:b, h:h + 1].cpu()
        ro, rs = oracle.kda_fwd(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(x["beta"]),
                                np.array([0, b - a]),
                                x["init_state"][n:n + 1, h:h + 1].cpu())
        worst_o = max(worst_o, rel_l2_per_head(out[a:b, h:h + 1].float().cpu().numpy(), ro,
                                               [0, b - a]))
        worst_s = max(worst_s, rel_l2_states(fin[n:n + 1, h:h + 1].cpu().numpy(), rs))
    assert worst_o <= TOL_BF16 and worst_s <= TOL_BF16, (worst_o, worst_s)


def test_long_prefill_full_size_sampled():
    """1 x 65536 tokens, H=32, mixed decay: 3 heads against the oracle."""
    _sampled_full_size(W.named("long_prefill_bf16"), [(0, 0), (0, 17), (0, 31)])


def test_varlen_prefill_full_size_sampled():
    """64 packed sequences, lengths U[512, 16384], H=32: the longest, the shortest
    and four more (sequence, head) pairs against the oracle."""
    spec = W.named("varlen_prefill_bf16")
    lens = list(spec.seqlens)
    longest, shortest = lens.index(max(lens)), lens.index(min(lens))
    _sampled_full_size(spec, [(longest, 0), (shortest, 31), (0, 5), (63, 12), (31, 20), (17, 9)])


def test_device_status_is_clean_after_a_call():
    spec = W.custom_prefill([200], num_heads=2, d=128, seed=27)
    d = to_dev(W.prefill_inputs(spec))
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"],
                  workspace=ws)
    assert kda_workspace_status(ws) == 0


def test_rejects_wrong_arguments_without_launching():
    spec = W.custom_prefill([64], num_heads=2, d=128, seed=28)
    d = to_dev(W.prefill_inputs(spec))
    with pytest.raises(KdaError) as ei:
        kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], d["init_state"],
                      workspace=torch.zeros(8, dtype=torch.uint8, device="cuda"))
    assert ei.value.code == -4
