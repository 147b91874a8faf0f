"""The optional input steps inside the kernels (kda_shape.prep): SiLU and then the
L2 norm of every (token, head) row of q and k, and the sigmoid of a write-strength
logit ("22580: от GPT-2 до Kimi K3", section "DeltaNet, или Fast Weight
Programmers", the forward with a per-token write strength).

Each kernel gets raw q, k (not normalised) and beta logits; the oracle applies
oracle.preprocess to the same values and runs the recurrence, and the two are
compared element by element with the usual tolerances."""
import numpy as np
import pytest
import torch

import oracle
from kimi_delta_attention_fwd_gb300 import (kda_chunk_fwd, kda_chunk_fwd_workspace_bytes,
                                            kda_decode_step, kda_recurrent_fwd)
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, TOL_F32, rel_l2_per_head, rel_l2_states, to_dev

pytestmark = pytest.mark.gpu

ALL = dict(qk_silu=True, qk_l2norm=True, beta_sigmoid=True)
FLAG_SETS = [ALL, dict(qk_l2norm=True), dict(qk_silu=True, beta_sigmoid=True),
             dict(beta_sigmoid=True)]
LENS = [1, 63, 65, 300, 200]


def _qk_scale(flags):
    # without the norm the raw keys must keep beta ||k||^2 below 2 (a stable delta rule)
    return 1.0 if flags.get("qk_l2norm") else 0.1


def _gates(x, mode):
    """(g for the GPU call, per-channel g for the oracle)."""
    if mode == "channel":
        return x["g"], x["g"]
    if mode == "scalar":
        g_tok = x["g"][..., 0].contiguous()
        return g_tok, g_tok.unsqueeze(-1).expand_as(x["g"]).contiguous()
    return None, torch.zeros_like(x["g"])


def _oracle_prefill(x, g_ref, flags):
    q, k, b = oracle.preprocess(x["q"], x["k"], x["beta"], **flags)
    return oracle.kda_fwd(q, k, x["v"], g_ref, b, x["cu_seqlens"], x["init_state"])


def _prefill(x, g, flags, **kw):
    d = to_dev(x)
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], None if g is None else g.cuda(), d["beta"],
                             d["cu_seqlens"], d["init_state"], check=True, **flags, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), fin.cpu().numpy()


@pytest.mark.parametrize("flags", FLAG_SETS, ids=["all", "l2", "silu+sigmoid", "sigmoid"])
@pytest.mark.parametrize("algo,io,d,tol", [("tensor", "bf16", 128, TOL_BF16),
                                            ("simt", "bf16", 128, TOL_BF16),
                                            ("simt", "f32", 64, TOL_F32)])
def test_prefill_input_steps(flags, algo, io, d, tol):
    x = W.prefill_inputs(W.custom_prefill(LENS, num_heads=2, d=d, io=io, seed=61), raw=True,
                         qk_scale=_qk_scale(flags))
    out, fin = _prefill(x, x["g"], flags, algo=algo)
    ro, rs = _oracle_prefill(x, x["g"], flags)
    assert rel_l2_per_head(out, ro, x["cu_seqlens"].numpy()) <= tol
    assert rel_l2_states(fin, rs) <= tol


@pytest.mark.parametrize("mode", ["scalar", "none"])
def test_tensor_prefill_input_steps_other_gates(mode):
    x = W.prefill_inputs(W.custom_prefill(LENS, num_heads=2, d=128, gate="mixed", seed=62),
                         raw=True)
    g_gpu, g_ref = _gates(x, mode)
    out, fin = _prefill(x, g_gpu, ALL, algo="tensor")
    ro, rs = _oracle_prefill(x, g_ref, ALL)
    assert rel_l2_per_head(out, ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin, rs) <= TOL_BF16


def test_tensor_schedules_agree_with_input_steps():
    """The solve-helper schedule (few sequence-heads, full workspace) and the plain
    one (256-byte workspace) run the same input steps: identical results."""
    x = W.prefill_inputs(W.custom_prefill([700, 129], num_heads=2, d=128, seed=63), raw=True)
    T, H = x["q"].shape[0], 2
    need = kda_chunk_fwd_workspace_bytes(2, T, H, 128, 128)
    assert need > 256
    full = torch.zeros(need, dtype=torch.uint8, device="cuda")
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    a = _prefill(x, x["g"], ALL, algo="tensor", workspace=full)
    b = _prefill(x, x["g"], ALL, algo="tensor", workspace=small)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    ro, rs = _oracle_prefill(x, x["g"], ALL)
    assert rel_l2_per_head(a[0], ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(a[1], rs) <= TOL_BF16


@pytest.mark.parametrize("algo", ["tensor", "simt"])
def test_zero_rows_stay_finite(algo):
    """Rows of q and k that are all zero normalise to zero (F.normalize's eps),
    so nothing is written or read for them and nothing becomes NaN."""
    x = W.prefill_inputs(W.custom_prefill([130, 70], num_heads=2, d=128, seed=64), raw=True)
    for t in (0, 5, 64, 129, 131):
        x["q"][t] = 0
        x["k"][t] = 0
    out, fin = _prefill(x, x["g"], ALL, algo=algo)
    assert np.isfinite(out).all() and np.isfinite(fin).all()
    ro, rs = _oracle_prefill(x, x["g"], ALL)
    assert rel_l2_per_head(out, ro, x["cu_seqlens"].numpy()) <= TOL_BF16
    assert rel_l2_states(fin, rs) <= TOL_BF16


@pytest.mark.parametrize("io,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128)])
def test_decode_input_steps(io, tol, dk, dv):
    spec = W.DecodeSpec(6, 3, dk, dv, 10, io, "std", 65)
    y = W.decode_inputs(spec, raw=True)
    st = y["state"].clone().cuda()
    outs = []
    for t in range(spec.steps):
        outs.append(kda_decode_step(y["q"][t].cuda(), y["k"][t].cuda(), y["v"][t].cuda(),
                                    y["g"][t].cuda(), y["beta"][t].cuda(), st, **ALL).float().cpu())
    q, k, b = oracle.preprocess(y["q"], y["k"], y["beta"], **ALL)
    ro, rs = oracle.kda_decode_steps(q, k, y["v"], y["g"], b, y["state"])
    got = torch.stack(outs).numpy()
    g2 = np.swapaxes(got, 0, 1).reshape(-1, spec.num_heads, spec.d_v)
    r2 = np.swapaxes(ro, 0, 1).reshape(-1, spec.num_heads, spec.d_v)
    cu = np.arange(spec.num_seqs + 1) * spec.steps
    assert rel_l2_per_head(g2, r2, cu) <= tol
    assert rel_l2_states(st.cpu().numpy(), rs) <= tol


@pytest.mark.parametrize("io,tol", [("bf16", TOL_BF16), ("f32", TOL_F32)])
def test_recurrent_input_steps(io, tol):
    x = W.prefill_inputs(W.custom_prefill([0, 1, 3, 9, 17], num_heads=2, d=128, io=io, seed=66),
                         raw=True)
    d = to_dev(x)
    out, fin = kda_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 d["init_state"], **ALL)
    torch.cuda.synchronize()
    ro, rs = _oracle_prefill(x, x["g"], ALL)
    assert rel_l2_per_head(out.float().cpu().numpy(), ro, x["cu_seqlens"].numpy()) <= tol
    assert rel_l2_states(fin.cpu().numpy(), rs) <= tol


@pytest.mark.parametrize("name,pairs", [("prefill_bf16", [(0, 0), (1, 7), (2, 11), (3, 15)]),
                                        ("long_prefill_16k_bf16", [(0, 0), (0, 31)])])
def test_input_steps_at_full_size_sampled(name, pairs):
    """The benchmark workloads (4 x 4096 x 16 heads, plain schedule; 1 x 16384 x 32 heads,
    solve helpers) from raw inputs with all three steps, sampled (sequence, head) pairs
    against the oracle."""
    x = W.prefill_inputs(W.named(name), device="cuda", raw=True)
    out, fin = kda_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                             x["init_state"], check=True, **ALL)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(fin).all()
    cu = x["cu_seqlens"].cpu().tolist()
    for n, h in pairs:
        a, b = cu[n], cu[n + 1]
        sl = lambda t: t[a:b, h:h + 1].cpu()
        q, k, beta = oracle.preprocess(sl(x["q"]), sl(x["k"]), sl(x["beta"]), **ALL)
        ro, rs = oracle.kda_fwd(q, k, sl(x["v"]), sl(x["g"]), beta, np.array([0, b - a]),
                                x["init_state"][n:n + 1, h:h + 1].cpu())
        eo = rel_l2_per_head(out[a:b, h:h + 1].float().cpu().numpy(), ro, [0, b - a])
        es = rel_l2_states(fin[n:n + 1, h:h + 1].cpu().numpy(), rs)
        assert eo <= TOL_BF16 and es <= TOL_BF16, (n, h, eo, es)


# ------------------------------------------------------------------ the gate step
# g holds gate logits x and the kernels take log alpha = -c softplus(x)
# (KDA_PREP_G_SOFTPLUS, c = gate_scale); the oracle gets oracle.gate_from_logits(x, c)
# of the same (rounded) logits.
@pytest.mark.parametrize("recipe", ["std", "mixed"])
@pytest.mark.parametrize("algo,io,d,tol", [("tensor", "bf16", 128, TOL_BF16),
                                            ("simt", "bf16", 128, TOL_BF16),
                                            ("simt", "f32", 64, TOL_F32)])
def test_prefill_softplus_gate(recipe, algo, io, d, tol):
    spec = W.custom_prefill(LENS, num_heads=2, d=d, io=io, gate=recipe, seed=63)
    x = W.prefill_inputs(spec, raw_gate=True)
    c = W.gate_scale(spec)
    out, fin = _prefill(x, x["g"], {}, algo=algo, g_softplus=True, gate_scale=c)
    g_ref = oracle.gate_from_logits(x["g"], c)
    ro, rs = oracle.kda_fwd(x["q"], x["k"], x["v"], g_ref, x["beta"], x["cu_seqlens"],
                            x["init_state"])
    assert rel_l2_per_head(out, ro, x["cu_seqlens"].numpy()) <= tol
    assert rel_l2_states(fin, rs) <= tol


@pytest.mark.parametrize("schedule", ["helper", "plain"])
def test_tensor_prefill_softplus_gate_all_steps(schedule):
    """Every input step at once, per-token gate logits too, both schedules."""
    spec = W.custom_prefill(LENS, num_heads=2, d=128, gate="mixed", seed=64)
    x = W.prefill_inputs(spec, raw=True, raw_gate=True)
    ws = None if schedule == "helper" else torch.zeros(512, dtype=torch.uint8, device="cuda")
    for mode in ("channel", "scalar"):
        g_gpu, g_logit = _gates(x, mode)
        out, fin = _prefill(x, g_gpu, dict(ALL, g_softplus=True), algo="tensor", workspace=ws)
        ro, rs = _oracle_prefill(x, oracle.gate_from_logits(g_logit, 1.0), ALL)
        assert rel_l2_per_head(out, ro, x["cu_seqlens"].numpy()) <= TOL_BF16
        assert rel_l2_states(fin, rs) <= TOL_BF16


@pytest.mark.parametrize("io,d,tol", [("bf16", 128, TOL_BF16), ("f32", 64, TOL_F32)])
def test_decode_and_recurrent_softplus_gate(io, d, tol):
    ds = W.DecodeSpec(5, 2, d, d, 3, io, "std", 65)
    y = W.decode_inputs(ds, raw_gate=True)
    c = W.gate_scale(ds)
    g_ref = oracle.gate_from_logits(y["g"], c)
    ro, rs = oracle.kda_decode_steps(y["q"], y["k"], y["v"], g_ref, y["beta"], y["state"])
    st = y["state"].clone().cuda()
    outs = []
    for t in range(ds.steps):
        outs.append(kda_decode_step(y["q"][t].cuda(), y["k"][t].cuda(), y["v"][t].cuda(),
                                    y["g"][t].cuda(), y["beta"][t].cuda(), st, g_softplus=True,
                                    gate_scale=c).float().cpu().numpy())
    np.testing.assert_array_less(
        np.linalg.norm(np.stack(outs) - ro) / np.linalg.norm(ro), tol)
    assert rel_l2_states(st.cpu().numpy(), rs) <= tol
    # the same steps as one recurrent pass per sequence
    N = ds.num_seqs
    pack = lambda t: t.transpose(0, 1).reshape(N * ds.steps, *t.shape[2:]).contiguous().cuda()
    cu = torch.arange(N + 1, dtype=torch.int32, device="cuda") * ds.steps
    o2, f2 = kda_recurrent_fwd(pack(y["q"]), pack(y["k"]), pack(y["v"]), pack(y["g"]),
                               pack(y["beta"]), cu, y["state"].cuda(), g_softplus=True,
                               gate_scale=c)
    ro_packed = np.swapaxes(ro, 0, 1).reshape(N * ds.steps, 2, d)
    np.testing.assert_array_less(
        np.linalg.norm(o2.float().cpu().numpy() - ro_packed) / np.linalg.norm(ro_packed), tol)
    assert rel_l2_states(f2.cpu().numpy(), rs) <= tol
