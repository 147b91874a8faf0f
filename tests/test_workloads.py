"""The seeded input recipe: sizes of the named workloads and the value
distributions (unit-norm q and k, g <= 0, beta in (0, 1), state std 0.02)."""
import torch

from kimi_delta_attention_fwd_gb300 import workloads as W


def test_named_sizes():
    t = W.named("tiny_fp32")
    assert (t.total_tokens, t.num_heads, t.d_k, t.io_dtype, t.init, t.seed) == (256, 2, 64, "f32", "zeros", 0)
    p = W.named("prefill_bf16")
    assert (p.num_seqs, p.total_tokens, p.num_heads, p.d_k) == (4, 4 * 4096, 16, 128)
    lp = W.named("long_prefill_bf16")
    assert (lp.total_tokens, lp.num_heads, lp.gate) == (65536, 32, "mixed")
    d = W.named("decode_bf16")
    assert (d.num_seqs, d.num_heads, d.steps, d.d_k) == (256, 32, 128, 128)
    v = W.named("varlen_prefill_bf16")
    assert v.num_seqs == 64 and all(512 <= x <= 16384 for x in v.seqlens)
    assert 450_000 < v.total_tokens < 630_000  # ~540K expected
    assert W.named("varlen_prefill_bf16").seqlens == v.seqlens  # seeded


def test_value_distributions_and_layout():
    spec = W.custom_prefill([70, 0, 130], num_heads=3, d=64, io="f32", seed=5)
    x = W.prefill_inputs(spec)
    T = 200
    assert x["q"].shape == (T, 3, 64) and x["v"].shape == (T, 3, 64) and x["beta"].shape == (T, 3)
    assert x["cu_seqlens"].tolist() == [0, 70, 70, 200] and x["cu_seqlens"].dtype == torch.int32
    torch.testing.assert_close(x["q"].norm(dim=-1), torch.ones(T, 3), rtol=0, atol=1e-5)
    torch.testing.assert_close(x["k"].norm(dim=-1), torch.ones(T, 3), rtol=0, atol=1e-5)
    assert (x["g"] <= 0).all() and (x["g"] > -1.0).all()
    assert (x["beta"] > 0).all() and (x["beta"] < 1).all()
    assert 0.015 < x["init_state"].std().item() < 0.025
    mixed = W.prefill_inputs(W.custom_prefill([512], 2, 64, "bf16", gate="mixed", seed=1))
    assert mixed["g"].dtype == torch.bfloat16 and (mixed["g"] <= 0).all()
    assert mixed["g"].float().mean().item() < -0.1  # softplus(N(-2, 1)) ~ 0.2 on average


def test_seeded_and_deterministic():
    spec = W.custom_prefill([33], num_heads=2, d=64, seed=9)
    a, b = W.prefill_inputs(spec), W.prefill_inputs(spec)
    for key in ("q", "k", "v", "g", "beta", "init_state"):
        assert torch.equal(a[key], b[key])
    d = W.decode_inputs(W.DecodeSpec(4, 2, 64, 64, 3))
    assert d["q"].shape == (3, 4, 2, 64) and d["state"].shape == (4, 2, 64, 64)


def test_raw_inputs_are_the_same_draws_before_the_input_steps():
    """raw=True keeps q, k (times qk_scale) and beta as drawn, before the L2 norm and the
    sigmoid of the recipe; every other tensor is the same."""
    spec = W.custom_prefill([70, 33], num_heads=2, d=64, io="f32", seed=7)
    a = W.prefill_inputs(spec)
    b = W.prefill_inputs(spec, raw=True, qk_scale=0.5)
    for key in ("v", "g", "init_state", "cu_seqlens"):
        assert torch.equal(a[key], b[key])
    torch.testing.assert_close(b["k"] / b["k"].norm(dim=-1, keepdim=True), a["k"], rtol=1e-6, atol=1e-6)
    torch.testing.assert_close(b["q"] / b["q"].norm(dim=-1, keepdim=True), a["q"], rtol=1e-6, atol=1e-6)
    torch.testing.assert_close(torch.sigmoid(b["beta"]), a["beta"], rtol=1e-6, atol=1e-7)
    c = W.prefill_inputs(spec, raw=True)
    torch.testing.assert_close(b["q"], 0.5 * c["q"], rtol=0, atol=0)
    d = W.decode_inputs(W.DecodeSpec(3, 2, 64, 64, 4, "f32", "std", 5))
    e = W.decode_inputs(W.DecodeSpec(3, 2, 64, 64, 4, "f32", "std", 5), raw=True)
    assert torch.equal(d["v"], e["v"]) and torch.equal(d["state"], e["state"])
    torch.testing.assert_close(torch.sigmoid(e["beta"]), d["beta"], rtol=1e-6, atol=1e-7)
