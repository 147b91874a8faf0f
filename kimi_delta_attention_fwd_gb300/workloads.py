"""Seeded synthetic inputs for the KDA forward workloads.

This module is shared by the tests, the benchmark, the smoke check and the
oracle side; it holds none of the KDA arithmetic (no decay, no delta rule, no
chunking), only the input recipe:

  q, k   ~ N(0, 1), then L2-normalised per (token, head) over d_k
  v      ~ N(0, 1)
  g      = log(alpha) = -softplus(N(0, 1)) * 0.1      ("std" gate: alpha in ~(0.9, 1))
         = -softplus(N(-2, 1))                       ("mixed" gate: slow and fast decay)
  beta   = sigmoid(N(0, 1))                           one scalar per (token, head)
  state  ~ N(0, 0.02) (standard deviation 0.02), or zeros

drawn in fp32 from one torch generator per workload in the fixed order
q, k, v, g, beta, state, then rounded (round-to-nearest-even) to the I/O dtype.
Both the CUDA path and the oracle receive the rounded values.

With raw=True the same draws are kept before the two input steps the library can
apply itself (kda_shape.prep): q and k stay N(0, 1) * qk_scale (not normalised)
and beta stays its N(0, 1) logit.  With raw_gate=True g holds the gate logits x
(std: the N(0, 1) draw, mixed: the draw - 2) from which the recipe's log alpha is
-c softplus(x), c = gate_scale(spec) (0.1 std, 1 mixed).

Named workloads (sizes as stated for the KDA forward benchmarks):
  tiny_fp32            1 seq x 256 tokens, H=2, d=64, fp32 I/O, zero state, seed 0
  prefill_bf16         4 seqs x 4096 tokens, H=16, d=128, bf16 I/O, seed 1
  long_prefill_bf16    1 seq x 65536 tokens, H=32, d=128, mixed gate, seed 2
  long_prefill_16k_bf16  1 seq x 16384 tokens, otherwise as long_prefill_bf16: the same
                       32 sequence-heads (and schedule) at a quarter of the tokens, small
                       enough for a full profiler capture
  decode_bf16          256 seqs x H=32, d=128, 128 consecutive single-token steps, seed 3
  varlen_prefill_bf16  64 seqs, lengths ~ U[512, 16384], H=32, d=128, seed 4
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import torch
import torch.nn.functional as F


@dataclasses.dataclass(frozen=True)
class PrefillSpec:
    seqlens: tuple            # tokens of each packed sequence
    num_heads: int
    d_k: int
    d_v: int
    io_dtype: str = "bf16"    # "bf16" or "f32"
    gate: str = "std"         # "std" or "mixed"
    init: str = "normal"      # "normal" (N(0, 0.02)) or "zeros"
    seed: int = 0

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))

    @property
    def num_seqs(self) -> int:
        return len(self.seqlens)


@dataclasses.dataclass(frozen=True)
class DecodeSpec:
    num_seqs: int
    num_heads: int
    d_k: int
    d_v: int
    steps: int
    io_dtype: str = "bf16"
    gate: str = "std"
    seed: int = 3


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    """n sequence lengths uniform on the integers [lo, hi] (seeded, CPU generator)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen))


def named(name: str):
    """The named workloads listed in the module docstring."""
    if name == "tiny_fp32":
        return PrefillSpec((256,), 2, 64, 64, "f32", "std", "zeros", 0)
    if name == "prefill_bf16":
        return PrefillSpec((4096,) * 4, 16, 128, 128, "bf16", "std", "normal", 1)
    if name == "long_prefill_bf16":
        return PrefillSpec((65536,), 32, 128, 128, "bf16", "mixed", "normal", 2)
    if name == "long_prefill_16k_bf16":
        return PrefillSpec((16384,), 32, 128, 128, "bf16", "mixed", "normal", 2)
    if name == "decode_bf16":
        return DecodeSpec(256, 32, 128, 128, 128, "bf16", "std", 3)
    if name == "varlen_prefill_bf16":
        return PrefillSpec(varlen_lengths(64, 512, 16384, 4), 32, 128, 128, "bf16", "std",
                           "normal", 4)
    raise KeyError(name)


NAMES = ("tiny_fp32", "prefill_bf16", "long_prefill_bf16", "long_prefill_16k_bf16",
         "decode_bf16", "varlen_prefill_bf16")


def torch_dtype(io: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[io]


def _gate(shape, kind, gen, device, raw=False):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if kind == "std":
        return x if raw else -F.softplus(x) * 0.1
    if kind == "mixed":
        return x - 2.0 if raw else -F.softplus(x - 2.0)
    raise ValueError(kind)


def gate_scale(spec) -> float:
    """c of the recipe's log alpha = -c softplus(logit) (see raw_gate)."""
    return {"std": 0.1, "mixed": 1.0}[spec.gate]


def _unit_normal(shape, gen, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    return x / x.norm(dim=-1, keepdim=True)


def _qk(shape, gen, device, raw, qk_scale):
    if raw:
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * qk_scale
    return _unit_normal(shape, gen, device)


def _beta(shape, gen, device, raw):
    x = torch.randn(shape, generator=gen, device=device)
    return x if raw else torch.sigmoid(x)


def prefill_inputs(spec: PrefillSpec, device: str = "cpu", raw: bool = False,
                   qk_scale: float = 1.0, raw_gate: bool = False) -> dict:
    """Inputs of one prefill call, laid out as the library expects:
    q, k, g [T, H, d_k]; v [T, H, d_v]; beta [T, H] (all io dtype);
    cu_seqlens int32 [N+1]; init_state fp32 [N, H, d_k, d_v] or None.
    raw=True: q, k and beta before the input steps; raw_gate=True: g as gate logits
    (module docstring)."""
    gen = torch.Generator(device=device).manual_seed(spec.seed)
    T, H, dk, dv = spec.total_tokens, spec.num_heads, spec.d_k, spec.d_v
    dt = torch_dtype(spec.io_dtype)
    q = _qk((T, H, dk), gen, device, raw, qk_scale).to(dt)
    k = _qk((T, H, dk), gen, device, raw, qk_scale).to(dt)
    v = torch.randn((T, H, dv), generator=gen, device=device).to(dt)
    g = _gate((T, H, dk), spec.gate, gen, device, raw_gate).to(dt)
    beta = _beta((T, H), gen, device, raw).to(dt)
    if spec.init == "normal":
        init = torch.randn((spec.num_seqs, H, dk, dv), generator=gen, device=device) * 0.02
    elif spec.init == "zeros":
        init = None
    else:
        raise ValueError(spec.init)
    cu = torch.zeros(spec.num_seqs + 1, dtype=torch.int32)
    if spec.num_seqs:
        cu[1:] = torch.cumsum(torch.tensor(spec.seqlens, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, cu_seqlens=cu.to(device), init_state=init)


def decode_inputs(spec: DecodeSpec, device: str = "cpu", raw: bool = False,
                  qk_scale: float = 1.0, raw_gate: bool = False) -> dict:
    """Inputs of `steps` consecutive decode steps: q, k, g [steps, N, H, d_k];
    v [steps, N, H, d_v]; beta [steps, N, H]; state fp32 [N, H, d_k, d_v].
    raw=True: q, k and beta before the input steps (module docstring)."""
    gen = torch.Generator(device=device).manual_seed(spec.seed)
    S, N, H, dk, dv = spec.steps, spec.num_seqs, spec.num_heads, spec.d_k, spec.d_v
    dt = torch_dtype(spec.io_dtype)
    q = _qk((S, N, H, dk), gen, device, raw, qk_scale).to(dt)
    k = _qk((S, N, H, dk), gen, device, raw, qk_scale).to(dt)
    v = torch.randn((S, N, H, dv), generator=gen, device=device).to(dt)
    g = _gate((S, N, H, dk), spec.gate, gen, device, raw_gate).to(dt)
    beta = _beta((S, N, H), gen, device, raw).to(dt)
    state = torch.randn((N, H, dk, dv), generator=gen, device=device) * 0.02
    return dict(q=q, k=k, v=v, g=g, beta=beta, state=state)


def custom_prefill(seqlens: Sequence[int], num_heads: int, d: int = 128, io: str = "bf16",
                   gate: str = "std", init: str = "normal", seed: int = 0,
                   d_v: Optional[int] = None) -> PrefillSpec:
    return PrefillSpec(tuple(int(x) for x in seqlens), num_heads, d, d_v or d, io, gate, init,
                       seed)
