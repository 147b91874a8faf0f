"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on the
same seeded inputs and measure the error the way the tolerance is stated
(max over (sequence, head) of ||x - x_ref||_2 / ||x_ref||_2, separately for
the outputs of that head and for its final state)."""
import numpy as np
import torch

import oracle
from kimi_delta_attention_fwd_gb300 import kda_chunk_fwd

TOL_F32 = 1e-4   # fp32 I/O
TOL_BF16 = 2e-2  # bf16 I/O, fp32 state


def rel_l2_per_head(out, ref, cu):
    """out, ref: [T, H, d_v]; returns the max over (seq, head) of the relative L2
    error of that head's outputs (empty sequences skipped)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    cu = np.asarray(cu)
    worst = 0.0
    for n in range(len(cu) - 1):
        a, b = out[cu[n]:cu[n + 1]], ref[cu[n]:cu[n + 1]]
        if a.shape[0] == 0:
            continue
        num = np.sqrt(((a - b) ** 2).sum(axis=(0, 2)))
        den = np.sqrt((b ** 2).sum(axis=(0, 2)))
        worst = max(worst, float((num / np.maximum(den, 1e-300)).max()))
    return worst


def rel_l2_states(st, ref):
    """st, ref: [N, H, d_k, d_v] -> max over (seq, head)."""
    st = np.asarray(st, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if st.size == 0:
        return 0.0
    num = np.sqrt(((st - ref) ** 2).sum(axis=(2, 3)))
    den = np.sqrt((ref ** 2).sum(axis=(2, 3)))
    return float((num / np.maximum(den, 1e-300)).max())


def to_dev(x, dev="cuda"):
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def run_gpu_prefill(x, algo="auto", **kw):
    d = to_dev(x)
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], algo=algo, check=True, **kw)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), (None if fin is None else fin.cpu().numpy())


def run_oracle_prefill(x, **kw):
    return oracle.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["cu_seqlens"],
                          x["init_state"], **kw)
