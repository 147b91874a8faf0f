"""Device-side check of the packed-sequence offsets.

Each kernel that reads cu_seqlens checks a sequence's two offsets before any access
they guide: offsets that decrease or leave [0, T_total] make the kernel skip that
sequence (nothing read or written for it, its final state left as it was) and record
KDA_ERR_SEQLENS, while the valid sequences of the same call are computed as usual.

For safety every tensor here is allocated with room for 256 token rows while the
call declares 128: even a kernel that missed the check would stay inside its buffers.
"""
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import (kda_chunk_fwd, kda_last_device_status,
                                            kda_recurrent_fwd, workspace_status_words)
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import TOL_BF16, TOL_F32, rel_l2_per_head, rel_l2_states, run_oracle_prefill

pytestmark = pytest.mark.gpu

ROWS, T = 256, 128


def _inputs(io, d, seed):
    """256 rows of inputs; the calls below use the first 128 as T_total."""
    spec = W.custom_prefill([ROWS // 4] * 4, num_heads=2, d=d, io=io, seed=seed)
    x = W.prefill_inputs(spec)
    return {kk: (vv.cuda() if isinstance(vv, torch.Tensor) else vv) for kk, vv in x.items()}, x


BAD = {
    "decreasing": [0, 64, 40, 40],    # sequence 1 = [64, 40); sequence 2 empty
    "beyond_end": [0, 64, 200, 128],  # sequence 1 = [64, 200) passes T_total = 128, 2 = [200, 128)
    "negative": [0, -8, 64, 128],     # sequences 0 = [0, -8) and 1 = [-8, 64); 2 = [64, 128) valid
}


def _valid(cu, n):
    return 0 <= cu[n] <= cu[n + 1] <= T


def _check_sequences(x, cu, out, fin, tol):
    """Skipped sequences keep their final state; valid ones match the oracle run on
    them alone."""
    for n in range(len(cu) - 1):
        lo, hi = cu[n], cu[n + 1]
        if not _valid(cu, n):
            assert torch.equal(fin[n], torch.full_like(fin[n], 7.0))
            continue
        xs = {"q": x["q"][lo:hi], "k": x["k"][lo:hi], "v": x["v"][lo:hi], "g": x["g"][lo:hi],
              "beta": x["beta"][lo:hi], "cu_seqlens": torch.tensor([0, hi - lo], dtype=torch.int32),
              "init_state": x["init_state"][n:n + 1]}
        ro, rs = run_oracle_prefill(xs)
        if hi > lo:
            assert rel_l2_per_head(out[lo:hi].float().cpu().numpy(), ro,
                                   xs["cu_seqlens"].numpy()) <= tol
        assert rel_l2_states(fin[n:n + 1].cpu().numpy(), rs) <= tol


def _views(d):
    """The tensors as the call sees them: T = 128 declared rows of 256 allocated."""
    return {kk: (vv[:T] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in d.items()}


@pytest.mark.parametrize("bad", list(BAD))
@pytest.mark.parametrize("io,d,algo", [("bf16", 128, "tensor"), ("bf16", 128, "simt"),
                                        ("f32", 64, "simt")])
def test_prefill_skips_and_reports_bad_offsets(bad, io, d, algo):
    dd, x = _inputs(io, d, seed=60)
    cu = torch.tensor(BAD[bad], dtype=torch.int32, device="cuda")
    v = _views(dd)
    init = dd["init_state"][:3].contiguous()
    fin = torch.full_like(init, 7.0)
    out = torch.full((ROWS, 2, d), 5.0, dtype=dd["q"].dtype, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    kda_chunk_fwd(v["q"], v["k"], v["v"], v["g"], v["beta"], cu, init, out=out[:T], final_state=fin,
                  workspace=ws, algo=algo)
    words = workspace_status_words(ws)
    assert words[0] == 11, words  # KDA_ERR_SEQLENS
    assert torch.equal(out[T:], torch.full_like(out[T:], 5.0))  # nothing past T_total written
    _check_sequences(x, BAD[bad], out, fin, TOL_F32 if io == "f32" else TOL_BF16)


@pytest.mark.parametrize("bad", list(BAD))
def test_recurrent_skips_and_reports_bad_offsets(bad):
    dd, x = _inputs("bf16", 128, seed=61)
    kda_last_device_status()  # start from a clear word
    cu = torch.tensor(BAD[bad], dtype=torch.int32, device="cuda")
    v = _views(dd)
    init = dd["init_state"][:3].contiguous()
    fin = torch.full_like(init, 7.0)
    out = torch.full((ROWS, 2, 128), 5.0, dtype=dd["q"].dtype, device="cuda")
    kda_recurrent_fwd(v["q"], v["k"], v["v"], v["g"], v["beta"], cu, init, out=out[:T],
                      final_state=fin)
    assert kda_last_device_status() == -11
    assert kda_last_device_status() == 0  # read and cleared
    assert torch.equal(out[T:], torch.full_like(out[T:], 5.0))
    _check_sequences(x, BAD[bad], out, fin, TOL_BF16)


def test_valid_offsets_leave_the_status_clear():
    dd, x = _inputs("bf16", 128, seed=62)
    cu = torch.tensor([0, 30, 128], dtype=torch.int32, device="cuda")
    v = _views(dd)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    kda_chunk_fwd(v["q"], v["k"], v["v"], v["g"], v["beta"], cu, dd["init_state"][:2].contiguous(),
                  workspace=ws)
    assert workspace_status_words(ws)[0] == 0
    kda_recurrent_fwd(v["q"], v["k"], v["v"], v["g"], v["beta"], cu, dd["init_state"][:2].contiguous())
    assert kda_last_device_status() == 0
