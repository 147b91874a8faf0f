"""The binding on a stream that is not the current one: outputs, final states and the
default workspace it allocates belong to the stream the kernels run on, so the
caching allocator cannot hand them to other work while the kernels still use them.
The results equal those of the same call on the current stream."""
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import kda_chunk_fwd, kda_decode_step, kda_recurrent_fwd
from kimi_delta_attention_fwd_gb300 import workloads as W

from parity import to_dev

pytestmark = pytest.mark.gpu


def test_prefill_on_a_side_stream_with_default_workspace():
    x = W.prefill_inputs(W.custom_prefill([700, 90], num_heads=3, d=128, seed=70))
    d = to_dev(x)
    ref_o, ref_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 d["init_state"])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], stream=side)
    # work on the current stream meanwhile: allocations there must not reuse the side
    # stream's blocks while its kernels run
    junk = [torch.full((1 << 20,), 3.0, device="cuda") for _ in range(8)]
    side.synchronize()
    del junk
    assert torch.equal(out, ref_o) and torch.equal(fin, ref_f)


def test_decode_and_recurrent_on_a_side_stream():
    y = W.decode_inputs(W.DecodeSpec(5, 2, 128, 128, 2, "bf16", "std", 71))
    st0 = y["state"].cuda()
    args = [y[n][0].cuda() for n in ("q", "k", "v", "g", "beta")]
    st_ref = st0.clone()
    ref = kda_decode_step(*args, st_ref)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    st = st0.clone()
    torch.cuda.current_stream().synchronize()
    o = kda_decode_step(*args, st, stream=side)
    side.synchronize()
    assert torch.equal(o, ref) and torch.equal(st, st_ref)
    x = W.prefill_inputs(W.custom_prefill([3, 4], num_heads=2, d=128, seed=72))
    d = to_dev(x)
    ro, rf = kda_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                               d["init_state"])
    side.wait_stream(torch.cuda.current_stream())
    o2, f2 = kda_recurrent_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                               d["init_state"], stream=side)
    side.synchronize()
    assert torch.equal(o2, ro) and torch.equal(f2, rf)


def test_segment_scan_on_a_side_stream_with_default_workspace():
    """One long sequence (the segment-parallel scan: seven launches on the call's stream,
    its tables, states and ring in the default workspace) on a side stream: the same bits
    as on the current stream."""
    x = W.prefill_inputs(W.custom_prefill([10007], num_heads=2, d=128, seed=73))
    d = to_dev(x)
    ref_o, ref_f = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                 d["init_state"])
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    out, fin = kda_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                             d["init_state"], stream=side)
    junk = [torch.full((1 << 22,), 3.0, device="cuda") for _ in range(8)]
    side.synchronize()
    del junk
    assert torch.equal(out, ref_o) and torch.equal(fin, ref_f)
