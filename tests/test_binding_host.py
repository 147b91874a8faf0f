"""Host-side checks of the Python binding (no GPU): every entry point refuses
tensors that are not on a CUDA device, or have the wrong rank, before anything
reaches the C ABI (a host pointer there would reach the kernels), and the
metadata checks name what is wrong.  No compute call is made."""
import pytest
import torch

from kimi_delta_attention_fwd_gb300 import kda
from kimi_delta_attention_fwd_gb300 import (kda_chunk_fwd, kda_decode_step, kda_recurrent_fwd,
                                            kda_workspace_status)

T, H, D, N = 10, 2, 64, 2


def _prefill_args(dtype=torch.float32):
    z = lambda *s: torch.zeros(*s, dtype=dtype)
    cu = torch.tensor([0, 4, T], dtype=torch.int32)
    return z(T, H, D), z(T, H, D), z(T, H, D), z(T, H, D), z(T, H), cu


def test_cpu_tensors_are_refused_by_every_entry_point():
    q, k, v, g, b, cu = _prefill_args()
    with pytest.raises(ValueError, match="CUDA tensors only"):
        kda_chunk_fwd(q, k, v, g, b, cu)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        kda_recurrent_fwd(q, k, v, g, b, cu)
    st = torch.zeros(N, H, D, D)
    with pytest.raises(ValueError, match="CUDA tensors only"):
        kda_decode_step(q[:N], k[:N], v[:N], g[:N], b[:N], st)
    with pytest.raises(ValueError, match="CUDA workspace only"):
        kda_workspace_status(torch.zeros(256, dtype=torch.uint8))


@pytest.mark.parametrize("which", ["q", "v", "g", "beta", "cu_seqlens"])
def test_wrong_rank_is_named_before_anything_else(which):
    q, k, v, g, b, cu = _prefill_args()
    args = dict(q=q, k=k, v=v, g=g, beta=b, cu_seqlens=cu)
    args[which] = args[which].reshape(-1)  # rank 1 (cu_seqlens: rank 2 below)
    if which == "cu_seqlens":
        args[which] = cu.reshape(1, -1)
    for fn in (kda_chunk_fwd, kda_recurrent_fwd):
        with pytest.raises(ValueError, match=f"{which} has"):
            fn(args["q"], args["k"], args["v"], args["g"], args["beta"], args["cu_seqlens"])


def test_decode_state_rank_is_checked():
    q, k, v, g, b, _ = _prefill_args()
    with pytest.raises(ValueError, match="state has 3 dimensions"):
        kda_decode_step(q[:N], k[:N], v[:N], g[:N], b[:N], torch.zeros(N, H, D * D))


def test_gate_layouts_map_to_the_abi():
    g3, g2 = torch.zeros(T, H, D), torch.zeros(T, H)
    assert kda._gate_of(g3, T, H, D) == (kda.KDA_GATE_CHANNEL, (T, H, D))
    assert kda._gate_of(g2, T, H, D) == (kda.KDA_GATE_SCALAR, (T, H))
    assert kda._gate_of(None, T, H, D) == (kda.KDA_GATE_NONE, None)


def test_input_step_bits():
    assert kda._prep_bits(False, False, False) == 0
    assert kda._prep_bits(True, False, False) == kda.KDA_PREP_QK_SILU == 1
    assert kda._prep_bits(False, True, False) == kda.KDA_PREP_QK_L2NORM == 2
    assert kda._prep_bits(False, False, True) == kda.KDA_PREP_BETA_SIGMOID == 4
    assert kda._prep_bits(True, True, True) == 7


def test_shape_struct_fields():
    s = kda._make_shape(3, 100, 4, 128, 64, None, kda.KDA_BF16, "tensor", kda.KDA_GATE_SCALAR, 5)
    assert (s.num_seqs, s.total_tokens, s.num_heads, s.d_k, s.d_v, s.chunk_size) == (3, 100, 4, 128, 64, 64)
    assert s.scale == 0.0  # the library's d_k^-1/2
    assert (s.io_dtype, s.algo, s.gate, s.prep) == (kda.KDA_BF16, 1, kda.KDA_GATE_SCALAR, 5)
    assert kda._make_shape(1, 1, 1, 64, 64, 0.5, kda.KDA_F32).scale == 0.5


def test_metadata_checks_name_the_problem():
    cpu = torch.device("cpu")
    x = torch.zeros(T, H, D)
    kda._check_io("x", x, (T, H, D), torch.float32, cpu)
    with pytest.raises(TypeError, match="x: dtype"):
        kda._check_io("x", x.to(torch.bfloat16), (T, H, D), torch.float32, cpu)
    with pytest.raises(ValueError, match="x: shape"):
        kda._check_io("x", x, (T, H, D + 1), torch.float32, cpu)
    with pytest.raises(ValueError, match="contiguous"):
        kda._check_io("x", x.transpose(0, 1), (H, T, D), torch.float32, cpu)
    with pytest.raises(ValueError, match="is on cpu"):
        kda._check_io("x", x, (T, H, D), torch.float32, torch.device("cuda", 0))


def test_workspace_checks():
    ws = torch.zeros(512, dtype=torch.uint8)
    kda._check_workspace(ws, torch.device("cpu"))
    with pytest.raises(ValueError, match="workspace is on cpu"):
        kda._check_workspace(ws, torch.device("cuda", 0))
    with pytest.raises(ValueError, match="contiguous"):
        kda._check_workspace(ws[::2], torch.device("cpu"))


def test_sequence_offsets_check():
    ok = torch.tensor([0, 0, 3, 7, 7], dtype=torch.int32)
    kda._check_cu_seqlens(ok, 7)
    kda._check_cu_seqlens(ok, 9)  # trailing tokens belong to no sequence
    kda._check_cu_seqlens(torch.tensor([0], dtype=torch.int32), 0)
    with pytest.raises(ValueError, match="start at 0"):
        kda._check_cu_seqlens(torch.tensor([1, 3], dtype=torch.int32), 3)
    with pytest.raises(ValueError, match="nondecreasing"):
        kda._check_cu_seqlens(torch.tensor([0, 5, 4], dtype=torch.int32), 5)
    with pytest.raises(ValueError, match="beyond the 6 tokens"):
        kda._check_cu_seqlens(torch.tensor([0, 3, 7], dtype=torch.int32), 6)
