"""The host decode tool (kimi_delta_attention_fwd_gb300.host_decode): one KDA decode step
on the CPU cores, against the fp64 oracle on the same values, over several steps, in
every gate layout and with the thread count varied.  No GPU."""
import numpy as np
import pytest

import oracle
from kimi_delta_attention_fwd_gb300 import host_decode
from kimi_delta_attention_fwd_gb300 import workloads as W

TOL = 1e-5  # fp32 arithmetic against fp64


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (32, 16)])
def test_decode_steps_match_the_oracle(gate, dk, dv):
    spec = W.DecodeSpec(6, 3, dk, dv, 4, "f32", "mixed", 31)
    y = W.decode_inputs(spec)
    g = y["g"]
    if gate == "scalar":
        g = g[..., 0]
    g_ref = None if gate == "none" else (g if gate == "channel" else
                                         g.unsqueeze(-1).expand(-1, -1, -1, dk))
    if g_ref is None:
        import torch
        g_ref = torch.zeros_like(y["g"])
    ro, rs = oracle.kda_decode_steps(y["q"], y["k"], y["v"], g_ref, y["beta"], y["state"])
    st = y["state"].numpy().copy()
    outs = [host_decode.decode_step(y["q"][t], y["k"][t], y["v"][t],
                                    None if gate == "none" else g[t], y["beta"][t], st)
            for t in range(spec.steps)]
    assert _rel(np.stack(outs), ro) <= TOL
    assert _rel(st, rs) <= TOL


def test_thread_count_does_not_change_the_result():
    y = W.decode_inputs(W.DecodeSpec(7, 5, 64, 64, 1, "f32", "std", 32))
    res = []
    for threads in (1, 2, 3, 64):
        st = y["state"].numpy().copy()
        o = host_decode.decode_step(y["q"][0], y["k"][0], y["v"][0], y["g"][0], y["beta"][0], st,
                                    threads=threads)
        res.append((o, st))
    for o, st in res[1:]:
        assert np.array_equal(o, res[0][0]) and np.array_equal(st, res[0][1])
    assert host_decode.default_threads() >= 1


def test_rejects_bad_arguments():
    st = np.zeros((1, 1, 4, 4), dtype=np.float32)
    with pytest.raises(ValueError):
        host_decode.decode_step(np.zeros((1, 1, 5)), np.zeros((1, 1, 4)), np.zeros((1, 1, 4)),
                                None, np.zeros((1, 1)), st)
    with pytest.raises(TypeError):
        host_decode.decode_step(np.zeros((1, 1, 4)), np.zeros((1, 1, 4)), np.zeros((1, 1, 4)),
                                None, np.zeros((1, 1)), st.astype(np.float64))


def test_the_gpu_library_does_not_link_the_tool():
    """The tool stays outside libkda_gb300.so: none of its symbols are there."""
    import subprocess
    from kimi_delta_attention_fwd_gb300 import build as kbuild
    lib = kbuild.build()
    syms = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True,
                          text=True).stdout
    assert "kda_host_decode" not in syms
