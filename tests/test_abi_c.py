"""include/kda.h as a C header: a plain C program includes it, links against
libkda_gb300.so and calls the entry points.  Without a GPU (or with bad arguments) the
calls return their documented error codes, and nothing needs C++ or torch."""
import os
import shutil
import subprocess

import pytest

from kimi_delta_attention_fwd_gb300 import build as kbuild

C_SRC = r"""
#include <stdio.h>
#include "kda.h"

int main(void) {
  kda_shape s = {2, 128, 4, 128, 128, 64, 0.0f, KDA_BF16, KDA_ALGO_AUTO, KDA_GATE_CHANNEL, 0,
                 0.0f};
  if (kda_version() < 1004) return 10;
  size_t ws = kda_chunk_fwd_workspace_bytes(&s);
  if (ws < 256) return 11;
  if (kda_chunk_fwd_selected_algo(&s) != KDA_ALGO_TENSOR) return 12;
  kda_shape bad = s;
  bad.d_k = 96;
  if (kda_chunk_fwd_workspace_bytes(&bad) != 0) return 13;
  if (kda_chunk_fwd(&bad, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0) != KDA_ERR_SHAPE) return 14;
  if (kda_chunk_fwd(NULL, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0) != KDA_ERR_NULL) return 15;
  bad = s;
  bad.prep = 16;
  if (kda_decode_step(&bad, 0, 0, 0, 0, 0, 0, 0, 0) != KDA_ERR_SHAPE) return 16;
  bad = s;
  bad.gate_scale = 1.0f / 0.0f;
  if (kda_chunk_fwd_workspace_bytes(&bad) != 0) return 18;
  bad = s;
  bad.prep = KDA_PREP_G_SOFTPLUS;
  bad.gate_scale = 0.1f;
  if (kda_chunk_fwd_workspace_bytes(&bad) < 256) return 19;
  if (kda_workspace_status(NULL, 0) != KDA_ERR_NULL) return 17;
  printf("%s\n", kda_status_string(KDA_ERR_GATE_RANGE));
  return 0;
}
"""


def test_header_compiles_and_links_as_c(tmp_path):
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    lib = kbuild.build()
    src = tmp_path / "use_kda.c"
    src.write_text(C_SRC)
    exe = tmp_path / "use_kda"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", kbuild.INCLUDE, "-I", cuda_inc,
                    str(src), "-o", str(exe), lib, "-Wl,-rpath," + os.path.dirname(lib)],
                   check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, (res.returncode, res.stdout, res.stderr)
    assert "decay" in res.stdout
