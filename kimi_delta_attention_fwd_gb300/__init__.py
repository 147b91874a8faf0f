"""GB300 (sm_103a) Kimi Delta Attention forward: chunkwise prefill over packed
variable-length sequences and the single-token decode step, as hand-written
CUDA kernels behind the C ABI of include/kda.h.

Importing the package loads nothing; the CUDA library is opened on the first
call (and a missing library raises).
"""
from .kda import (KdaError, kda_chunk_fwd, kda_chunk_fwd_selected_algo,
                  kda_chunk_fwd_workspace_bytes, kda_decode_step, kda_last_device_status,
                  kda_recurrent_fwd, kda_status_string, kda_version, kda_workspace_status,
                  load_library, workspace_status_words)

__all__ = ["KdaError", "kda_chunk_fwd", "kda_chunk_fwd_selected_algo",
           "kda_chunk_fwd_workspace_bytes", "kda_decode_step", "kda_last_device_status",
           "kda_recurrent_fwd", "kda_status_string", "kda_version", "kda_workspace_status",
           "load_library", "workspace_status_words"]
