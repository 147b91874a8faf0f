// Internal launcher interface shared by the library's translation units.
// Not part of the public ABI (that is include/kda.h).
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// KDA_PREP_* bits of kda_shape.prep (include/kda.h), for the kernels
constexpr int kPrepSilu = 1, kPrepL2 = 2, kPrepBetaSigmoid = 4;

// Status block at the start of the workspace, written by the prefill kernels.
// word 0: first error code recorded (0 = none), word 1: detail (where).
constexpr size_t kStatusBytes = 256;

struct ChunkArgs {
  int num_seqs, total_tokens, num_heads, d_k, d_v;
  float scale;
  bool bf16;
  const void *q, *k, *v, *g, *beta;
  int gate;           // kda_gate: 0 g per key channel, 1 per (token, head), 2 none (g unused)
  int prep;           // KDA_PREP_* bits: SiLU / L2 norm of q and k, sigmoid of beta
  const float *init_state;
  const int32_t *cu_seqlens;
  void *out;
  float *final_state;
  uint32_t *status;   // device status block (kStatusBytes)
  void *scratch;      // workspace after the status block
  size_t scratch_bytes;
  int num_sms;
  int test_flags;     // bit 0: make the tensor-core kernel time out one wait (test hook)
};

struct DecodeArgs {
  int num_seqs, num_heads, d_k, d_v;
  float scale;
  bool bf16;
  const void *q, *k, *v, *g, *beta;
  int gate;           // kda_gate, as in ChunkArgs
  int prep;           // KDA_PREP_* bits, as in ChunkArgs
  float *state;
  void *out;
};

struct RecurrentArgs {
  int num_seqs, total_tokens, num_heads, d_k, d_v;
  float scale;
  bool bf16;
  const void *q, *k, *v, *g, *beta;
  int gate;                   // kda_gate, as in ChunkArgs
  int prep;                   // KDA_PREP_* bits, as in ChunkArgs
  const float *init_state;    // or NULL (zeros)
  const int32_t *cu_seqlens;  // device [N + 1]
  const int32_t *accepted;    // device [N] or NULL: tokens whose state final_state keeps
  void *out;                  // or NULL
  float *final_state;         // or NULL; may alias init_state
};

// Each returns cudaSuccess or the launch error; a shape the launcher does not
// handle returns cudaErrorInvalidValue without launching.
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
cudaError_t launch_recurrent(const RecurrentArgs &a, cudaStream_t stream);
cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t stream);
cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t stream);
bool chunk_tc_supported(int d_k, int d_v, bool bf16);
// Scratch that lets the tensor-core path run every schedule (0 = none needed).
size_t chunk_tc_scratch_bytes(int num_seqs, int num_heads, int d_k, int d_v);

}  // namespace kda
