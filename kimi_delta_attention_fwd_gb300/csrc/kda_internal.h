// Internal launcher interface shared by the library's translation units.
// Not part of the public ABI (that is include/kda.h).
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

// KDA_PREP_* bits of kda_shape.prep (include/kda.h), for the kernels
constexpr int kPrepSilu = 1, kPrepL2 = 2, kPrepBetaSigmoid = 4, kPrepGSoftplus = 8;

// Status block at the start of the workspace, written by the prefill kernels.
// word 0: first error code recorded (0 = none, else minus a KDA_ERR_* code),
// word 1: detail (where), word 2: the schedule the tensor-core kernel ran
// (kSchedPlain or kSchedHelpers), word 3: sequence-heads recomputed token by token
// because a chunk's decay left the tensor-core range.
constexpr size_t kStatusBytes = 256;
constexpr uint32_t kSchedPlain = 1, kSchedHelpers = 2, kSchedSegments = 3;
// device-reported codes (minus the KDA_ERR_* value)
constexpr uint32_t kStatusTimeout = 7, kStatusGateRange = 8, kStatusSeqlens = 11;

#ifdef __CUDACC__
// log alpha from a gate logit x (KDA_PREP_G_SOFTPLUS): -c softplus(x), with
// softplus(x) = max(x, 0) + log(1 + e^-|x|) (no overflow for large |x|)
__device__ __forceinline__ float neg_softplus(float x, float c) {
  return -c * (fmaxf(x, 0.f) + log1pf(__expf(-fabsf(x))));
}
// The log decay a kernel uses for a g value: the value itself, or -c softplus(x)
// when the gate step is on (kPrep instantiations only).
template <bool kPrep>
__device__ __forceinline__ float gate_log(float x, int prep, float c) {
  return (kPrep && (prep & kPrepGSoftplus)) ? neg_softplus(x, c) : x;
}

// Sequence n's tokens [bos, eos) from the packed offsets, checked on the device before
// any access they guide: offsets that decrease or leave [0, T] give an empty range,
// record kStatusSeqlens in *status (when given) and return false.
__device__ __forceinline__ bool seq_range(const int32_t *cu, int n, int T, uint32_t *status,
                                          int &bos, int &eos) {
  const int b = cu[n], e = cu[n + 1];
  if (0 <= b && b <= e && e <= T) {
    bos = b;
    eos = e;
    return true;
  }
  bos = eos = 0;
  if (status) atomicCAS(status, 0u, kStatusSeqlens);
  return false;
}
#endif

struct ChunkArgs {
  int num_seqs, total_tokens, num_heads, d_k, d_v;
  float scale;
  bool bf16;
  const void *q, *k, *v, *g, *beta;
  int gate;           // kda_gate: 0 g per key channel, 1 per (token, head), 2 none (g unused)
  int prep;           // KDA_PREP_* bits: SiLU / L2 norm of q and k, sigmoid of beta, softplus gate
  float gate_scale;   // c of log alpha = -c softplus(x) (KDA_PREP_G_SOFTPLUS)
  const float *init_state;
  const int32_t *cu_seqlens;
  void *out;
  float *final_state;
  uint32_t *status;   // device status block (kStatusBytes)
  uint32_t *pair_flags;  // [N * H] zeroed words for pairs to recompute exactly, or NULL
  void *scratch;      // workspace after the status block (and the flags)
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
  float gate_scale;   // as in ChunkArgs
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
  float gate_scale;           // as in ChunkArgs
  const float *init_state;    // or NULL (zeros)
  const int32_t *cu_seqlens;  // device [N + 1]
  const int32_t *accepted;    // device [N] or NULL: tokens whose state final_state keeps
  void *out;                  // or NULL
  float *final_state;         // or NULL; may alias init_state
  uint32_t *status;           // device word for errors, or NULL (the library's own word)
  const uint32_t *only_flags; // device [N * H] or NULL: run only the pairs whose flag is set
  const uint32_t *only_count; // device word or NULL: nothing runs while it is 0
};

// Each returns cudaSuccess or the launch error; a shape the launcher does not
// handle returns cudaErrorInvalidValue without launching.
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);
cudaError_t launch_recurrent(const RecurrentArgs &a, cudaStream_t stream);
// Reads (after synchronising `stream`) and clears the device status word that the
// recurrent kernels of this library record on the current device.
cudaError_t take_device_status(uint32_t *word, cudaStream_t stream);
cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t stream);
cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t stream);
bool chunk_tc_supported(int d_k, int d_v, bool bf16);
// Scratch that lets the tensor-core path run every schedule (0 = none needed).
size_t chunk_tc_scratch_bytes(int num_seqs, int total_tokens, int num_heads, int d_k, int d_v);

}  // namespace kda
