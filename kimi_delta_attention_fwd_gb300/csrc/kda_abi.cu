// extern "C" entry points of the KDA forward library: argument validation,
// kernel selection, status handling.  See include/kda.h for the contract.
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kda.h"
#include "kda_internal.h"

namespace {

bool aligned(const void *p, uintptr_t bytes) {
  return p == nullptr || (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}
bool aligned16(const void *p) { return aligned(p, 16); }

// Common shape checks; `decode` relaxes the chunk/algo fields.
int check_shape(const kda_shape *s, bool decode) {
  if (!s) return KDA_ERR_NULL;
  if (s->num_seqs < 0 || s->total_tokens < 0 || s->num_heads < 1) return KDA_ERR_SHAPE;
  if (!((s->d_k == 64 || s->d_k == 128) && (s->d_v == 64 || s->d_v == 128))) return KDA_ERR_SHAPE;
  if (s->io_dtype != KDA_F32 && s->io_dtype != KDA_BF16) return KDA_ERR_SHAPE;
  if (!(s->scale == s->scale) || isinf(s->scale)) return KDA_ERR_SHAPE;
  if (s->gate < KDA_GATE_CHANNEL || s->gate > KDA_GATE_NONE) return KDA_ERR_SHAPE;
  if (s->prep & ~(KDA_PREP_QK_SILU | KDA_PREP_QK_L2NORM | KDA_PREP_BETA_SIGMOID | KDA_PREP_G_SOFTPLUS))
    return KDA_ERR_SHAPE;
  if (!(s->gate_scale == s->gate_scale) || isinf(s->gate_scale)) return KDA_ERR_SHAPE;
  if (decode) {
    if (s->total_tokens != s->num_seqs) return KDA_ERR_SHAPE;
  } else {
    if (s->chunk_size != 0 && s->chunk_size != 64) return KDA_ERR_SHAPE;
    if (s->algo < KDA_ALGO_AUTO || s->algo > KDA_ALGO_SIMT) return KDA_ERR_SHAPE;
  }
  // element counts must stay addressable with 64-bit offsets and 32-bit token ids
  if ((int64_t)s->num_seqs * s->num_heads > (int64_t)INT32_MAX) return KDA_ERR_SHAPE;
  return KDA_OK;
}

float effective_scale(const kda_shape *s) {
  return s->scale > 0.f ? s->scale : 1.0f / sqrtf((float)s->d_k);
}
float effective_gate_scale(const kda_shape *s) { return s->gate_scale > 0.f ? s->gate_scale : 1.0f; }

// The library carries sm_103a code only.
int check_device(int *num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_DEVICE;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_DEVICE;
  if (major != 10 || minor != 3) return KDA_ERR_DEVICE;
  if (num_sms) *num_sms = sms;
  return KDA_OK;
}

bool use_tensor_path(const kda_shape *s) {
  const bool bf16 = s->io_dtype == KDA_BF16;
  if (s->algo == KDA_ALGO_SIMT) return false;
  if (s->algo == KDA_ALGO_TENSOR) return true;
  return kda::chunk_tc_supported(s->d_k, s->d_v, bf16);
}

// Per-pair flags after the status block: the tensor-core path marks there the
// sequence-heads whose decay left its range, which a second kernel then recomputes
// token by token.  Without a gate there is no decay and no flag.
size_t flag_bytes(const kda_shape *s) {
  if (!use_tensor_path(s) || s->gate == KDA_GATE_NONE) return 0;
  const size_t pairs = (size_t)s->num_seqs * (size_t)s->num_heads;
  return (pairs * sizeof(uint32_t) + 255) / 256 * 256;
}

}  // namespace

namespace kda {
// The workspace a call needs to give the same results as with
// kda_chunk_fwd_workspace_bytes(): the status block and the recomputation flags
// (the helpers' ring only speeds a call up).  0 for an invalid shape.
size_t chunk_fwd_required_workspace(const kda_shape *s) {
  if (check_shape(s, false) != KDA_OK) return 0;
  return kStatusBytes + flag_bytes(s);
}
}  // namespace kda

extern "C" {

// 1.1: kda_recurrent_fwd; 1.2: kda_shape.prep; 1.3: device-checked offsets
// (KDA_ERR_SEQLENS, kda_last_device_status), the exact recomputation of sequence-heads
// beyond the tensor-core decay range, kda_noalloc_status; 1.4: KDA_PREP_G_SOFTPLUS and
// kda_shape.gate_scale; 1.5: the segment-parallel scan of one sequence
int kda_version(void) { return 1005; }

const char *kda_status_string(int status) {
  switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL: return "a required pointer is NULL";
    case KDA_ERR_SHAPE: return "unsupported or inconsistent sizes";
    case KDA_ERR_ALIGN: return "a pointer is not aligned as the ABI requires";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_LAUNCH: return "CUDA rejected a launch or an asynchronous call";
    case KDA_ERR_DEVICE: return "current device is not sm_103 or lacks a needed driver entry point";
    case KDA_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel gave up";
    case KDA_ERR_GATE_RANGE: return "a chunk's cumulative decay exceeded the tensor-core path's range";
    case KDA_ERR_UNSUPPORTED: return "the requested algorithm does not support this dtype or size";
    case KDA_ERR_NOALLOC_LIMIT: return "the shape needs more scratch than the built-in no-allocation buffer";
    case KDA_ERR_SEQLENS: return "cu_seqlens offsets decrease or leave [0, total_tokens] (found on the device)";
    default: return "unknown status";
  }
}

size_t kda_chunk_fwd_workspace_bytes(const kda_shape *s) {
  if (check_shape(s, false) != KDA_OK) return 0;
  size_t bytes = kda::kStatusBytes + flag_bytes(s);
  if (use_tensor_path(s))
    bytes += kda::chunk_tc_scratch_bytes(s->num_seqs, s->total_tokens, s->num_heads, s->d_k, s->d_v);
  return bytes;
}

int kda_chunk_fwd_selected_algo(const kda_shape *s) {
  const int rc = check_shape(s, false);
  if (rc != KDA_OK) return rc;
  if (!use_tensor_path(s)) return KDA_ALGO_SIMT;
  if (!kda::chunk_tc_supported(s->d_k, s->d_v, s->io_dtype == KDA_BF16)) return KDA_ERR_UNSUPPORTED;
  return KDA_ALGO_TENSOR;
}

int kda_chunk_fwd(const kda_shape *s, const void *q, const void *k, const void *v, const void *g,
                  const void *beta, const float *init_state, const int32_t *cu_seqlens, void *out,
                  float *final_state, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  int rc = check_shape(s, false);
  if (rc != KDA_OK) return rc;
  const bool need_g = s->gate != KDA_GATE_NONE;
  if (!need_g) g = nullptr;  // not read
  if (s->total_tokens > 0 && (!q || !k || !v || (need_g && !g) || !beta || !out)) return KDA_ERR_NULL;
  if (s->num_seqs > 0 && !cu_seqlens) return KDA_ERR_NULL;
  if (!workspace) return KDA_ERR_WORKSPACE;
  if (workspace_bytes < kda::kStatusBytes) return KDA_ERR_WORKSPACE;  // the schedule fits the rest
  const uintptr_t esz = s->io_dtype == KDA_BF16 ? 2 : 4;
  const bool g_ok = s->gate == KDA_GATE_CHANNEL ? aligned16(g) : aligned(g, esz);
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !g_ok || !aligned(beta, esz) ||
      !aligned16(init_state) || !aligned(cu_seqlens, 4) || !aligned16(out) ||
      !aligned16(final_state) || !aligned16(workspace))
    return KDA_ERR_ALIGN;
  const bool tensor = use_tensor_path(s);
  if (tensor && !kda::chunk_tc_supported(s->d_k, s->d_v, s->io_dtype == KDA_BF16))
    return KDA_ERR_UNSUPPORTED;
  int num_sms = 0;
  rc = check_device(&num_sms);
  if (rc != KDA_OK) return rc;

  // the flags of the exact recomputation, when the workspace has room for them
  const size_t fbytes = flag_bytes(s);
  const bool flags = fbytes > 0 && workspace_bytes >= kda::kStatusBytes + fbytes;
  const size_t head = kda::kStatusBytes + (flags ? fbytes : 0);
  if (cudaMemsetAsync(workspace, 0, head, stream) != cudaSuccess) return KDA_ERR_LAUNCH;
  if (s->num_seqs == 0) return KDA_OK;

  kda::ChunkArgs a;
  a.num_seqs = s->num_seqs;
  a.total_tokens = s->total_tokens;
  a.num_heads = s->num_heads;
  a.d_k = s->d_k;
  a.d_v = s->d_v;
  a.scale = effective_scale(s);
  a.bf16 = s->io_dtype == KDA_BF16;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.gate = s->gate;
  a.prep = s->prep;
  a.gate_scale = effective_gate_scale(s);
  a.init_state = init_state;
  a.cu_seqlens = cu_seqlens;
  a.out = out;
  a.final_state = final_state;
  a.status = static_cast<uint32_t *>(workspace);
  a.pair_flags = flags ? reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(workspace) +
                                                      kda::kStatusBytes)
                       : nullptr;
  a.scratch = static_cast<unsigned char *>(workspace) + head;
  a.scratch_bytes = workspace_bytes - head;
  a.num_sms = num_sms;
  // Test hook: KDA_TEST_FORCE_WAIT_TIMEOUT=1 makes the tensor-core kernel wait once on a
  // barrier that nothing arrives on, so its bounded-wait error path can be exercised.
  const char *force = getenv("KDA_TEST_FORCE_WAIT_TIMEOUT");
  a.test_flags = (force && force[0] == '1') ? 1 : 0;
  cudaError_t err = tensor ? kda::launch_chunk_tc(a, stream) : kda::launch_chunk_simt(a, stream);
  if (err == cudaErrorInvalidValue) return KDA_ERR_UNSUPPORTED;
  if (err != cudaSuccess) return KDA_ERR_LAUNCH;
  if (a.pair_flags) {
    // The sequence-heads the tensor-core kernel marked (a chunk's decay beyond its range)
    // are recomputed token by token with exact decays; the kernel leaves at once when
    // none was marked (status word 3 counts them).
    kda::RecurrentArgs r;
    r.num_seqs = a.num_seqs;
    r.total_tokens = a.total_tokens;
    r.num_heads = a.num_heads;
    r.d_k = a.d_k;
    r.d_v = a.d_v;
    r.scale = a.scale;
    r.bf16 = a.bf16;
    r.q = q; r.k = k; r.v = v; r.g = g; r.beta = beta;
    r.gate = a.gate;
    r.prep = a.prep;
    r.gate_scale = a.gate_scale;
    r.init_state = init_state;
    r.cu_seqlens = cu_seqlens;
    r.accepted = nullptr;
    r.out = out;
    r.final_state = final_state;
    r.status = a.status;
    r.only_flags = a.pair_flags;
    r.only_count = a.status + 3;
    err = kda::launch_recurrent(r, stream);
    if (err != cudaSuccess) return KDA_ERR_LAUNCH;
  }
  return KDA_OK;
}

int kda_recurrent_fwd(const kda_shape *s, const void *q, const void *k, const void *v,
                      const void *g, const void *beta, const float *init_state,
                      const int32_t *cu_seqlens, const int32_t *accepted, void *out,
                      float *final_state, cudaStream_t stream) {
  int rc = check_shape(s, false);
  if (rc != KDA_OK) return rc;
  const bool need_g = s->gate != KDA_GATE_NONE;
  if (!need_g) g = nullptr;  // not read
  if (!out && !final_state) return KDA_OK;  // nothing to produce
  if (s->total_tokens > 0 && (!q || !k || !v || (need_g && !g) || !beta)) return KDA_ERR_NULL;
  if (s->num_seqs > 0 && !cu_seqlens) return KDA_ERR_NULL;
  const uintptr_t esz = s->io_dtype == KDA_BF16 ? 2 : 4;
  if (!aligned(q, esz) || !aligned(k, esz) || !aligned(v, esz) || !aligned(g, esz) ||
      !aligned(beta, esz) || !aligned16(init_state) || !aligned(cu_seqlens, 4) ||
      !aligned(accepted, 4) || !aligned(out, 4 * esz) || !aligned16(final_state))
    return KDA_ERR_ALIGN;
  rc = check_device(nullptr);
  if (rc != KDA_OK) return rc;
  if (s->num_seqs == 0) return KDA_OK;
  kda::RecurrentArgs a;
  a.num_seqs = s->num_seqs;
  a.total_tokens = s->total_tokens;
  a.num_heads = s->num_heads;
  a.d_k = s->d_k;
  a.d_v = s->d_v;
  a.scale = effective_scale(s);
  a.bf16 = s->io_dtype == KDA_BF16;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.gate = s->gate;
  a.prep = s->prep;
  a.gate_scale = effective_gate_scale(s);
  a.init_state = init_state;
  a.cu_seqlens = cu_seqlens;
  a.accepted = accepted;
  a.out = out;
  a.final_state = final_state;
  a.status = nullptr;  // offsets found out of range go to the library's device word
  a.only_flags = nullptr;
  a.only_count = nullptr;
  const cudaError_t err = kda::launch_recurrent(a, stream);
  return err == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

int kda_decode_step(const kda_shape *s, const void *q, const void *k, const void *v, const void *g,
                    const void *beta, float *state, void *out, cudaStream_t stream) {
  int rc = check_shape(s, true);
  if (rc != KDA_OK) return rc;
  if (s->num_seqs == 0) return KDA_OK;
  if (s->gate == KDA_GATE_NONE) g = nullptr;  // not read
  if (!q || !k || !v || (s->gate != KDA_GATE_NONE && !g) || !beta || !state || !out)
    return KDA_ERR_NULL;
  const uintptr_t esz = s->io_dtype == KDA_BF16 ? 2 : 4;
  if (!aligned(q, esz) || !aligned(k, esz) || !aligned(v, esz) || !aligned(g, esz) ||
      !aligned(beta, esz) || !aligned16(state) || !aligned(out, 4 * esz))
    return KDA_ERR_ALIGN;
  rc = check_device(nullptr);
  if (rc != KDA_OK) return rc;
  kda::DecodeArgs a;
  a.num_seqs = s->num_seqs;
  a.num_heads = s->num_heads;
  a.d_k = s->d_k;
  a.d_v = s->d_v;
  a.scale = effective_scale(s);
  a.bf16 = s->io_dtype == KDA_BF16;
  a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta;
  a.gate = s->gate;
  a.prep = s->prep;
  a.gate_scale = effective_gate_scale(s);
  a.state = state;
  a.out = out;
  const cudaError_t err = kda::launch_decode(a, stream);
  return err == cudaSuccess ? KDA_OK : KDA_ERR_LAUNCH;
}

int kda_last_device_status(cudaStream_t stream) {
  uint32_t word = 0;
  if (kda::take_device_status(&word, stream) != cudaSuccess) return KDA_ERR_LAUNCH;
  return word == 0 ? KDA_OK : -(int)word;
}

int kda_workspace_status(const void *workspace, cudaStream_t stream) {
  if (!workspace) return KDA_ERR_NULL;
  uint32_t word[2] = {0, 0};
  if (cudaMemcpyAsync(word, workspace, sizeof(word), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return KDA_ERR_LAUNCH;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KDA_ERR_LAUNCH;
  return word[0] == 0 ? KDA_OK : -(int)word[0];
}

}  // extern "C"
