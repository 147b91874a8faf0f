/*
 * kda_host_decode.h -- C interface of the host (CPU) decode tool.
 *
 * A separate tool beside the GPU library (include/kda.h): it takes host buffers,
 * runs on the CPU cores, and shares no code with the GPU path.
 *
 * kda_host_decode_step: one recurrent step for N independent sequences, one token
 * each ("Kimi Delta Attention (KDA)", the five-line recurrence):
 *   alpha = exp(g),  S~ = Diag(alpha) S,  e = beta (v - S~^T k),  S <- S~ + k e^T,
 *   o = scale * S^T q
 *   q, k : [N, H, d_k] fp32    v, out : [N, H, d_v] fp32    beta : [N, H] fp32
 *   g    : [N, H, d_k] (KDA_HOST_GATE_CHANNEL), [N, H] (SCALAR: one log alpha for
 *          every key channel) or NULL (NONE: alpha = 1); g <= 0
 *   state: [N, H, d_k, d_v] fp32, updated in place
 *   scale <= 0 selects d_k^-1/2; threads < 1 selects one per online core.
 * All pointers are host pointers owned by the caller.  Returns 0 or a negative code.
 */
#ifndef KDA_HOST_DECODE_H_
#define KDA_HOST_DECODE_H_

#ifdef __cplusplus
extern "C" {
#endif

enum {
  KDA_HOST_OK = 0,
  KDA_HOST_ERR_NULL = -1,
  KDA_HOST_ERR_SHAPE = -2,
  KDA_HOST_ERR_MEMORY = -3,
  KDA_HOST_ERR_THREAD = -4
};
enum { KDA_HOST_GATE_CHANNEL = 0, KDA_HOST_GATE_SCALAR = 1, KDA_HOST_GATE_NONE = 2 };

int kda_host_decode_step(int num_seqs, int num_heads, int d_k, int d_v, float scale, int gate,
                         const float *q, const float *k, const float *v, const float *g,
                         const float *beta, float *state, float *out, int threads);

/* Threads kda_host_decode_step uses by default: one per online core. */
int kda_host_decode_default_threads(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_HOST_DECODE_H_ */
