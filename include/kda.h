/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention forward library.
 *
 * The operation ("Kimi Delta Attention (KDA)", brain.bigb.es, opening equation
 * and the five-line recurrence in the transposed d_k x d_v layout; "K3 架构图解"
 * Ch.08 column-vector form).  Per sequence and head, state S in R^{d_k x d_v}:
 *
 *   alpha_t = exp(g_t)                 (g_t = log alpha_t <= 0, one per key channel;
 *                                       see kda_gate for the one-per-token form of
 *                                       Gated DeltaNet and for DeltaNet, alpha = 1)
 *   S~_t    = Diag(alpha_t) S_{t-1}    forget
 *   e_t     = beta_t (v_t - S~_t^T k_t)  predict and correct (beta_t: one per token, head)
 *   S_t     = S~_t + k_t e_t^T         rank-one write
 *   o_t     = scale * S_t^T q_t        read after the write
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; nothing is
 *     allocated, freed or retained by the library.  Calls are asynchronous on
 *     `stream` (0 = legacy default stream) and enqueue kernels only.
 *   - Tensors are contiguous and row-major:
 *       q, k, g : [T_total, H, d_k]        v, out : [T_total, H, d_v]
 *       (g is [T_total, H] with KDA_GATE_SCALAR and unused with KDA_GATE_NONE)
 *       beta    : [T_total, H]             states : [N, H, d_k, d_v] fp32
 *       cu_seqlens : int32 [N + 1] (device), nondecreasing, cu[0] = 0,
 *                    cu[N] = T_total; sequence n owns tokens [cu[n], cu[n+1]).
 *                    The kernels check each sequence's pair of offsets on the
 *                    device before any access they guide: a sequence whose
 *                    offsets decrease or leave [0, T_total] is skipped (nothing
 *                    read or written for it, its final state left as it was) and
 *                    KDA_ERR_SEQLENS is recorded (kda_workspace_status for the
 *                    prefill, kda_last_device_status for kda_recurrent_fwd).
 *   - Alignment: states, workspace and (prefill) q, k, v, out and a per-channel g
 *     start on a 16-byte boundary; beta, a per-token g and (decode, recurrent)
 *     q, k, v, g on their element size;
 *     cu_seqlens and accepted on 4 bytes; the decode and recurrent outputs on 4
 *     elements.
 *   - q, k, v, g, beta and out have the I/O dtype (fp32 or bf16); states are
 *     always fp32.  q and k are used as given (normalisation belongs to the
 *     caller, or to the KDA_PREP_* steps below).  g must be finite and <= 0.
 *   - Return value: KDA_OK or a negative KDA_ERR_* code; on error nothing was
 *     enqueued.  No C++ exception crosses the ABI.
 */
#ifndef KDA_GB300_KDA_H_
#define KDA_GB300_KDA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  KDA_OK = 0,
  KDA_ERR_NULL = -1,           /* a required pointer is NULL */
  KDA_ERR_SHAPE = -2,          /* unsupported or inconsistent sizes */
  KDA_ERR_ALIGN = -3,          /* a pointer breaks the alignment stated below */
  KDA_ERR_WORKSPACE = -4,      /* workspace missing or too small */
  KDA_ERR_LAUNCH = -5,         /* CUDA rejected a launch or an async call */
  KDA_ERR_DEVICE = -6,         /* current device is not sm_103 or lacks a needed driver entry */
  KDA_ERR_DEVICE_TIMEOUT = -7, /* (device-reported) a bounded wait in a kernel gave up */
  KDA_ERR_GATE_RANGE = -8,     /* (device-reported) a chunk's decay exceeded the tensor-core path's range */
  KDA_ERR_UNSUPPORTED = -9,    /* the requested algorithm does not support this dtype or size */
  KDA_ERR_NOALLOC_LIMIT = -10, /* the shape needs more scratch than kda_chunk_fwd_noalloc's built-in buffer */
  KDA_ERR_SEQLENS = -11        /* (device-reported) cu_seqlens offsets decrease or leave [0, T_total] */
};

typedef enum { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

/* Which chunk-prefill kernel to run.  AUTO picks TENSOR for bf16 I/O with
 * d_k = d_v = 128 and SIMT otherwise. */
typedef enum { KDA_ALGO_AUTO = 0, KDA_ALGO_TENSOR = 1, KDA_ALGO_SIMT = 2 } kda_algo;

/* How g carries the decay.  The recurrence is the same in all three; only the
 * granularity of alpha_t differs ("Kimi Delta Attention (KDA)", the sections on
 * DeltaNet, on Gated DeltaNet's single retention gate, and on KDA's gate per key
 * channel):
 *   KDA_GATE_CHANNEL  g [T_total, H, d_k]: one log alpha per key channel (KDA)
 *   KDA_GATE_SCALAR   g [T_total, H]: one log alpha per (token, head), applied to
 *                     every key channel (Gated DeltaNet)
 *   KDA_GATE_NONE     alpha_t = 1 (DeltaNet); g is not read and may be NULL */
typedef enum { KDA_GATE_CHANNEL = 0, KDA_GATE_SCALAR = 1, KDA_GATE_NONE = 2 } kda_gate;

/* Weight-free input steps the kernels apply on the fly, as bits of
 * kda_shape.prep ("22580: от GPT-2 до Kimi K3", section "DeltaNet, или Fast
 * Weight Programmers", the forward with a per-token write strength; "K3 架构图解"
 * Ch.08 notes the real module normalises too):
 *   KDA_PREP_QK_SILU      q and k pass through silu(x) = x sigmoid(x)
 *   KDA_PREP_QK_L2NORM    then each (token, head) row of q and of k is divided
 *                         by max(||row||_2, 1e-12) over d_k
 *   KDA_PREP_BETA_SIGMOID beta holds logits; the write strength is sigmoid(beta)
 *   KDA_PREP_G_SOFTPLUS   g holds gate logits x; the log decay is
 *                         log alpha = -c softplus(x) = -c log(1 + e^x) <= 0, with
 *                         c = kda_shape.gate_scale (<= 0 selects 1): a decay rate made
 *                         positive by softplus, as the benchmark workloads draw it
 * The tensors in memory are left as they are.  0 = every input used as given
 * (the default, and the form of the benchmark workloads).  The fp32 paths
 * compute the SiLU in fp32; the tensor-core path (bf16 I/O) computes it on bf16
 * pairs with the hardware tanh, about 0.3 % relative error over a row, and rounds
 * a per-channel -c softplus(x) to bf16 before its chunk cumsum. */
enum { KDA_PREP_QK_SILU = 1, KDA_PREP_QK_L2NORM = 2, KDA_PREP_BETA_SIGMOID = 4,
       KDA_PREP_G_SOFTPLUS = 8 };

typedef struct {
  int32_t num_seqs;     /* N >= 0 (sequences; for decode: independent sequences, one token each) */
  int32_t total_tokens; /* T_total = cu_seqlens[N]; for decode must equal num_seqs */
  int32_t num_heads;    /* H >= 1 */
  int32_t d_k;          /* 64 or 128 */
  int32_t d_v;          /* 64 or 128 */
  int32_t chunk_size;   /* prefill chunk length: 0 or 64 (both mean 64); ignored by decode */
  float scale;          /* output scale; <= 0 selects d_k^-1/2 */
  int32_t io_dtype;     /* kda_dtype of q, k, v, g, beta, out */
  int32_t algo;         /* kda_algo (prefill only) */
  int32_t gate;         /* kda_gate: layout of g (0 = one per key channel) */
  int32_t prep;         /* KDA_PREP_* bits (0 = none); added in ABI 1.2 */
  float gate_scale;     /* c of KDA_PREP_G_SOFTPLUS (<= 0 selects 1); added in ABI 1.4 */
} kda_shape;

/*
 * Chunkwise-parallel prefill over packed variable-length sequences
 * ("Kimi Delta Attention (KDA)", section on the two schedules: chunk-local
 * cumulative log decays, the interaction matrices A^kk and A^qk, the
 * triangular solve (I + R_c)^-1, one sequential state scan across chunks, and
 * the output O_c = s S_c Q_c^boundary + E_c (A^qk_c)^T; the UT/WY form is the
 * chunked DeltaNet section of "22580: от GPT-2 до Kimi K3").  Gives the same
 * states and outputs as running the recurrence token by token.
 *
 *   q, k, v, g, beta : inputs as above (device).
 *   init_state  : [N, H, d_k, d_v] fp32, or NULL for zero initial states.
 *   cu_seqlens  : int32 [N + 1] on the device; read only by the kernels.
 *   out         : [T_total, H, d_v] (io dtype), written for every token.
 *   final_state : [N, H, d_k, d_v] fp32 or NULL; may alias init_state exactly
 *                 (in-place update); no other overlap is allowed.
 *   workspace   : device scratch (16-byte aligned) of at least 256 bytes: the
 *                 device status block read by kda_workspace_status().  With
 *                 kda_chunk_fwd_workspace_bytes() bytes every schedule can run;
 *                 a smaller workspace selects the schedule that fits.  The
 *                 one-chain schedules (plain, solve helpers) give bit-identical
 *                 results; the segment-parallel scan (below) rounds differently
 *                 and agrees with them within the bf16 tolerance.  Calls that
 *                 share one workspace must be ordered on one stream.
 * On the tensor-core path, a few long sequences with few heads (P >= 3 below, and fewer
 * than 2^30 tokens in the call) run as P segments of whole chunks each: the recurrence is affine in the start state, S_end = M S_start + B over any
 * stretch of tokens, so a first launch runs every sequence's segment 0 from the true
 * start and each middle segment from zero (B) and from the identity with V = 0 (M, as
 * d_k = d_v), a small kernel chains S_{p+1} = M_p S_p + B_p in fp32, and a second launch
 * runs segments 1 .. P - 1 from those states.  P = min((SMs / (N H) + 3) / 2, chunks of
 * the average sequence / 32), so the first launch's N H (2P - 3) CTAs fit in one wave;
 * each sequence is cut by its own length.
 * The tensor-core kernel forms its decay factors relative to each chunk's start, so
 * they stay finite while a chunk's total log decay per key channel is above -80.  A
 * sequence-head with a chunk beyond that (a very fast decay, alpha -> 0) is marked in
 * one flag word per sequence-head after the status block, and a second kernel of the
 * same call recomputes it token by token with exact decays (status word 3 counts such
 * sequence-heads).  That needs 256 + 4 N H bytes (rounded up to 256) of workspace,
 * included in kda_chunk_fwd_workspace_bytes(); with less, such a call reports
 * KDA_ERR_GATE_RANGE and its results are undefined.
 * Zero sequences or zero tokens are valid (nothing but the status reset is enqueued).
 * Sequences must be at most 2^31 - 1 tokens long in total; an empty sequence
 * copies its initial state to final_state.
 */
int kda_chunk_fwd(const kda_shape *shape, const void *q, const void *k, const void *v,
                  const void *g, const void *beta, const float *init_state,
                  const int32_t *cu_seqlens, void *out, float *final_state, void *workspace,
                  size_t workspace_bytes, cudaStream_t stream);

/* Bytes of workspace with which kda_chunk_fwd can run every schedule for this
 * shape (always >= 256), or 0 if the shape is invalid: the status block, on the
 * tensor-core path with a gate one flag word per sequence-head (rounded up to 256
 * bytes), and either, for few sequence-heads, a ring through which extra CTAs hand
 * over the chunk solve (4 x 16 KiB + 32 bytes per sequence-head) or, for 2 to 2048
 * sequences, the launch order (4 bytes per sequence, rounded up to 256) with which
 * the longest sequences start first when the launch takes more than one wave.  For
 * sequences that run as P >= 3 segments it is the larger of that and the segments'
 * room: the run tables and skip marks (48 P N + 4 N H bytes rounded up to 256), 4P - 5
 * fp32 states of d_k x d_v per sequence-head, and the solve helpers' ring for the larger
 * pass with at most 76 (run, head) pairs.  P depends on the current device's SM count
 * (152 assumed without a device). */
size_t kda_chunk_fwd_workspace_bytes(const kda_shape *shape);

/* The prefill kernel a call with this shape runs: KDA_ALGO_TENSOR or
 * KDA_ALGO_SIMT (AUTO resolved), or a negative KDA_ERR_* code. */
int kda_chunk_fwd_selected_algo(const kda_shape *shape);

/*
 * One recurrent step for N independent sequences, one token each (the "fused
 * recurrent" schedule of "Kimi Delta Attention (KDA)" with a single token):
 * state is read once, updated in place, and written once.
 *   q, k, g : [N, H, d_k]; v, out : [N, H, d_v]; beta : [N, H] (io dtype, device)
 *   state   : [N, H, d_k, d_v] fp32 (device), updated in place.
 * shape->total_tokens must equal shape->num_seqs; chunk_size and algo are ignored.
 */
int kda_decode_step(const kda_shape *shape, const void *q, const void *k, const void *v,
                    const void *g, const void *beta, float *state, void *out,
                    cudaStream_t stream);

/*
 * The recurrence token by token over short packed sequences: the "fused
 * recurrent" schedule of "Kimi Delta Attention (KDA)" (one program per sequence
 * and head that walks its tokens with the state held on chip), here with the
 * state read once and written once per call.  For speculative decoding ("K3
 * 架构图解", the section on speculative decoding: a recurrent state must roll
 * back the rejected drafts):
 *   1. verify: the draft tokens of each sequence as one packed sequence, with
 *      out and final_state = NULL: the outputs of every draft, state untouched;
 *   2. commit: the same call with out = NULL, final_state = the state (may alias
 *      init_state) and accepted[n] = the drafts sequence n keeps: the state
 *      advances over exactly those tokens.
 * Both can be combined in one call when the counts are known in advance.
 *
 *   q, k, v, g, beta, init_state, cu_seqlens : as for kda_chunk_fwd (device).
 *   accepted    : int32 [N] on the device, or NULL (= every token).  final_state
 *                 of sequence n is the state after its first accepted[n] tokens
 *                 (clamped to [0, length]).
 *   out         : [T_total, H, d_v] (io dtype) or NULL; when given, every token's
 *                 output is written.
 *   final_state : [N, H, d_k, d_v] fp32 or NULL; may alias init_state exactly.
 * chunk_size and algo are ignored.  Every (sequence, head) takes one pass over
 * its tokens, so this suits sequences of a few to a few dozen tokens; longer
 * ones belong to kda_chunk_fwd.  With out and final_state both NULL nothing is
 * enqueued.
 */
int kda_recurrent_fwd(const kda_shape *shape, const void *q, const void *k, const void *v,
                      const void *g, const void *beta, const float *init_state,
                      const int32_t *cu_seqlens, const int32_t *accepted, void *out,
                      float *final_state, cudaStream_t stream);

/*
 * kda_chunk_fwd for callers that cannot allocate device memory.  The method
 * itself has no counterpart to this: it exists for callers that own only their
 * input and output buffers (a host framework whose device memory is all
 * reserved by its own allocator, a plug-in handed tensors but no allocator, or
 * a latency-critical path where cudaMalloc, which can synchronise the device,
 * is not acceptable).
 *
 * Same arguments and results as kda_chunk_fwd, without the workspace: the
 * scratch comes from a 256 KiB buffer compiled into the library, which every
 * GPU that loads the library holds until the process exits.  The status block
 * and the recomputation flags (4 bytes per sequence-head) must fit in it: a shape
 * of more than 65,472 sequence-heads is rejected with KDA_ERR_NOALLOC_LIMIT.  The
 * schedule that fits the rest runs.  Nothing is allocated or freed.  The first
 * call on a device (made while that device is current) looks the buffer's
 * address up, again after a cudaDeviceReset, so make that first call before any
 * stream capture.  All calls on one device share the buffer and it keeps the
 * last call's contents (each call clears the status block and flags it needs);
 * calls whose kernels overlap on the GPU race on it, so order them on one stream.
 * kda_noalloc_status() reads the device status of the last call.
 */
int kda_chunk_fwd_noalloc(const kda_shape *shape, const void *q, const void *k, const void *v,
                          const void *g, const void *beta, const float *init_state,
                          const int32_t *cu_seqlens, void *out, float *final_state,
                          cudaStream_t stream);

/* Synchronises `stream` and returns the device status of the last
 * kda_chunk_fwd_noalloc on the current device (as kda_workspace_status does for a
 * caller workspace); with `words` non-NULL also copies the first four words of its
 * status block there (see kda_workspace_status).  The method has no counterpart to
 * this; it serves the callers of kda_chunk_fwd_noalloc, which own no workspace to
 * read. */
int kda_noalloc_status(uint32_t *words, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads the status block that the kernels of the
 * last kda_chunk_fwd on this workspace wrote: KDA_OK, KDA_ERR_DEVICE_TIMEOUT,
 * KDA_ERR_SEQLENS or KDA_ERR_GATE_RANGE.  A CUDA error while reading returns
 * KDA_ERR_LAUNCH.  Word 2 of the block holds the tensor-core schedule that ran
 * (1 plain, 2 with solve helpers, 3 the segment-parallel scan), word 3 the
 * sequence-heads recomputed token by token.
 */
int kda_workspace_status(const void *workspace, cudaStream_t stream);

/*
 * Synchronises `stream`, then returns and clears the first error the kernels of
 * kda_recurrent_fwd recorded on the current device since the last read: KDA_OK or
 * KDA_ERR_SEQLENS.  A CUDA error while reading returns KDA_ERR_LAUNCH.
 */
int kda_last_device_status(cudaStream_t stream);

/* Static English description of a status code. */
const char *kda_status_string(int status);

/* Library ABI version (major * 1000 + minor); 1001 added kda_recurrent_fwd,
 * 1002 the kda_shape.prep field, 1003 the device check of cu_seqlens
 * (KDA_ERR_SEQLENS, kda_last_device_status), the exact recomputation beyond the
 * tensor-core decay range and kda_noalloc_status, 1004 KDA_PREP_G_SOFTPLUS and
 * kda_shape.gate_scale, 1005 the segment-parallel scan of long sequences (schedule
 * word 3 and its workspace). */
int kda_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_H_ */
