// Chunkwise KDA prefill on CUDA cores, fp32 arithmetic throughout.
//
// This is the chunk schedule of "Kimi Delta Attention (KDA)" (brain.bigb.es,
// section on the two schedules), written for the d_k x d_v state layout.  For a
// chunk of C = 64 tokens with incoming state S (the d_v tile of this CTA):
//
//   G_i     = sum_{u <= i} g_u                        chunk-local cumulative log decay
//   Ebar_i  = beta_i (v_i - S^T (exp(G_i) * k_i))     preliminary errors
//   A_ij    = beta_i k_j^T D_{j+1:i} k_i   (j < i)    rho_ij, D_{j+1:i} = exp(G_i - G_j)
//   X_ij    = k_j^T D_{j+1:i} q_i          (j <= i)   chi_ij (diagonal included)
//   E       = (I + A)^-1 Ebar                          causal triangular solve
//   O_i     = s (S^T (exp(G_i) * q_i) + sum_{j <= i} X_ij e_j)
//   S_next  = Diag(exp(G_last)) S + sum_i (exp(G_last - G_i) * k_i) e_i^T
//
// The decays D_{j+1:i} are formed pairwise as exp(G_i - G_j) <= 1, so any g <= 0
// is handled without a range limit.  Rows past the end of a sequence are
// zero-filled (k = q = v = g = beta = 0), which writes and decays nothing.
//
// This kernel serves fp32 I/O (which needs ~1e-6 relative accuracy that bf16
// tensor-core operands cannot give) and any shape the tensor-core kernel does
// not take.  Grid: one CTA per (sequence, head, d_v tile of 32 columns).
#include <cuda_bf16.h>

#include "kda_internal.h"

namespace kda {
namespace {

constexpr int C = 64;         // chunk length
constexpr int BV = 32;        // d_v columns per CTA
constexpr int NT = 256;       // threads per CTA

template <typename IO>
__device__ __forceinline__ float ld_f32(const IO *p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float *p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16 *p) {
  return __bfloat162float(*p);
}
template <typename IO>
__device__ __forceinline__ void st_io(IO *p, float x);
template <>
__device__ __forceinline__ void st_io<float>(float *p, float x) { *p = x; }
template <>
__device__ __forceinline__ void st_io<__nv_bfloat16>(__nv_bfloat16 *p, float x) {
  *p = __float2bfloat16_rn(x);
}

// Input steps of kda_shape.prep in fp32 (see kda.h): silu(x) = x / (1 + e^-x), the
// sigmoid of a write-strength logit, and 1 / max(||x||, 1e-12) = rsqrt(max(||x||^2, 1e-24)).
__device__ __forceinline__ float silu_f32(float x) { return x / (1.f + __expf(-x)); }
__device__ __forceinline__ float sigmoid_f32(float x) { return 1.f / (1.f + __expf(-x)); }

template <int DK>
struct SimtSmem {
  static constexpr int LK = DK + 1;  // padded row length (conflict-free column walks)
  static constexpr int LV = BV + 1;
  float K[C][LK];      // raw keys; reused for K^end after the output step
  float Q[C][LK];      // raw queries
  float G[C][LK];      // cumulative log decay
  float EG[C][LK];     // exp(G)
  float V[C][LV];
  float E[C][LV];      // preliminary errors, solved in place
  float S[DK][LV];     // state tile
  float A[C][C + 1];   // rho (strictly lower)
  float X[C][C + 1];   // chi (lower, diagonal included)
  float beta[C];
};

template <typename IO, int DK>
__global__ void __launch_bounds__(NT)
    kda_chunk_simt_kernel(const IO *__restrict__ q, const IO *__restrict__ k,
                          const IO *__restrict__ v, const IO *__restrict__ g,
                          const IO *__restrict__ beta, const float *__restrict__ init_state,
                          const int32_t *__restrict__ cu_seqlens, IO *__restrict__ out,
                          float *__restrict__ final_state, int H, int DV, float scale,
                          int gate, int prep, float gs, int T, uint32_t *status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SimtSmem<DK> &sm = *reinterpret_cast<SimtSmem<DK> *>(smem_raw);

  const int pair = blockIdx.x;  // n * H + h
  const int n = pair / H, h = pair % H;
  const int col0 = blockIdx.y * BV;
  const int tid = threadIdx.x;
  // offsets out of order or out of range: no token read or written, no state stored
  int bos, eos;
  const bool seq_ok = seq_range(cu_seqlens, n, T, tid == 0 ? status : nullptr, bos, eos);
  const size_t state_off = (size_t)pair * DK * DV;

  for (int idx = tid; idx < DK * BV; idx += NT) {
    const int r = idx / BV, c = idx % BV;
    sm.S[r][c] = init_state ? init_state[state_off + (size_t)r * DV + col0 + c] : 0.f;
  }

  for (int c0 = bos; c0 < eos; c0 += C) {
    const int len = min(C, eos - c0);
    __syncthreads();  // previous chunk fully consumed

    // a1: load the chunk (zero rows past the end) ------------------------
    for (int idx = tid; idx < C * DK; idx += NT) {
      const int r = idx / DK, j = idx % DK;
      float kv = 0.f, qv = 0.f, gv = 0.f;
      if (r < len) {
        const size_t o = ((size_t)(c0 + r) * H + h) * DK + j;
        kv = ld_f32(k + o);
        qv = ld_f32(q + o);
        if (prep & kPrepSilu) {
          kv = silu_f32(kv);
          qv = silu_f32(qv);
        }
        // g per key channel (KDA), one per token for every channel (Gated DeltaNet), or 0
        // (gate logits through -c softplus with KDA_PREP_G_SOFTPLUS)
        if (gate == 0) gv = gate_log<true>(ld_f32(g + o), prep, gs);
        else if (gate == 1) gv = gate_log<true>(ld_f32(g + (size_t)(c0 + r) * H + h), prep, gs);
      }
      sm.K[r][j] = kv;
      sm.Q[r][j] = qv;
      sm.G[r][j] = gv;
    }
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int r = idx / BV, c = idx % BV;
      sm.V[r][c] = r < len ? ld_f32(v + ((size_t)(c0 + r) * H + h) * DV + col0 + c) : 0.f;
    }
    if (tid < C) {
      float b = 0.f;  // rows past the end write nothing, with or without the sigmoid
      if (tid < len) {
        b = ld_f32(beta + (size_t)(c0 + tid) * H + h);
        if (prep & kPrepBetaSigmoid) b = sigmoid_f32(b);
      }
      sm.beta[tid] = b;
    }
    __syncthreads();

    // optional L2 norm of each row of K and Q (zero rows stay zero), warp per row;
    // it overlaps the cumsum below, which reads G only
    if (prep & kPrepL2) {
      const int lane = tid & 31;
      for (int rr = tid >> 5; rr < 2 * C; rr += NT / 32) {
        float *x = rr < C ? sm.K[rr] : sm.Q[rr - C];
        float acc = 0.f;
        for (int j = lane; j < DK; j += 32) acc = fmaf(x[j], x[j], acc);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const float rn = rsqrtf(fmaxf(acc, 1e-24f));
        for (int j = lane; j < DK; j += 32) x[j] *= rn;
      }
    }

    // a1: per-channel inclusive cumulative sum of g inside the chunk ------
    for (int j = tid; j < DK; j += NT) {
      float acc = 0.f;
      for (int r = 0; r < C; ++r) {
        acc += sm.G[r][j];
        sm.G[r][j] = acc;
        sm.EG[r][j] = expf(acc);
      }
    }
    __syncthreads();

    // a2: interaction matrices rho (A) and chi (X), pairwise decays -------
    for (int p = tid; p < C * C; p += NT) {
      const int i = p / C, j = p % C;
      float a = 0.f, x = 0.f;
      if (j <= i) {
        for (int d = 0; d < DK; ++d) {
          const float kj = sm.K[j][d] * expf(sm.G[i][d] - sm.G[j][d]);
          a += sm.K[i][d] * kj;
          x += sm.Q[i][d] * kj;
        }
      }
      sm.A[i][j] = j < i ? sm.beta[i] * a : 0.f;
      sm.X[i][j] = x;
    }
    // preliminary errors Ebar = diag(beta) (V - (exp(G) * K) S)
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int i = idx / BV, c = idx % BV;
      float acc = 0.f;
      for (int d = 0; d < DK; ++d) acc += sm.EG[i][d] * sm.K[i][d] * sm.S[d][c];
      sm.E[i][c] = sm.beta[i] * (sm.V[i][c] - acc);
    }
    __syncthreads();

    // a3: E = (I + A)^-1 Ebar by blocked forward substitution -------------
    // Rows in blocks of 8: all threads first subtract the contribution of
    // every finished row, then one warp resolves the 8 x 8 diagonal block.
    for (int b = 0; b < C; b += 8) {
      if (b > 0) {
        const int i = b + tid / BV, c = tid % BV;  // NT == 8 * BV
        float acc = sm.E[i][c];
        for (int j = 0; j < b; ++j) acc -= sm.A[i][j] * sm.E[j][c];
        sm.E[i][c] = acc;
      }
      __syncthreads();
      if (tid < BV) {
        const int c = tid;
        for (int i = b + 1; i < b + 8; ++i) {
          float acc = sm.E[i][c];
          for (int j = b; j < i; ++j) acc -= sm.A[i][j] * sm.E[j][c];
          sm.E[i][c] = acc;
        }
      }
      __syncthreads();
    }

    // a5: output O = s ((exp(G) * Q) S + X E) -----------------------------
    for (int idx = tid; idx < C * BV; idx += NT) {
      const int i = idx / BV, c = idx % BV;
      if (i < len) {
        float acc = 0.f;
        for (int d = 0; d < DK; ++d) acc += sm.EG[i][d] * sm.Q[i][d] * sm.S[d][c];
        for (int j = 0; j <= i; ++j) acc += sm.X[i][j] * sm.E[j][c];
        st_io(out + ((size_t)(c0 + i) * H + h) * DV + col0 + c, scale * acc);
      }
    }
    __syncthreads();

    // a4: state pass S <- Diag(exp(G_last)) S + (K^end)^T E ----------------
    for (int idx = tid; idx < C * DK; idx += NT) {
      const int r = idx / DK, j = idx % DK;
      sm.K[r][j] *= expf(sm.G[C - 1][j] - sm.G[r][j]);  // K^end
    }
    __syncthreads();
    for (int idx = tid; idx < DK * BV; idx += NT) {
      const int d = idx / BV, c = idx % BV;
      float acc = sm.EG[C - 1][d] * sm.S[d][c];
      for (int i = 0; i < C; ++i) acc += sm.K[i][d] * sm.E[i][c];
      sm.S[d][c] = acc;
    }
  }
  __syncthreads();
  if (final_state && seq_ok) {
    for (int idx = tid; idx < DK * BV; idx += NT) {
      const int r = idx / BV, c = idx % BV;
      final_state[state_off + (size_t)r * DV + col0 + c] = sm.S[r][c];
    }
  }
}

template <typename IO, int DK>
cudaError_t launch_t(const ChunkArgs &a, cudaStream_t stream) {
  const int pairs = a.num_seqs * a.num_heads;
  if (pairs == 0) return cudaSuccess;
  const size_t smem = sizeof(SimtSmem<DK>);
  auto kern = kda_chunk_simt_kernel<IO, DK>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid(pairs, a.d_v / BV);
  kern<<<grid, NT, smem, stream>>>(
      static_cast<const IO *>(a.q), static_cast<const IO *>(a.k), static_cast<const IO *>(a.v),
      static_cast<const IO *>(a.g), static_cast<const IO *>(a.beta), a.init_state, a.cu_seqlens,
      static_cast<IO *>(a.out), a.final_state, a.num_heads, a.d_v, a.scale, a.gate, a.prep,
      a.gate_scale, a.total_tokens, a.status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_simt(const ChunkArgs &a, cudaStream_t stream) {
  if (a.d_v % BV != 0) return cudaErrorInvalidValue;
  if (a.d_k == 128) return a.bf16 ? launch_t<__nv_bfloat16, 128>(a, stream) : launch_t<float, 128>(a, stream);
  if (a.d_k == 64) return a.bf16 ? launch_t<__nv_bfloat16, 64>(a, stream) : launch_t<float, 64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kda
