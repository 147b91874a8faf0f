// Single-token KDA decode step (the "fused recurrent" schedule of
// "Kimi Delta Attention (KDA)", brain.bigb.es, with one token per sequence), and
// the same schedule over a few consecutive tokens per sequence (below):
//
//   S~ = Diag(exp(g)) S,  e = beta (v - S~^T k),  S <- S~ + k e^T,
//   o  = scale * S^T q = scale * (S~^T q + e (k . q))
//
// One CTA per (sequence, head).  The fp32 state tile [d_k, d_v] is read from
// HBM exactly once into registers (16-byte streaming loads), decayed, reduced
// over key channels for both S~^T k and S~^T q in the same pass, updated in
// registers and written back exactly once.  The work is HBM-bound: 2 * 4 *
// d_k * d_v bytes of state traffic against ~7 d_k d_v flops.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "kda_internal.h"

namespace kda {
namespace {

// First error the recurrent kernels recorded on this device (0 = none): offsets out
// of order or out of range.  Read and cleared by take_device_status().
__device__ uint32_t g_device_status;

template <typename IO>
__device__ __forceinline__ float to_f32(IO x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename IO>
__device__ __forceinline__ void store4(IO *p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float *p, float4 v) {
  *reinterpret_cast<float4 *>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16 *p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t *>(&a);
  u.y = *reinterpret_cast<uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(p) = u;
}

// Input steps of kda_shape.prep, in fp32: silu(x) = x / (1 + e^-x) (saturates to x
// and -0 without overflow), the logistic sigmoid of a write-strength logit, and
// 1 / max(||x||, 1e-12) as rsqrt(max(||x||^2, 1e-24)).
__device__ __forceinline__ float silu_f32(float x) { return x / (1.f + __expf(-x)); }
__device__ __forceinline__ float sigmoid_f32(float x) { return 1.f / (1.f + __expf(-x)); }
__device__ __forceinline__ float inv_norm_f32(float sumsq) { return rsqrtf(fmaxf(sumsq, 1e-24f)); }

// Sum over the 32 lanes of a warp, every lane gets the total.
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

constexpr int kDecodeThreads = 256;

// kPrep: the input steps of `prep` are compiled in (a call without them runs the
// instantiation that has none of their code).
template <typename IO, int DK, int DV, bool kPrep>
__global__ void __launch_bounds__(kDecodeThreads, 2)
    kda_decode_kernel(const IO *__restrict__ q, const IO *__restrict__ k,
                      const IO *__restrict__ v, const IO *__restrict__ g,
                      const IO *__restrict__ beta, float *__restrict__ state,
                      IO *__restrict__ out, float scale, int gate, int prep, float gs) {
  constexpr int TPR = DV / 4;               // threads covering one state row (float4 each)
  constexpr int RPP = kDecodeThreads / TPR;  // rows covered per pass of the block
  constexpr int RPT = DK / RPP;              // rows held by each thread
  static_assert(RPT * RPP == DK, "row split");

  __shared__ float s_q[DK], s_k[DK], s_a[DK], s_v[DV];
  __shared__ float4 s_red[2][RPP][TPR];
  __shared__ float4 s_e[TPR];
  __shared__ float s_kq, s_beta, s_rn[2];

  const int pair = blockIdx.x;  // n * H + h
  const int tid = threadIdx.x;
  const int c4 = tid % TPR;
  const int r0 = tid / TPR;

  // Issue the state loads first: they are the only HBM-heavy traffic.
  float4 *S4 = reinterpret_cast<float4 *>(state + (size_t)pair * DK * DV);
  float4 s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = __ldcs(&S4[(size_t)(r0 + i * RPP) * TPR + c4]);

  const size_t koff = (size_t)pair * DK, voff = (size_t)pair * DV;
  // alpha per key channel (KDA), one alpha for every channel (Gated DeltaNet), or 1 (DeltaNet)
  const float a_tok = gate == 1 ? __expf(gate_log<kPrep>(to_f32(g[pair]), prep, gs)) : 1.f;
  const bool silu = kPrep && (prep & kPrepSilu);
  for (int i = tid; i < DK; i += kDecodeThreads) {
    const float qi = to_f32(q[koff + i]), ki = to_f32(k[koff + i]);
    s_q[i] = silu ? silu_f32(qi) : qi;
    s_k[i] = silu ? silu_f32(ki) : ki;
    s_a[i] = gate == 0 ? __expf(gate_log<kPrep>(to_f32(g[koff + i]), prep, gs)) : a_tok;
  }
  for (int i = tid; i < DV; i += kDecodeThreads) s_v[i] = to_f32(v[voff + i]);
  if (tid == 0) {
    const float b = to_f32(beta[pair]);
    s_beta = kPrep && (prep & kPrepBetaSigmoid) ? sigmoid_f32(b) : b;
  }
  __syncthreads();
  if (kPrep && (prep & kPrepL2)) {  // warp 0: 1 / ||k||, warp 1: 1 / ||q||; then both rows scaled
    if (tid < 64) {
      const float *x = tid < 32 ? s_k : s_q;
      float acc = 0.f;
      for (int i = tid & 31; i < DK; i += 32) acc = fmaf(x[i], x[i], acc);
      acc = warp_sum(acc);
      if ((tid & 31) == 0) s_rn[tid >> 5] = inv_norm_f32(acc);
    }
    __syncthreads();
    for (int i = tid; i < DK; i += kDecodeThreads) {
      s_k[i] *= s_rn[0];
      s_q[i] *= s_rn[1];
    }
    __syncthreads();
  }

  if (tid < 32) {  // k . q
    float acc = 0.f;
    for (int i = tid; i < DK; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (tid == 0) s_kq = acc;
  }

  // Forget, then partial sums of S~^T k and S~^T q over this thread's rows.
  float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const int r = r0 + i * RPP;
    const float a = s_a[r], kr = s_k[r], qr = s_q[r];
    s[i].x *= a; s[i].y *= a; s[i].z *= a; s[i].w *= a;
    pk.x += s[i].x * kr; pk.y += s[i].y * kr; pk.z += s[i].z * kr; pk.w += s[i].w * kr;
    pq.x += s[i].x * qr; pq.y += s[i].y * qr; pq.z += s[i].z * qr; pq.w += s[i].w * qr;
  }
  s_red[0][r0][c4] = pk;
  s_red[1][r0][c4] = pq;
  __syncthreads();

  if (tid < TPR) {
    float4 P = s_red[0][0][tid], R = s_red[1][0][tid];
#pragma unroll
    for (int j = 1; j < RPP; ++j) {
      const float4 a = s_red[0][j][tid], b = s_red[1][j][tid];
      P.x += a.x; P.y += a.y; P.z += a.z; P.w += a.w;
      R.x += b.x; R.y += b.y; R.z += b.z; R.w += b.w;
    }
    const float bt = s_beta, kq = s_kq;
    const int c = 4 * tid;
    float4 e, o;
    e.x = bt * (s_v[c + 0] - P.x);
    e.y = bt * (s_v[c + 1] - P.y);
    e.z = bt * (s_v[c + 2] - P.z);
    e.w = bt * (s_v[c + 3] - P.w);
    o.x = scale * (R.x + e.x * kq);
    o.y = scale * (R.y + e.y * kq);
    o.z = scale * (R.z + e.z * kq);
    o.w = scale * (R.w + e.w * kq);
    s_e[tid] = e;
    store4<IO>(out + voff + c, o);
  }
  __syncthreads();

  // Rank-one write and the single store of the new state.
  const float4 e = s_e[c4];
#pragma unroll
  for (int i = 0; i < RPT; ++i) {
    const float kr = s_k[r0 + i * RPP];
    s[i].x += kr * e.x; s[i].y += kr * e.y; s[i].z += kr * e.z; s[i].w += kr * e.w;
    __stcs(&S4[(size_t)(r0 + i * RPP) * TPR + c4], s[i]);
  }
}

// Several consecutive tokens per sequence (the same fused recurrent schedule over a
// short packed sequence, for speculative verification: "K3 架构图解", the section on
// speculative decoding and the rollback a recurrent state needs after a rejected
// draft).  One CTA per (sequence, head) walks the sequence's tokens in order with
// the state in registers, read once and written once: the state after the first
// `acc` tokens goes to final_state (acc = accepted[n], clamped to the length, or
// the length), and the outputs of all tokens to out.
//
// Layout: warp w owns the state columns [CW w, CW w + CW) as CG groups of four;
// lane l holds column group l % CG of the rows l / CG + RG i.  Per token a lane
// forms the partial sums of S~^T k and S~^T q for its four columns over its rows,
// and an all-reduce over the RG lanes of its column group (xor shuffles) gives
// every lane its columns' sums: e, the output and the rank-one write follow in
// registers, with no barrier and no shared-memory reduction per token.  The
// inputs of kTokBlock tokens at a time are loaded into shared memory together
// (the first block while the state loads).
constexpr int kTokBlock = 8;
constexpr int kRecThreads = 256;  // 512 (8 columns per warp) measured slower

// 16-byte asynchronous copy global -> shared (L2 only), and the waits on this thread's
// copies; cp.async needs no barrier when a thread reads back only what it copied itself.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// waits until at most the most recently committed group of this thread is in flight
__device__ __forceinline__ void cp_async_wait_but_last() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// kFixup: the exact recomputation of the pairs a tensor-core prefill marked (only_flags,
// only_count); the plain launches run the instantiation without that code.
template <typename IO, int DK, int DV, bool kPrep, bool kFixup>
__global__ void __launch_bounds__(kRecThreads, 2)
    kda_recurrent_kernel(const IO *__restrict__ q, const IO *__restrict__ k,
                         const IO *__restrict__ v, const IO *__restrict__ g,
                         const IO *__restrict__ beta, const float *init_state,
                         const int32_t *__restrict__ cu_seqlens,
                         const int32_t *__restrict__ accepted, IO *__restrict__ out,
                         float *final_state, int H, float scale, int gate, int prep, float gs,
                         int npairs, bool staged, int T, uint32_t *status,
                         const uint32_t *only_flags, const uint32_t *only_count) {
  // only_flags: run only the pairs whose flag is set (the exact recomputation of pairs
  // the tensor-core prefill marked), and nothing at all while *only_count is 0
  if (kFixup && *only_count == 0u) return;
  constexpr int kWarps = kRecThreads / 32;
  static_assert(kTokBlock <= kWarps, "one warp per token of a block normalises its q and k");
  constexpr int CW = DV / kWarps;  // columns per warp (16 or 8)
  constexpr int CG = CW / 4;       // column groups of four per warp
  constexpr int RG = 32 / CG;      // lanes per column group = row stride
  constexpr int RPL = DK / RG;     // rows per lane
  static_assert(CW % 4 == 0 && RPL * RG == DK, "warp layout");

  // q, k and the decay of a token are stored with the key channels permuted, channel
  // r at (r % RG) RPL + r / RG, so that the RPL rows a lane holds (rg + RG i) are
  // contiguous and read as float4s
  __shared__ __align__(16) float s_q[kTokBlock][DK], s_k[kTokBlock][DK], s_a[kTokBlock][DK];
  __shared__ float s_v[kTokBlock][DV], s_beta[kTokBlock], s_alpha_tok[kTokBlock];

  // This thread's RPL state float4s of the next pair wait in shared memory, interleaved
  // over the block (float4 i of thread t at i * kRecThreads + t, so a warp's reads are
  // contiguous): each CTA walks pairs blockIdx.x, + gridDim.x, ..., and the state of its
  // next pair streams in while it runs the current pair's tokens.
  extern __shared__ __align__(16) float4 s_next[];
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int cg = lane % CG, rg = lane / CG;
  const int col = CW * w + 4 * cg;  // this lane's four columns
  auto prefetch = [&](int p) {
    if (init_state) {
      const float *src = init_state + (size_t)p * DK * DV + col;
#pragma unroll
      for (int i = 0; i < RPL; ++i) cp_async16(&s_next[i * kRecThreads + tid], src + (size_t)(rg + RG * i) * DV);
    }
    cp_async_commit();  // one group per pair, empty without an initial state
  };
  // The raw q, k, g (per key channel) and v rows of the first kTokBlock tokens of the
  // next pair follow in shared memory, [kTokBlock][q | k | g | v] in the I/O type, copied
  // in 16-byte pieces (the launch only stages with 16-byte aligned tensors).
  constexpr int kRawRow = 3 * DK + DV;  // elements per token
  IO *s_raw = reinterpret_cast<IO *>(s_next + RPL * kRecThreads);
  auto pair_steps = [&](int p, int &pbos) {
    const int pn = p / H;
    if (kFixup && only_flags[p] == 0u) return 0;
    // offsets out of order or out of range: no token (recorded when the pair runs)
    pbos = cu_seqlens[pn];
    const bool ok = 0 <= pbos && pbos <= cu_seqlens[pn + 1] && cu_seqlens[pn + 1] <= T;
    const int plen = ok ? cu_seqlens[pn + 1] - pbos : 0;
    const int pacc = accepted ? min(max(accepted[pn], 0), plen) : plen;
    return out ? plen : pacc;
  };
  // beta and a per-token log alpha of the next pair's first block wait in registers of
  // threads 0 .. kTokBlock - 1 (one token each)
  float beta_pre = 0.f, gtok_pre = 0.f;
  auto prefetch_inputs = [&](int p) {
    int pbos = 0;
    const int nb = min(kTokBlock, pair_steps(p, pbos));
    const int ph = p % H;
    if (tid < nb) {
      beta_pre = to_f32(beta[(size_t)(pbos + tid) * H + ph]);
      if (gate == 1) gtok_pre = to_f32(g[(size_t)(pbos + tid) * H + ph]);
    }
    constexpr int kPer = 16 / sizeof(IO);  // elements per 16-byte piece
    constexpr int kPieces = kRawRow / kPer;
    for (int ci = tid; ci < nb * kPieces; ci += kRecThreads) {
      const int j = ci / kPieces, e = (ci % kPieces) * kPer;  // token, element in the raw row
      const size_t row = (size_t)(pbos + j) * H + ph;
      const IO *src = nullptr;  // the g part only with one log alpha per key channel
      if (e < DK) src = q + row * DK + e;
      else if (e < 2 * DK) src = k + row * DK + (e - DK);
      else if (e < 3 * DK) src = gate == 0 ? g + row * DK + (e - 2 * DK) : nullptr;
      else src = v + row * DV + (e - 3 * DK);
      if (src) cp_async16(s_raw + j * kRawRow + e, src);
    }
    cp_async_commit();
  };
  if (staged && (int)blockIdx.x < npairs) {
    prefetch(blockIdx.x);
    prefetch_inputs(blockIdx.x);
  }

  for (int pair = blockIdx.x; pair < npairs; pair += gridDim.x) {  // pair = n * H + h
  if (kFixup && only_flags[pair] == 0u) continue;  // (fixup launches are unstaged)
  const int n = pair / H, h = pair % H;
  // offsets out of order or out of range: no token and no state written for the pair (the
  // test is written so that bos and len stay reloadable from cu_seqlens: no extra registers)
  const int bos = cu_seqlens[n];
  const bool seq_ok = 0 <= bos && bos <= cu_seqlens[n + 1] && cu_seqlens[n + 1] <= T;
  const int len = seq_ok ? cu_seqlens[n + 1] - bos : 0;
  if (!seq_ok && tid == 0) atomicCAS(status, 0u, kStatusSeqlens);
  const int acc = accepted ? min(max(accepted[n], 0), len) : len;
  const int steps = out ? len : acc;  // outputs need every token, the state only the first acc

  const size_t soff = (size_t)pair * DK * DV + col;
  float4 s[RPL];
  // staged: in flight are [state(pair)], [inputs(pair)], so waiting for all but the
  // last group gives this pair's state; its inputs are waited for below
  const bool more = staged && pair + (int)gridDim.x < npairs;
  if (staged) cp_async_wait_but_last();
  if (init_state && staged) {
#pragma unroll
    for (int i = 0; i < RPL; ++i) s[i] = s_next[i * kRecThreads + tid];
  } else if (init_state) {  // one pair per CTA: straight into registers
#pragma unroll
    for (int i = 0; i < RPL; ++i)
      s[i] = __ldcs(reinterpret_cast<const float4 *>(init_state + soff + (size_t)(rg + RG * i) * DV));
  } else {
#pragma unroll
    for (int i = 0; i < RPL; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // this thread's state slots are free again: the next pair's state streams in (the
  // last pair commits an empty group, so that "all but the last group" below still
  // covers this pair's inputs)
  if (more) prefetch(pair + gridDim.x);
  else if (staged) cp_async_commit();
  auto store_state = [&]() {
#pragma unroll
    for (int i = 0; i < RPL; ++i)
      __stcs(reinterpret_cast<float4 *>(final_state + soff + (size_t)(rg + RG * i) * DV), s[i]);
  };
  if (final_state && acc == 0 && seq_ok) store_state();
  if (more && steps == 0) {  // nothing reads this pair's staged inputs
    cp_async_wait_but_last();  // they have landed before the next pair's overwrite them
    prefetch_inputs(pair + gridDim.x);
  }

  for (int tb = 0; tb < steps; tb += kTokBlock) {
    const int nb = min(kTokBlock, steps - tb);
    // the block's inputs, once every thread is done with the previous block's (of this
    // pair or of the CTA's previous pair)
    if (tb > 0 || pair != (int)blockIdx.x) __syncthreads();
    const bool from_raw = staged && tb == 0;  // the first block was staged
    if (from_raw) {
      if (tid < nb) {
        s_beta[tid] = kPrep && (prep & kPrepBetaSigmoid) ? sigmoid_f32(beta_pre) : beta_pre;
        if (gate == 1) s_alpha_tok[tid] = __expf(gate_log<kPrep>(gtok_pre, prep, gs));
      }
      cp_async_wait_but_last();  // [inputs(pair)] done; [state(next)] may be in flight
      __syncthreads();           // every thread's pieces
    }
    for (int idx = tid; idx < nb * DK; idx += kRecThreads) {
      const int j = idx / DK, i = idx % DK;
      if (!from_raw) break;
      const IO *rr = s_raw + j * kRawRow;
      const float qi = to_f32(rr[i]), ki = to_f32(rr[DK + i]);
      const int pi = (i % RG) * RPL + i / RG;
      s_q[j][pi] = kPrep && (prep & kPrepSilu) ? silu_f32(qi) : qi;
      s_k[j][pi] = kPrep && (prep & kPrepSilu) ? silu_f32(ki) : ki;
      s_a[j][pi] = gate == 0 ? __expf(gate_log<kPrep>(to_f32(rr[2 * DK + i]), prep, gs))
                             : (gate == 1 ? s_alpha_tok[j] : 1.f);
    }
    for (int idx = tid; idx < nb * DV; idx += kRecThreads) {
      if (!from_raw) break;
      const int j = idx / DV, i = idx % DV;
      s_v[j][i] = to_f32(s_raw[j * kRawRow + 3 * DK + i]);
    }
    for (int idx = tid; idx < nb * DK; idx += kRecThreads) {
      if (from_raw) break;
      const int j = idx / DK, i = idx % DK;
      const size_t row = (size_t)(bos + tb + j) * H + h;
      const float qi = to_f32(q[row * DK + i]), ki = to_f32(k[row * DK + i]);
      const int pi = (i % RG) * RPL + i / RG;
      s_q[j][pi] = kPrep && (prep & kPrepSilu) ? silu_f32(qi) : qi;
      s_k[j][pi] = kPrep && (prep & kPrepSilu) ? silu_f32(ki) : ki;
      s_a[j][pi] = gate == 0 ? __expf(gate_log<kPrep>(to_f32(g[row * DK + i]), prep, gs))
                             : (gate == 1 ? __expf(gate_log<kPrep>(to_f32(g[row]), prep, gs)) : 1.f);
    }
    for (int idx = tid; idx < nb * DV; idx += kRecThreads) {
      if (from_raw) break;
      const int j = idx / DV, i = idx % DV;
      s_v[j][i] = to_f32(v[((size_t)(bos + tb + j) * H + h) * DV + i]);
    }
    if (tid < nb && !from_raw) {
      const float b = to_f32(beta[(size_t)(bos + tb + tid) * H + h]);
      s_beta[tid] = kPrep && (prep & kPrepBetaSigmoid) ? sigmoid_f32(b) : b;
    }
    __syncthreads();
    // the raw rows have been read by every thread: the next pair's may stream in
    if (more && tb == 0) prefetch_inputs(pair + gridDim.x);
    if (kPrep && (prep & kPrepL2)) {  // warp w divides token w's k and q by their norms
      if (w < nb) {
        float sk = 0.f, sq = 0.f;
        for (int i = lane; i < DK; i += 32) {
          sk = fmaf(s_k[w][i], s_k[w][i], sk);
          sq = fmaf(s_q[w][i], s_q[w][i], sq);
        }
        sk = inv_norm_f32(warp_sum(sk));
        sq = inv_norm_f32(warp_sum(sq));
        for (int i = lane; i < DK; i += 32) {
          s_k[w][i] *= sk;
          s_q[w][i] *= sq;
        }
      }
      __syncthreads();
    }

    for (int jt = 0; jt < nb; ++jt) {
      const int t = tb + jt;
      // forget, then this lane's partial sums of S~^T k, S~^T q (4 columns) and k . q
      float4 pk = make_float4(0.f, 0.f, 0.f, 0.f), pq = pk;
      float kq = 0.f;
      const float4 *a4 = reinterpret_cast<const float4 *>(&s_a[jt][rg * RPL]);
      const float4 *k4 = reinterpret_cast<const float4 *>(&s_k[jt][rg * RPL]);
      const float4 *q4 = reinterpret_cast<const float4 *>(&s_q[jt][rg * RPL]);
#pragma unroll
      for (int i4 = 0; i4 < RPL / 4; ++i4) {
        const float4 av = a4[i4], kv = k4[i4], qv = q4[i4];
        const float aa[4] = {av.x, av.y, av.z, av.w}, ka[4] = {kv.x, kv.y, kv.z, kv.w},
                    qa[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // row rg + RG (4 i4 + e)
          const float a = aa[e], kr = ka[e], qr = qa[e];
          float4 &u = s[4 * i4 + e];
          u.x *= a; u.y *= a; u.z *= a; u.w *= a;
          pk.x = fmaf(u.x, kr, pk.x); pk.y = fmaf(u.y, kr, pk.y);
          pk.z = fmaf(u.z, kr, pk.z); pk.w = fmaf(u.w, kr, pk.w);
          pq.x = fmaf(u.x, qr, pq.x); pq.y = fmaf(u.y, qr, pq.y);
          pq.z = fmaf(u.z, qr, pq.z); pq.w = fmaf(u.w, qr, pq.w);
          kq = fmaf(kr, qr, kq);
        }
      }
      // all-reduce over the lanes of this column group (they differ in rg: xor CG, 2 CG, ...)
#pragma unroll
      for (int o = CG; o < 32; o <<= 1) {
        pk.x += __shfl_xor_sync(0xffffffffu, pk.x, o);
        pk.y += __shfl_xor_sync(0xffffffffu, pk.y, o);
        pk.z += __shfl_xor_sync(0xffffffffu, pk.z, o);
        pk.w += __shfl_xor_sync(0xffffffffu, pk.w, o);
        pq.x += __shfl_xor_sync(0xffffffffu, pq.x, o);
        pq.y += __shfl_xor_sync(0xffffffffu, pq.y, o);
        pq.z += __shfl_xor_sync(0xffffffffu, pq.z, o);
        pq.w += __shfl_xor_sync(0xffffffffu, pq.w, o);
        kq += __shfl_xor_sync(0xffffffffu, kq, o);
      }
      const float bt = s_beta[jt];
      float4 e4;
      e4.x = bt * (s_v[jt][col + 0] - pk.x);
      e4.y = bt * (s_v[jt][col + 1] - pk.y);
      e4.z = bt * (s_v[jt][col + 2] - pk.z);
      e4.w = bt * (s_v[jt][col + 3] - pk.w);
      if (out && rg == 0) {
        float4 o;
        o.x = scale * (pq.x + e4.x * kq);
        o.y = scale * (pq.y + e4.y * kq);
        o.z = scale * (pq.z + e4.z * kq);
        o.w = scale * (pq.w + e4.w * kq);
        store4<IO>(out + ((size_t)(bos + t) * H + h) * DV + col, o);
      }
      // rank-one write
#pragma unroll
      for (int i4 = 0; i4 < RPL / 4; ++i4) {
        const float4 kv = k4[i4];
        const float ka[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float kr = ka[e];
          float4 &u = s[4 * i4 + e];
          u.x = fmaf(kr, e4.x, u.x); u.y = fmaf(kr, e4.y, u.y);
          u.z = fmaf(kr, e4.z, u.z); u.w = fmaf(kr, e4.w, u.w);
        }
      }
      if (final_state && t == acc - 1) store_state();
    }
  }
  }  // pairs
  if (staged) cp_async_wait_all();  // no copy in flight when the CTA leaves (a last pair without tokens)
}

template <typename IO, int DK, int DV>
cudaError_t launch_recurrent_t(const RecurrentArgs &a, cudaStream_t stream) {
  const long long pairs = (long long)a.num_seqs * a.num_heads;
  if (pairs == 0 || (!a.out && !a.final_state)) return cudaSuccess;
  auto kern = a.prep ? kda_recurrent_kernel<IO, DK, DV, true, false>
                     : kda_recurrent_kernel<IO, DK, DV, false, false>;
  if (a.only_flags) {  // the tensor-core path's recomputation: bf16, d_k = d_v = 128 only
    if constexpr (std::is_same<IO, __nv_bfloat16>::value && DK == 128 && DV == 128)
      kern = a.prep ? kda_recurrent_kernel<IO, DK, DV, true, true>
                    : kda_recurrent_kernel<IO, DK, DV, false, true>;
    else
      return cudaErrorInvalidValue;
  }
  // with two or more tokens per sequence on average: persistent CTAs, two per SM (the
  // launch bound), each staging its next pair's state in DK * DV * 4 bytes of dynamic
  // shared memory while it runs the current one (4 drafts 0.288 -> 0.277 ms, 8 drafts
  // 0.417 -> 0.391 ms); with about one, one CTA per pair (the staging does not pay there)
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  const int smem = DK * DV * 4 + kTokBlock * (3 * DK + DV) * (int)sizeof(IO);
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  // the exact recomputation of marked pairs runs unstaged, two CTAs per SM at most
  const bool staged = !a.only_flags && (long long)a.total_tokens >= 2LL * a.num_seqs &&
                      pairs > 2LL * sms && al16(a.q) && al16(a.k) && al16(a.v) &&
                      (a.gate != 0 || al16(a.g));
  const long long grid = staged ? 2LL * sms : (a.only_flags ? std::min(pairs, 2LL * sms) : pairs);
  uint32_t *status = a.status;
  if (!status && cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_device_status) != cudaSuccess)
    return cudaErrorInvalidDevice;
  kern<<<(unsigned)grid, kRecThreads, staged ? smem : 0, stream>>>(
      static_cast<const IO *>(a.q), static_cast<const IO *>(a.k), static_cast<const IO *>(a.v),
      static_cast<const IO *>(a.g), static_cast<const IO *>(a.beta), a.init_state, a.cu_seqlens,
      a.accepted, static_cast<IO *>(a.out), a.final_state, a.num_heads, a.scale, a.gate, a.prep,
      a.gate_scale, static_cast<int>(pairs), staged, a.total_tokens, status, a.only_flags,
      a.only_count);
  return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_recurrent_io(const RecurrentArgs &a, cudaStream_t stream) {
  if (a.d_k == 128 && a.d_v == 128) return launch_recurrent_t<IO, 128, 128>(a, stream);
  if (a.d_k == 128 && a.d_v == 64) return launch_recurrent_t<IO, 128, 64>(a, stream);
  if (a.d_k == 64 && a.d_v == 128) return launch_recurrent_t<IO, 64, 128>(a, stream);
  if (a.d_k == 64 && a.d_v == 64) return launch_recurrent_t<IO, 64, 64>(a, stream);
  return cudaErrorInvalidValue;
}

template <typename IO, int DK, int DV>
cudaError_t launch_decode_t(const DecodeArgs &a, cudaStream_t stream) {
  const int pairs = a.num_seqs * a.num_heads;
  if (pairs == 0) return cudaSuccess;
  auto kern = a.prep ? kda_decode_kernel<IO, DK, DV, true> : kda_decode_kernel<IO, DK, DV, false>;
  kern<<<pairs, kDecodeThreads, 0, stream>>>(
      static_cast<const IO *>(a.q), static_cast<const IO *>(a.k), static_cast<const IO *>(a.v),
      static_cast<const IO *>(a.g), static_cast<const IO *>(a.beta), a.state,
      static_cast<IO *>(a.out), a.scale, a.gate, a.prep, a.gate_scale);
  return cudaGetLastError();
}

template <typename IO>
cudaError_t launch_decode_io(const DecodeArgs &a, cudaStream_t stream) {
  if (a.d_k == 128 && a.d_v == 128) return launch_decode_t<IO, 128, 128>(a, stream);
  if (a.d_k == 128 && a.d_v == 64) return launch_decode_t<IO, 128, 64>(a, stream);
  if (a.d_k == 64 && a.d_v == 128) return launch_decode_t<IO, 64, 128>(a, stream);
  if (a.d_k == 64 && a.d_v == 64) return launch_decode_t<IO, 64, 64>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
  return a.bf16 ? launch_decode_io<__nv_bfloat16>(a, stream) : launch_decode_io<float>(a, stream);
}

cudaError_t take_device_status(uint32_t *word, cudaStream_t stream) {
  *word = 0;
  cudaError_t err = cudaMemcpyFromSymbolAsync(word, g_device_status, sizeof(uint32_t), 0,
                                              cudaMemcpyDeviceToHost, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  if (err == cudaSuccess && *word != 0) {
    static const uint32_t zero = 0;
    err = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(uint32_t), 0,
                                  cudaMemcpyHostToDevice, stream);
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  }
  return err;
}

cudaError_t launch_recurrent(const RecurrentArgs &a, cudaStream_t stream) {
  return a.bf16 ? launch_recurrent_io<__nv_bfloat16>(a, stream)
                : launch_recurrent_io<float>(a, stream);
}

}  // namespace kda
