// Chunkwise KDA prefill on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// The chunk algebra is the chunkwise schedule of "Kimi Delta Attention (KDA)"
// (brain.bigb.es, section on the two schedules) in the WY / UT form of the
// chunked DeltaNet section of "22580: от GPT-2 до Kimi K3", for the d_k x d_v
// state layout.  For a chunk of C = 64 rows with incoming state S and
// G = chunk-local inclusive cumsum of g (per key channel), Gl = G of the last row:
//
//   Kb   = K * exp(G - Gl)     Qb = Q * exp(G - Gl)     Kend = K * exp(Gl - G)
//   [Kb; Qb] Kend^T            -> rows: A^kk / beta_i (j < i), A^qk (j <= i)
//   T    = (I + A^kk)^-1,  Tb = T diag(beta)           (fp32 triangular solve)
//   Pb   = A^qk Tb
//   [Tb; Pb] [Kb | V]          -> Wbar = Tb Kb, U = Tb V; Pb Kb, O_intra = Pb V
//   W    = Wbar diag(e^Gl)     Q' = (Qb - Pb Kb) diag(e^Gl)
//   [E; O/s] = [U; O_intra] + [-W; Q'] S                (state-dependent)
//   S   <- diag(e^Gl) S + Kend^T E                       (state-dependent)
//
// Anchoring the decay at the chunk end keeps every factor finite as long as a
// chunk's total log decay per channel stays above -80 (checked; beyond it the
// call reports KDA_ERR_GATE_RANGE).  The products use bf16 operands with fp32
// accumulation in tensor memory; the state, the cumsum and the solve are fp32.
//
// One CTA owns (sequence, head, 64-column d_v tile) and walks its chunks in
// order.  Warp roles:
//   warps 0-3  K-side: everything that does not depend on S, one chunk ahead
//   warps 4-7  S-side: holds S (fp32, one key channel per thread) in registers
//              and runs the two state-dependent products per chunk
//   warp  8    TMA producer (q, k, g, v boxes into a 2-stage ring) and TMEM owner
// Every wait on an mbarrier is bounded; on timeout the CTA records
// KDA_ERR_DEVICE_TIMEOUT in the status word and runs to completion without
// waiting again (outputs are then undefined, nothing blocks or faults).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kda_internal.h"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int BV = 64;                      // d_v columns per CTA
constexpr int kThreads = 288;
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMinChunkLogDecay = -80.f;
constexpr uint32_t kStatusTimeout = 7;      // -KDA_ERR_DEVICE_TIMEOUT
constexpr uint32_t kStatusGateRange = 8;    // -KDA_ERR_GATE_RANGE

// Shared memory map (offsets from a 1024-byte aligned base).
struct L {
  // stage: [k ch0-63 | q ch0-63] [k ch64-127 | q ch64-127] [g ch0-63] [g ch64-127] [v tile]
  static constexpr uint32_t kKQ1 = 16384, kQoff = 8192, kG = 32768, kV = 49152;
  static constexpr uint32_t kStageBytes = 49152 + C * BV * 2;
  static constexpr uint32_t kKend = 2 * kStageBytes;          // 2 x [ch0-63 | ch64-127]
  static constexpr uint32_t kTP = kKend + 2 * 16384;          // [Tb rows 0-63 | A^qk / Pb rows 64-127]
  static constexpr uint32_t kSb = kTP + 16384;                // S in bf16, [DK rows][BV]
  static constexpr uint32_t kEb = kSb + DK * BV * 2;          // E in bf16, [C rows][BV]
  static constexpr uint32_t kAf = kEb + C * BV * 2;           // fp32 A^kk [64][65]
  static constexpr uint32_t kTf = kAf + 64 * 65 * 4;          // fp32 T [64][65]
  static constexpr uint32_t kBeta = kTf + 64 * 65 * 4;        // fp32 beta [64]
  static constexpr uint32_t kGamma = kBeta + 256;             // fp32 e^Gl [2][128]
  static constexpr uint32_t kBars = kGamma + 1024;            // mbarriers
  static constexpr uint32_t kMisc = kBars + 128;              // tmem slot, abort flag
  static constexpr uint32_t kTotal = kMisc + 64;
  static constexpr uint32_t kAlloc = kTotal + 1024;
};
static_assert(L::kKend % 1024 == 0 && L::kTP % 1024 == 0 && L::kSb % 1024 == 0 &&
                  L::kEb % 1024 == 0 && L::kAf % 1024 == 0,
              "operand tiles must be 1024-byte aligned");
static_assert(L::kAlloc <= 232448, "shared memory budget");

// mbarrier slots
enum : uint32_t {
  kFull0 = 0, kEmpty0 = 2, kReady0 = 4, kDone0 = 6, kMmaK = 8, kMmaS = 9, kFinK = 10, kFinS = 11,
  kNever = 12, kNumBars = 13
};

// TMEM columns
constexpr uint32_t kD1 = 0, kDP = 64, kD2 = 128, kAcc0 = 256, kD4 = 256 + 2 * BV;

struct TcParams {
  const __nv_bfloat16 *beta;
  const float *init_state;
  const int32_t *cu_seqlens;
  __nv_bfloat16 *out;
  float *final_state;
  uint32_t *status;
  int H;
  float scale;
  int flags;  // bit 0: test hook, wait once on a barrier nothing arrives on
};

struct Ctx {
  uint32_t bars;
  volatile int *abort;
  uint32_t *status;
  __device__ __forceinline__ uint32_t bar(uint32_t i) const { return bars + 8 * i; }
  __device__ __forceinline__ void wait(uint32_t i, uint32_t parity) const {
    if (*abort) return;
    if (!mbar_wait(bar(i), parity, kWaitCycles)) {
      *abort = 1;
      atomicCAS(status, 0u, kStatusTimeout);
    }
  }
};

__device__ __forceinline__ void unpack8(uint4 r, float (&f)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}
__device__ __forceinline__ void st8(uint32_t addr, const float (&f)[8]) {
  const uint4 p = pack8(f);
  st_shared_v4(addr, p.x, p.y, p.z, p.w);
}
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
    kda_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_g,
                        const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  float *Af = reinterpret_cast<float *>(smem + L::kAf);
  float *Tf = reinterpret_cast<float *>(smem + L::kTf);
  float *betas = reinterpret_cast<float *>(smem + L::kBeta);
  float *gamma = reinterpret_cast<float *>(smem + L::kGamma);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  constexpr int kTiles = DV / BV;
  const int tile = blockIdx.x % kTiles;
  const int pair = blockIdx.x / kTiles;
  const int H = p.H;
  const int n = pair / H, h = pair % H;
  const int bos = p.cu_seqlens[n], eos = p.cu_seqlens[n + 1];
  const int nchunks = (eos - bos + C - 1) / C;

  Ctx ctx{sbase + L::kBars, abort_flag, p.status};

  if (tid == 0) {
    *abort_flag = 0;
    for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(ctx.bar(i), 1);
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if ((tid & 31) == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_g);
      tma_prefetch_desc(&tm_v);
      int issued[2] = {-1, -1};
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1;
        if (c >= 2) ctx.wait(kEmpty0 + s, ((c >> 1) - 1) & 1);
        if (*abort_flag) break;
        const uint32_t st = sbase + s * L::kStageBytes;
        const uint32_t fb = ctx.bar(kFull0 + s);
        const int t0 = bos + c * C;
        mbar_arrive_expect_tx(fb, L::kStageBytes);
        tma_load_3d(st, &tm_k, fb, 0, h, t0);
        tma_load_3d(st + L::kQoff, &tm_q, fb, 0, h, t0);
        tma_load_3d(st + L::kKQ1, &tm_k, fb, 64, h, t0);
        tma_load_3d(st + L::kKQ1 + L::kQoff, &tm_q, fb, 64, h, t0);
        tma_load_3d(st + L::kG, &tm_g, fb, 0, h, t0);
        tma_load_3d(st + L::kG + 8192, &tm_g, fb, 64, h, t0);
        tma_load_3d(st + L::kV, &tm_v, fb, tile * BV, h, t0);
        issued[s] = c;
      }
      // never leave a copy in flight: wait (bounded) for the last load of each stage
      for (int s = 0; s < 2; ++s)
        if (issued[s] >= 0) mbar_wait(ctx.bar(kFull0 + s), (issued[s] >> 1) & 1, kWaitCycles);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ K-side
    const int t = tid;  // 0..127
    const uint32_t lane_base = static_cast<uint32_t>(32 * warp) << 16;
    if ((p.flags & 1) && t == 0) {
      // test hook: a wait that can only time out
      if (!mbar_wait(ctx.bar(kNever), 0, 2000000LL)) {
        *abort_flag = 1;
        atomicCAS(p.status, 0u, kStatusTimeout);
      }
    }
    uint32_t kph = 0;
    const int cg = t & 15, half = cg >> 3, ck = cg & 7, rg = t >> 4;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      const int t0 = bos + c * C;
      const int len = min(C, eos - t0);
      const uint32_t st = sbase + s * L::kStageBytes;
      const uint32_t kend = sbase + L::kKend + s * 16384;
      if (c >= 2) ctx.wait(kDone0 + s, ((c >> 1) - 1) & 1);  // Kend[s], ACC[s], gamma[s] free
      ctx.wait(kFull0 + s, (c >> 1) & 1);
      if (t < C) betas[t] = t < len ? __bfloat162float(p.beta[(size_t)(t0 + t) * H + h]) : 0.f;

      // a1: chunk-local cumulative log decay, 8 rows x 8 channels per thread
      const uint32_t kq = st + half * L::kKQ1;
      const uint32_t ga = st + L::kG + half * 8192;
      float gl[8][8], run[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) run[j] = 0.f;
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = rg * 8 + rr;
        float gv[8];
        unpack8(ld_shared_v4(ga + sw128(r, ck)), gv);
        const bool valid = r < len;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          run[j] += valid ? gv[j] : 0.f;
          gl[rr][j] = run[j];
        }
      }
      float *part = Af;  // [8][128] partial sums (Af is free here)
#pragma unroll
      for (int j = 0; j < 8; ++j) part[rg * 128 + cg * 8 + j] = run[j];
      bar_sync(1, 128);
      float pre[8], tot[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) pre[j] = tot[j] = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float v = part[q * 128 + cg * 8 + j];
          if (q < rg) pre[j] += v;
          tot[j] += v;
        }
      }
      if (rg == 0) {
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          gamma[s * 128 + cg * 8 + j] = fast_exp2(tot[j] * kLog2e);
          bad |= !(tot[j] >= kMinChunkLogDecay);
        }
        if (bad) atomicCAS(p.status, 0u, kStatusGateRange);
      }
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = rg * 8 + rr;
        float kv[8], qv[8], f[8], fe[8];
        unpack8(ld_shared_v4(kq + sw128(r, ck)), kv);
        unpack8(ld_shared_v4(kq + L::kQoff + sw128(r, ck)), qv);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float d = (pre[j] + gl[rr][j] - tot[j]) * kLog2e;  // (G - Gl) log2 e <= 0
          f[j] = fast_exp2(d);
          fe[j] = fast_exp2(-d);
        }
        float kb[8], qb[8], ke[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          kb[j] = kv[j] * f[j];
          qb[j] = qv[j] * f[j];
          ke[j] = kv[j] * fe[j];
        }
        st8(kq + sw128(r, ck), kb);
        st8(kq + L::kQoff + sw128(r, ck), qb);
        st8(kend + half * 8192 + sw128(r, ck), ke);
      }
      fence_async_smem();
      bar_sync(1, 128);

      // a2: [Kb; Qb] Kend^T -> D1 (rows 0-63: K^kk, rows 64-127: A^qk)
      if (t == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, false, false);
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
          const uint64_t ad = sdesc_sw128(st + (k8 >> 2) * L::kKQ1 + (k8 & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(kend + (k8 >> 2) * 8192 + (k8 & 3) * 32, 16, 1024);
          mma_bf16(tmem + kD1, ad, bd, id, k8 > 0);
        }
        mma_commit(ctx.bar(kMmaK));
      }
      ctx.wait(kMmaK, kph++ & 1);
      tc_fence_after();
      {
        float a[32];
        if (t < 64) {
          const float bi = betas[t];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tmem_ld32(tmem + lane_base + kD1 + 32 * hh, a);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int j = 32 * hh + jj;
              Af[t * 65 + j] = j < t ? bi * a[jj] : 0.f;
            }
          }
        } else {
          const int i = t - 64;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tmem_ld32(tmem + lane_base + kD1 + 32 * hh, a);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float v[8];
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int j = 32 * hh + 8 * q + jj;
                v[jj] = j <= i ? a[8 * q + jj] : 0.f;
              }
              st8(sbase + L::kTP + sw128(64 + i, 4 * hh + q), v);
            }
          }
        }
      }
      tc_fence_before();
      bar_sync(1, 128);

      // a3: T = (I + A^kk)^-1, 16 x 16 diagonal blocks by forward substitution,
      // then the off-diagonal blocks by block diagonals:
      //   T_IJ = -T_II sum_{J <= K < I} A_IK T_KJ
      if (t < 64) {
        const int I = t >> 4, cc = t & 15;
        const float *Ab = Af + (16 * I) * 65 + 16 * I;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) x[r] = r == cc ? 1.f : 0.f;
#pragma unroll
        for (int r = 1; r < 16; ++r) {
          float acc = 0.f;
#pragma unroll
          for (int m = 0; m < r; ++m) acc = fmaf(Ab[r * 65 + m], x[m], acc);
          if (r > cc) x[r] = -acc;
        }
        float *Tb = Tf + (16 * I) * 65 + 16 * I + cc;
#pragma unroll
        for (int r = 0; r < 16; ++r) Tb[r * 65] = x[r];
      }
      bar_sync(1, 128);
      float *Ys = reinterpret_cast<float *>(smem + (ga - sbase) - half * 8192);  // stage g area
      for (int d = 1; d < 4; ++d) {
        const int nb = 4 - d;
        for (int e = t; e < nb * 256; e += 128) {
          const int b = e >> 8, r = (e >> 4) & 15, cc = e & 15;
          const int I = d + b, J = b;
          const float *arow = Af + (16 * I + r) * 65;
          float acc = 0.f;
          for (int K = J; K < I; ++K) {
#pragma unroll
            for (int m = 0; m < 16; ++m)
              acc = fmaf(arow[16 * K + m], Tf[(16 * K + m) * 65 + 16 * J + cc], acc);
          }
          Ys[(b * 16 + r) * 17 + cc] = acc;
        }
        bar_sync(1, 128);
        for (int e = t; e < nb * 256; e += 128) {
          const int b = e >> 8, r = (e >> 4) & 15, cc = e & 15;
          const int I = d + b, J = b;
          const float *trow = Tf + (16 * I + r) * 65 + 16 * I;
          float acc = 0.f;
          for (int m = 0; m <= r; ++m) acc = fmaf(trow[m], Ys[(b * 16 + m) * 17 + cc], acc);
          Tf[(16 * I + r) * 65 + 16 * J + cc] = -acc;
        }
        bar_sync(1, 128);
      }
      {  // Tb = T diag(beta) -> TP rows 0-63
        const int i = t & 63, hh = t >> 6;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int j = 32 * hh + 8 * q + jj;
            v[jj] = j <= i ? Tf[i * 65 + j] * betas[j] : 0.f;
          }
          st8(sbase + L::kTP + sw128(i, 4 * hh + q), v);
        }
      }
      fence_async_smem();
      bar_sync(1, 128);

      // Pb = A^qk Tb  (M = 128 with Tb stacked on top; rows 64-127 are used)
      if (t == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, 64, false, true);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const uint64_t ad = sdesc_sw128(sbase + L::kTP + k4 * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sbase + L::kTP + k4 * 2048, 8192, 1024);
          mma_bf16(tmem + kDP, ad, bd, id, k4 > 0);
        }
        mma_commit(ctx.bar(kMmaK));
      }
      ctx.wait(kMmaK, kph++ & 1);
      tc_fence_after();
      if (t >= 64) {
        const int i = t - 64;
        float a[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          tmem_ld32(tmem + lane_base + kDP + 32 * hh, a);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) v[jj] = a[8 * q + jj];
            st8(sbase + L::kTP + sw128(64 + i, 4 * hh + q), v);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_sync(1, 128);

      // [Tb; Pb] [Kb | V] -> D2 (Wbar | Pb Kb) and ACC[s] (U | O_intra)
      if (t == 0) {
        tc_fence_after();
        constexpr uint32_t id_k = idesc_bf16(128, 128, false, true);
        constexpr uint32_t id_v = idesc_bf16(128, BV, false, true);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const uint64_t ad = sdesc_sw128(sbase + L::kTP + k4 * 32, 16, 1024);
          const uint64_t bk = sdesc_sw128(st + k4 * 2048, L::kKQ1, 1024);
          const uint64_t bv = sdesc_sw128(st + L::kV + k4 * 2048, 8192, 1024);
          mma_bf16(tmem + kD2, ad, bk, id_k, k4 > 0);
          mma_bf16(tmem + kAcc0 + s * BV, ad, bv, id_v, k4 > 0);
        }
        mma_commit(ctx.bar(kMmaK));
      }
      ctx.wait(kMmaK, kph++ & 1);
      tc_fence_after();
      {  // -W -> over Kb, Q' -> over Qb (the A operand of the state product)
        const int i = t & 63;
        const uint32_t qoff = t < 64 ? 0u : L::kQoff;
        float a[32];
#pragma unroll
        for (int cc4 = 0; cc4 < 4; ++cc4) {
          tmem_ld32(tmem + lane_base + kD2 + 32 * cc4, a);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int ch0 = 32 * cc4 + 8 * q;
            const uint32_t addr = st + (ch0 >> 6) * L::kKQ1 + qoff + sw128(i, (ch0 & 63) >> 3);
            float v[8];
            if (t < 64) {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) v[jj] = -a[8 * q + jj] * gamma[s * 128 + ch0 + jj];
            } else {
              float qb[8];
              unpack8(ld_shared_v4(addr), qb);
#pragma unroll
              for (int jj = 0; jj < 8; ++jj)
                v[jj] = (qb[jj] - a[8 * q + jj]) * gamma[s * 128 + ch0 + jj];
            }
            st8(addr, v);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_sync(1, 128);
      if (t == 0) mbar_arrive(ctx.bar(kReady0 + s));
    }
    if (t == 0) {  // all K-side MMAs retired before TMEM is released
      mma_commit(ctx.bar(kFinK));
      mbar_wait(ctx.bar(kFinK), 0, kWaitCycles);
    }
  } else {
    // ------------------------------------------------------------ S-side
    const int t = tid - 128;  // key channel of the state row this thread holds
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp - 4)) << 16;
    const size_t soff = (size_t)pair * DK * DV + (size_t)t * DV + tile * BV;
    float S[BV];
    if (p.init_state) {
#pragma unroll
      for (int j = 0; j < BV; j += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(p.init_state + soff + j);
        S[j] = v.x; S[j + 1] = v.y; S[j + 2] = v.z; S[j + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < BV; ++j) S[j] = 0.f;
    }
    uint32_t sph = 0;
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      const int t0 = bos + c * C;
      const int len = min(C, eos - t0);
      const uint32_t st = sbase + s * L::kStageBytes;
#pragma unroll
      for (int q = 0; q < BV / 8; ++q) {
        float v[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) v[jj] = S[8 * q + jj];
        st8(sbase + L::kSb + sw128(t, q), v);
      }
      fence_async_smem();
      bar_sync(2, 128);
      ctx.wait(kReady0 + s, (c >> 1) & 1);
      tc_fence_after();
      // a4/a5: [U; O_intra] += [-W; Q'] S
      if (t == 0) {
        constexpr uint32_t id = idesc_bf16(128, BV, false, true);
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8) {
          const uint64_t ad = sdesc_sw128(st + (k8 >> 2) * L::kKQ1 + (k8 & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sbase + L::kSb + k8 * 2048, 8192, 1024);
          mma_bf16(tmem + kAcc0 + s * BV, ad, bd, id, 1);
        }
        mma_commit(ctx.bar(kMmaS));
        mma_commit(ctx.bar(kEmpty0 + s));  // the stage may be refilled once this retires
      }
      ctx.wait(kMmaS, sph++ & 1);
      tc_fence_after();
      {
        float a[32];
        if (t < 64) {  // E rows -> bf16 operand
#pragma unroll
          for (int hh = 0; hh < BV / 32; ++hh) {
            tmem_ld32(tmem + lane_base + kAcc0 + s * BV + 32 * hh, a);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float v[8];
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) v[jj] = a[8 * q + jj];
              st8(sbase + L::kEb + sw128(t, 4 * hh + q), v);
            }
          }
        } else {  // output rows
          const int i = t - 64;
          __nv_bfloat16 *orow = p.out + ((size_t)(t0 + i) * H + h) * DV + tile * BV;
#pragma unroll
          for (int hh = 0; hh < BV / 32; ++hh) {
            tmem_ld32(tmem + lane_base + kAcc0 + s * BV + 32 * hh, a);
            if (i < len) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                float v[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) v[jj] = p.scale * a[8 * q + jj];
                *reinterpret_cast<uint4 *>(orow + 32 * hh + 8 * q) = pack8(v);
              }
            }
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_sync(2, 128);
      // a4: Kend^T E -> D4
      if (t == 0) {
        tc_fence_after();
        constexpr uint32_t id = idesc_bf16(128, BV, true, true);
        const uint32_t kend = sbase + L::kKend + s * 16384;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const uint64_t ad = sdesc_sw128(kend + k4 * 2048, 8192, 1024);
          const uint64_t bd = sdesc_sw128(sbase + L::kEb + k4 * 2048, 8192, 1024);
          mma_bf16(tmem + kD4, ad, bd, id, k4 > 0);
        }
        mma_commit(ctx.bar(kMmaS));
      }
      ctx.wait(kMmaS, sph++ & 1);
      tc_fence_after();
      {
        const float gm = gamma[s * 128 + t];
        float a[32];
#pragma unroll
        for (int hh = 0; hh < BV / 32; ++hh) {
          tmem_ld32(tmem + lane_base + kD4 + 32 * hh, a);
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) S[32 * hh + jj] = fmaf(gm, S[32 * hh + jj], a[jj]);
        }
      }
      tc_fence_before();
      bar_sync(2, 128);
      if (t == 0) mbar_arrive(ctx.bar(kDone0 + s));
    }
    if (p.final_state) {
#pragma unroll
      for (int j = 0; j < BV; j += 4)
        *reinterpret_cast<float4 *>(p.final_state + soff + j) =
            make_float4(S[j], S[j + 1], S[j + 2], S[j + 3]);
    }
    if (t == 0) {
      mma_commit(ctx.bar(kFinS));
      mbar_wait(ctx.bar(kFinS), 0, kWaitCycles);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// [T, H, 128] bf16 tensor, boxes of 64 channels x 1 head x 64 tokens, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int T, int H) {
  const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t strides[2] = {128 * 2, (cuuint64_t)H * 128 * 2};
  const cuuint32_t box[3] = {64, 1, 64};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool chunk_tc_supported(int d_k, int d_v, bool bf16) { return bf16 && d_k == 128 && d_v == 128; }
size_t chunk_tc_scratch_bytes(int, int, int, int) { return 0; }

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t stream) {
  if (!chunk_tc_supported(a.d_k, a.d_v, a.bf16)) return cudaErrorInvalidValue;
  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mg, mv;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mg, 0, sizeof(mg));
  memset(&mv, 0, sizeof(mv));
  if (a.total_tokens > 0) {
    if (!make_map(&mq, a.q, a.total_tokens, a.num_heads) ||
        !make_map(&mk, a.k, a.total_tokens, a.num_heads) ||
        !make_map(&mg, a.g, a.total_tokens, a.num_heads) ||
        !make_map(&mv, a.v, a.total_tokens, a.num_heads))
      return cudaErrorInvalidValue;
  }
  TcParams prm;
  prm.beta = static_cast<const __nv_bfloat16 *>(a.beta);
  prm.init_state = a.init_state;
  prm.cu_seqlens = a.cu_seqlens;
  prm.out = static_cast<__nv_bfloat16 *>(a.out);
  prm.final_state = a.final_state;
  prm.status = a.status;
  prm.H = a.num_heads;
  prm.scale = a.scale;
  prm.flags = a.test_flags;
  const long long blocks = (long long)a.num_seqs * a.num_heads * (DV / BV);
  if (blocks == 0) return cudaSuccess;
  cudaError_t err = cudaFuncSetAttribute(kda_chunk_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (err != cudaSuccess) return err;
  kda_chunk_tc_kernel<<<(unsigned)blocks, kThreads, L::kAlloc, stream>>>(mq, mk, mg, mv, prm);
  return cudaGetLastError();
}

}  // namespace kda
