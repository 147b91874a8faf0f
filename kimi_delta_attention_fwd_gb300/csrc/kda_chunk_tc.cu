// Chunkwise KDA prefill on the sm_103a tensor cores (tcgen05 + TMA + TMEM).
//
// The chunk algebra is the chunkwise schedule of "Kimi Delta Attention (KDA)"
// (brain.bigb.es, section on the two schedules) in the WY / UT form of the
// chunked DeltaNet section of "22580: от GPT-2 до Kimi K3", for the d_k x d_v
// state layout.  For a chunk of C = 64 rows with incoming state S, G = the
// chunk-local inclusive cumsum of g (per key channel) and gamma = exp(G_last),
// the write strengths beta folded into the rows of K and V:
//
//   Kb  = diag(beta) K * exp(G)   Qh = Q * exp(G)   Kc = K * exp(-G)   Vb = diag(beta) V
//   [Kb; Qh] Kc^T              -> rows: A^kk (j < i, beta_i included), A^qk (j <= i)
//   T   = (I + A^kk)^-1                                (fp32 triangular solve)
//   W   = T Kb                                         ([T; A^qk] Kb, rows 0-63)
//   with E = U - W S, U = T Vb and X = Qh S + A^qk Vb, all transposed (d_v rows):
//   [(E - Vb)^T | X^T] = Vb^T [T; A^qk]^T - Vb^T [I | 0] + S^T [-W; Qh]^T
//   O^T / s            = X^T + (E - Vb)^T A^qk^T       (= (Qh S + A^qk E)^T)
//   S^T <- (S^T + (E - Vb)^T Kc + Vb^T Kc) Diag(gamma) (= gamma (S + Kc^T E), transposed)
//
// The output is the inter-chunk term Qh S plus the masked intra-chunk product
// A^qk applied to the new values E.  E - Vb is the operand the state side rounds
// to bf16 for both of its last products: the Vb^T A^qk^T and Vb^T Kc terms it is
// combined with are formed from Vb itself, so they add back what was subtracted.
// E - Vb = (T - I) Vb - W S scales with beta like E does, so its bf16 rounding
// stays small against E for small write strengths too.  (E - Vb)^T in bf16 is the A
// operand of the state side's last products, in tensor memory.
//
// The state side works on S^T, one d_v row per TMEM lane: S^T in bf16 is the A
// operand (in tensor memory) of its first product, and each of its products covers
// the whole d_v = 128 in one M = 128 instruction.  One CTA therefore owns a
// (sequence, head) and does the state-independent work of each chunk once.
//
// exp(G) <= 1 and exp(-G) <= exp(-G_last); every factor stays finite as long
// as a chunk's total log decay per channel is above -80.  The state side checks
// it per chunk; a sequence-head that leaves the range is marked in the
// workspace's per-pair flags, its outputs and final state are left unwritten,
// and the launcher's next kernel recomputes it token by token with exact decays
// (without room for the flags the call reports KDA_ERR_GATE_RANGE instead).  The
// products use bf16 operands with fp32 accumulation in tensor memory; the state,
// the cumsum and the solve are fp32.
//
// One CTA walks the chunks of its (sequence, head) in order.  Warp roles:
//   warps 0-7    K-side: two groups of 4 warps on alternating chunks, everything
//                that does not depend on S; group kw owns stage kw
//   warps 8-15   state side: S^T (fp32) in registers, thread (d_v row, key-channel
//                half); the state-dependent products of each chunk
// The TMA loads that refill a stage are issued by whoever releases each part: a
// K-side group its g tile (after the solve), the state side its k and q tiles
// (after its first product has read [-W; Qh]) and its v tile (after the chunk's
// outputs, staged there, have been stored by TMA).  With few sequence-heads, one or
// two more CTAs per sequence-head run the solve of its chunks ("Solve helpers" below);
// a few long sequences with few heads are cut into segments that run side by side and are
// chained through their affine state maps ("Segment-parallel scan" below).
// Every wait on an mbarrier is bounded; on timeout the CTA records
// KDA_ERR_DEVICE_TIMEOUT in the status word and runs to completion without
// waiting again (outputs are then undefined, nothing blocks or faults).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <type_traits>

#include "kda_internal.h"
#include "kda_tc_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int C = 64;
constexpr int DK = 128;
constexpr int DV = 128;
constexpr int kThreads = 512;  // 8 K-side warps, 8 state-side warps
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr uint32_t kWaitCycles32 = 2000000000u;  // ~1 s: the bound of the in-loop waits (32-bit clock)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMinGamma = 1.8e-35f;  // about exp(-80): the state side checks gamma = exp(G_last)

// Solve helpers (few sequence-heads).  With at most 76 (sequence, head) pairs and
// room for the ring, the launch is cooperative (all CTAs resident) and each pair
// gets hpp = 2 (at most 50 pairs) or 1 helper CTAs beside its tile: K-side group kw
// of helper hp solves the chunks c = hp + hpp kw + 2 hpp i (the state-independent
// [T; A^qk]) and hands each to the tile through a ring in the workspace, slot
// c % 4 holding chunk c's 16 KiB shared-memory image.  Each slot has two words: the
// last chunk published + 1 (a release store after the image) and the number of
// reads so far (a release add by the tile once its copy is in shared memory); a
// helper overwrites a slot when the tile has read the chunk four before.
// Every wait on these words is bounded.
constexpr int kRingSlots = 4;
constexpr uint32_t kRingSlotBytes = 16384;
constexpr int kHelperMaxPairs = 76;  // (1 + helpers) CTAs per sequence-head, one per SM, all resident
constexpr int kGl = 3;               // G_last slots: chunk c + 3 reuses chunk c's

// Compact fp32 layout of the 64 x 64 unit-lower-triangular solve (12 KB):
// the four 16 x 16 diagonal blocks, the sub-diagonal blocks (1,0) and (3,2), and
// the lower-left 32 x 32 block; row strides keep 16-byte alignment and spread
// the rows of a column over the shared-memory banks.
constexpr int kSdLd = 20, kSlLd = 36, kYLd = 40;
__device__ __forceinline__ int sd_idx(int blk, int r, int c) { return (blk * 16 + r) * kSdLd + c; }
__device__ __forceinline__ int so_idx(int blk, int r, int c) { return (blk * 16 + r) * kSdLd + c; }
__device__ __forceinline__ int sl_idx(int r, int c) { return r * kSlLd + c; }

// Shared memory map (offsets from a 1024-byte aligned base).
struct L {
  // stage: [k ch0-63 | q ch0-63] [k ch64-127 | q ch64-127] [g ch0-63] [g ch64-127]
  //        [v ch0-63] [v ch64-127];
  // the g area later holds the fp32 A^kk / T in the compact solve layout; the k rows
  // hold Kb, then -W; the q rows Qh ([-W; Qh] is the B operand of the state product);
  // the v area holds Vb, then the chunk's outputs for their TMA store
  static constexpr uint32_t kKQ1 = 16384, kQoff = 8192, kG = 32768, kV = 49152;
  static constexpr uint32_t kStageBytes = 65536;
  static constexpr uint32_t kKc = 2 * kStageBytes;      // 3 x Kc [ch0-63 | ch64-127], slot = chunk % 3
  static constexpr uint32_t kTP = kKc + 3 * 16384;        // 2 x [T rows 0-63 | A^qk rows 64-127]
  static constexpr uint32_t kNegI = kTP + 2 * 16384;      // -I, 64 x 64 bf16 (K-major B operand)
  static constexpr uint32_t kGlast = kNegI + 8192;        // gamma = exp(G_last) [kGl][128]
  static constexpr uint32_t kBars = kGlast + kGl * 512;   // mbarriers
  static constexpr uint32_t kMisc = kBars + 256;          // tmem slot, abort / skip flags, issued loads
  static constexpr uint32_t kTotal = kMisc + 64;
  static constexpr uint32_t kAlloc = kTotal + 1024;
};
static_assert(L::kKc % 1024 == 0 && L::kTP % 1024 == 0 && L::kNegI % 1024 == 0,
              "operand tiles must be 1024-byte aligned");
static_assert(L::kAlloc <= 232448, "shared memory budget");

// mbarrier slots (count 1 each; [s] = stage / K-side group, [b] = Kc / G_last slot)
enum : uint32_t {
  kFullQ0 = 0, kFullG0 = 2, kFullK0 = 4, kFullV0 = 6,  // part of stage s loaded
  kReady0 = 8,     // K-side -> state side: the chunk's state-independent operands are complete
  kGmRead0 = 10,   // state side -> K-side: G_last[b] has been read (3 slots)
  kKcFree0 = 13,   // state side -> K-side: Kc[b] and TP of that chunk read (3 slots)
  kMmaK0 = 16, kMmaS = 18, kFinK0 = 19, kFinS = 21, kNever = 22,
  kTPReady0 = 23,  // K-side -> state side: [T; A^qk] (and Vb, with helpers) of the stage are complete
  kNumBars = 25
};
static_assert(kNumBars * 8 <= 256, "mbarrier area");

// TMEM columns
//   [128 kw, +128)  K-side group kw: G, then D1 (+0), then D2 (-W before the epilogue)
//   [256, 320)      S^T in bf16 pairs: the A operand of the state product
//   [320, 448)      [(E - Vb)^T | X^T], then [. | O^T / s]
//   [256, 384)      (Kc^T E)^T: over S^T and the first half of the above, once both are read
//   [448, 480)      [Ltri; Ltri] in bf16 pairs: the A operand of the cumsum product
//   [480, 512)      (E - Vb)^T in bf16 pairs: the A operand of the state side's last products
constexpr uint32_t kRA = 256, kRD1 = 320, kRD4 = 256, kRLtri = 448, kREV = 480;

struct TcParams {
  const __nv_bfloat16 *beta;
  const __nv_bfloat16 *g_tok;  // [T, H] log alpha per (token, head) when gate == 1
  int gate;                    // 0: g per key channel (TMA), 1: per token (g_tok), 2: none
  int prep;                    // KDA_PREP_* bits: silu / L2 norm of q and k, sigmoid of beta,
                               // softplus of the gate
  float gate_scale;            // c of log alpha = -c softplus(x)
  int helpers_per_pair;        // 1 or 2 (solve-helper schedule)
  const float *init_state;
  const int32_t *cu_seqlens;
  __nv_bfloat16 *out;
  float *final_state;
  uint32_t *status;
  uint32_t *pair_flags;      // [P]: set for a pair whose decay left the range (or NULL)
  int T;                     // tokens in all (cu_seqlens must stay within [0, T])
  int H;
  float scale;
  int flags;  // bit 0: test hook, wait once on a barrier nothing arrives on
  int npairs;                // P, the number of (sequence, head) pairs
  uint8_t *ring;             // [P][kRingSlots][kRingSlotBytes]
  uint32_t *ring_flags;      // [P][kRingSlots][2]: chunk + 1 published, consumptions (zeroed)
  const int32_t *order;      // plain schedule: sequences longest first (CTA i takes sequence
                             // order[i / H], head i % H), or NULL for the given order
  int seq_stride;            // 1: sequence n spans cu_seqlens[n] .. cu_seqlens[n + 1]; 4 (the
                             // segment passes): cu_seqlens holds runs {first token, end token,
                             // kRun* mode, sequence} instead, order unused
  const uint32_t *head_skip; // runs: (sequence, head) pairs to skip ([N][H], fixed for the
                             // launch), or NULL
};

// Modes of a segment run (the segment-parallel scan of long sequences): V enters as zero
// (from the identity as start state the run then gives the segment's transfer matrix); the
// outputs are not stored; the run is skipped altogether.
constexpr int kRunZeroV = 1, kRunNoOut = 2, kRunSkip = 4;

// Global-memory hand-over between CTAs of one launch (all resident: cooperative launch).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_gpu_add(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

struct Ctx {
  uint32_t bars;
  volatile int *abort;
  uint32_t *status;
  __device__ __forceinline__ uint32_t bar(uint32_t i) const { return bars + 8 * i; }
  // Bounded wait on mbarrier i (about 1 s of SM clock); a timeout is recorded in the
  // CTA's abort flag, which ends every later wait at once and is reported in the status
  // word when the CTA leaves (one site, so each inlined wait stays small).
  __device__ __forceinline__ void wait(uint32_t i, uint32_t parity) const {
    if (*abort || mbar_try_wait(bar(i), parity)) return;
    const uint32_t t0 = static_cast<uint32_t>(clock());
    while (!mbar_try_wait(bar(i), parity)) {
      if (static_cast<uint32_t>(clock()) - t0 > kWaitCycles32) {
        *abort = 1;
        return;
      }
    }
  }
  // Bounded wait until the global word *w (written by another CTA) reaches target;
  // a timeout anywhere in the launch (the status word) ends it at once.
  __device__ __forceinline__ void wait_global(const uint32_t *w, uint32_t target) const {
    if (*abort) return;
    const long long t0 = clock64();
    while (ld_acquire_gpu(w) < target) {
      if (*reinterpret_cast<volatile uint32_t *>(status) == kStatusTimeout ||
          clock64() - t0 > kWaitCycles) {
        *abort = 1;
        atomicCAS(status, 0u, kStatusTimeout);
        return;
      }
      __nanosleep(64);
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
__device__ __forceinline__ uint32_t tf32_bits(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// silu(x) = x sigmoid(x) = x (1 + tanh(x / 2)) / 2 on a bf16 pair, every step in bf16
// (the hardware tanh and three bf16x2 operations: a relative error of a few 2^-9 per
// element, about 0.3 % over a row, against the 2 % tolerance of bf16 I/O)
__device__ __forceinline__ uint32_t silu_bf16x2(uint32_t x) {
  constexpr uint32_t kHalf2 = 0x3F003F00u;  // (0.5, 0.5) in bf16
  uint32_t t, sg;
  asm("tanh.approx.bf16x2 %0, %1;" : "=r"(t) : "r"(mul_bf16x2(x, kHalf2)));
  asm("fma.rn.bf16x2 %0, %1, %2, %2;" : "=r"(sg) : "r"(t), "r"(kHalf2));
  return mul_bf16x2(x, sg);
}
// Sums of squares of the 32 rows rbase .. rbase + 31 of two 64-row bf16 tiles (k and q)
// in the stage layout (two 64-channel halves kKQ1 apart, 128-byte rows, 128-byte
// swizzle), as the diagonals of X X^T on the warp-level tensor instructions: per tile
// and 16-row block, eight 16 x 16 slices of X, each one ldmatrix and two MMAs whose B
// operand is the slice's own rows; the four accumulator chains are interleaved.  Exact
// bf16 products, fp32 sums.  Lane l gets the sums of row rbase + l.
__device__ __forceinline__ void row_sumsq32x2(uint32_t tk, uint32_t tq, int rbase, int lane,
                                              float &ssk, float &ssq) {
  const int m = lane >> 3, rr = lane & 7;  // ldmatrix: this lane addresses row rr of matrix m
  const int g = lane >> 2;                 // MMA fragment row of this lane
  float d[2][2][2][4];                     // [tile][block][column half][fragment]
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 4; ++e) d[i][b][h][e] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {  // 16 channels per step
    const uint32_t chunk = static_cast<uint32_t>(2 * (ks & 3) + (m >> 1));
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const uint32_t row = static_cast<uint32_t>(rbase + 16 * b + rr + 8 * (m & 1));
      const uint32_t off = (ks >> 2) * L::kKQ1 + sw128(row, chunk);
      uint32_t ak[4], aq[4];
      ldmatrix_x4(ak, tk + off);
      ldmatrix_x4(aq, tq + off);
      mma_bf16_16x8x16(d[0][b][0], ak, ak[0], ak[2]);  // columns = rows 0-7 of the block
      mma_bf16_16x8x16(d[0][b][1], ak, ak[1], ak[3]);  // columns = rows 8-15
      mma_bf16_16x8x16(d[1][b][0], aq, aq[0], aq[2]);
      mma_bf16_16x8x16(d[1][b][1], aq, aq[1], aq[3]);
    }
  }
  // the diagonal: lane 4 g + g / 2 holds rows g (column half 0) and g + 8 (half 1)
  const int want = lane & 15, gw = want & 7, src = 4 * gw + (gw >> 1), bw = lane >> 4;
  float out[2] = {0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const float lo = (g & 1) ? d[i][b][0][1] : d[i][b][0][0];
      const float hi = (g & 1) ? d[i][b][1][3] : d[i][b][1][2];
      const float vlo = __shfl_sync(0xffffffffu, lo, src);
      const float vhi = __shfl_sync(0xffffffffu, hi, src);
      if (bw == b) out[i] = want >= 8 ? vhi : vlo;
    }
  ssk = out[0];
  ssq = out[1];
}

// kSched = false: every CTA is a (sequence, head) tile that solves its own chunks
// (the plain schedule); true: CTAs P .. (1 + hpp) P - 1 are solve helpers for the
// first P.  kPrep: the input steps of TcParams::prep are compiled in (a call without
// them runs the instantiation that has none of their code).  kChan: g is one log alpha per
// key channel, compiled in (the per-token and no-gate code is left out, which keeps the
// hot loops smaller for the instruction cache); without it the gate mode is read from
// TcParams::gate.
template <bool kSched, bool kPrep, bool kChan>
__global__ void __launch_bounds__(kThreads, 1)
    kda_chunk_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_g,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  float *glast = reinterpret_cast<float *>(smem + L::kGlast);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kMisc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 4);
  // set by the state side once this pair's decay has left the range: nothing more is stored
  // bit 0: no chunk runs and nothing is written; bit 1: the outputs are not stored
  volatile int *skip_flag = reinterpret_cast<volatile int *>(smem + L::kMisc + 8);
  // the last chunk loaded into each stage part [stage][q, g, k, v] (-1: none), for the drain
  volatile int *issued = reinterpret_cast<volatile int *>(smem + L::kMisc + 16);
  // the token coordinate of the V tile of chunk 0: bos, or far below zero when V enters as
  // zero (the tiles then lie wholly outside the tensor and TMA fills them with zeros)
  volatile int *v_tok0 = reinterpret_cast<volatile int *>(smem + L::kMisc + 48);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  // roles: a tile CTA (one per pair) runs everything, or with helpers takes each chunk's
  // [T; A^qk] from the ring; a helper (pair, hp) runs the chunk solve of the chunks
  // c = hp + hpp kw + 2 hpp i of its K-side group kw and publishes it
  const int P = p.npairs;
  const bool helper = kSched && (int)blockIdx.x >= P;  // (a tile "fed" by helpers otherwise)
  const int hpp = kSched ? p.helpers_per_pair : 1;
  const int hb = (int)blockIdx.x - P;
  const int hp = helper ? hb % hpp : 0;
  const int pair = helper ? hb / hpp
                          : (kSched || !p.order ? (int)blockIdx.x
                                                : p.order[blockIdx.x / p.H] * p.H + (int)(blockIdx.x % p.H));
  // the chunks a stage / K-side group kw takes: c = c_first(kw) + i * c_step, phase i & 1
  const int c_step = helper ? 2 * hpp : 2;
  const int c_shift = helper && hpp == 2 ? 2 : 1;
  uint32_t *rflags = kSched ? p.ring_flags + (size_t)pair * kRingSlots * 2 : nullptr;
  uint8_t *rdata = kSched ? p.ring + (size_t)pair * kRingSlots * kRingSlotBytes : nullptr;
  const int H = p.H;
  const int n = pair / H, h = pair % H;
  // a pair whose offsets are out of order or out of range runs no chunk and writes nothing
  // (its skip flag is set below); bos and eos stay reloadable from cu_seqlens
  const bool seg_run = p.seq_stride == 4;
  const int32_t *bnd = p.cu_seqlens + (seg_run ? 4 * n : n);
  const int bos = bnd[0];
  const bool seq_ok = 0 <= bos && bos <= bnd[1] && bnd[1] <= p.T;
  // a segment run is skipped when its table says so, or when an earlier pass marked its head
  // for the exact recomputation (whose outputs and final state replace the run's); the tile
  // and its solve helpers must agree, so the marks come from a copy taken before the launch
  const bool run_skip = seg_run && ((bnd[2] & kRunSkip) || (p.head_skip && p.head_skip[bnd[3] * H + h]));
  const int eos = seq_ok && !run_skip ? bnd[1] : bos;
  const int nchunks = (eos - bos + C - 1) / C;

  Ctx ctx{sbase + L::kBars, abort_flag, p.status};

  // TMA loads of the stage parts of chunk c (stage s), each completing on its full barrier
  auto stage_at = [&](int st_idx) { return sbase + st_idx * L::kStageBytes; };
  auto load_q = [&](int sidx, int c) {
    const uint32_t fb = ctx.bar(kFullQ0 + sidx), st = stage_at(sidx);
    mbar_arrive_expect_tx(fb, 16384);
    tma_load_3d(st + L::kQoff, &tm_q, fb, 0, h, bos + c * C);
    tma_load_3d(st + L::kKQ1 + L::kQoff, &tm_q, fb, 64, h, bos + c * C);
    issued[4 * sidx + 0] = c;
  };
  auto load_g = [&](int sidx, int c) {
    const uint32_t fb = ctx.bar(kFullG0 + sidx), st = stage_at(sidx);
    if (kChan || p.gate == 0) {
      mbar_arrive_expect_tx(fb, 16384);
      tma_load_3d(st + L::kG, &tm_g, fb, 0, h, bos + c * C);
      tma_load_3d(st + L::kG + 8192, &tm_g, fb, 64, h, bos + c * C);
    } else {
      mbar_arrive(fb);  // no g tile: the part's phase still completes
    }
    issued[4 * sidx + 1] = c;
  };
  auto load_k = [&](int sidx, int c) {
    const uint32_t fb = ctx.bar(kFullK0 + sidx), st = stage_at(sidx);
    mbar_arrive_expect_tx(fb, 16384);
    tma_load_3d(st, &tm_k, fb, 0, h, bos + c * C);
    tma_load_3d(st + L::kKQ1, &tm_k, fb, 64, h, bos + c * C);
    issued[4 * sidx + 2] = c;
  };
  auto load_v = [&](int sidx, int c) {
    const uint32_t fb = ctx.bar(kFullV0 + sidx), st = stage_at(sidx);
    mbar_arrive_expect_tx(fb, 16384);
    const int tok = *v_tok0 + c * C;
    tma_load_3d(st + L::kV, &tm_v, fb, 0, h, tok);
    tma_load_3d(st + L::kV + 8192, &tm_v, fb, 64, h, tok);
    issued[4 * sidx + 3] = c;
  };

  if (tid == 0) {
    *abort_flag = 0;
    *skip_flag = (seq_ok && !run_skip ? 0 : 1) | (seg_run && (bnd[2] & kRunNoOut) ? 2 : 0);
    *v_tok0 = seg_run && (bnd[2] & kRunZeroV) ? -(1 << 30) : bos;  // T < 2^30: c C - 2^30 < 0
    for (int i = 0; i < 8; ++i) issued[i] = -1;
    if (!seq_ok) atomicCAS(p.status, 0u, kStatusSeqlens);
    for (uint32_t i = 0; i < kNumBars; ++i) mbar_init(ctx.bar(i), 1);
    fence_mbar_init();
    if (blockIdx.x == 0) p.status[2] = seg_run ? kSchedSegments : (kSched ? kSchedHelpers : kSchedPlain);
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp < 4) {
    // the cumsum product's constant A operand [Ltri; Ltri] (Ltri[r][u] = (u <= r)) in
    // tensor memory, bf16 pairs: lane m holds row m mod 64
    const int r = tid & 63;
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 32; ++j)
      w[j] = (2 * j <= r ? 0x3F80u : 0u) | ((2 * j + 1 <= r ? 0x3F80u : 0u) << 16);
    tmem_st32(tmem + (static_cast<uint32_t>(32 * warp) << 16) + kRLtri, w);
  } else if (warp >= 8 && warp < 10) {
    // -I (64 x 64, bf16, K-major rows): the state side subtracts Vb^T with it
    const int r = tid - 256;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = (8 * j + 2 * e == r ? 0xBF80u : 0u) | ((8 * j + 2 * e + 1 == r ? 0xBF80u : 0u) << 16);
      st_shared_v4(sbase + L::kNegI + sw128(r, j), w[0], w[1], w[2], w[3]);
    }
    fence_async_smem();
  } else if (tid == 128 || tid == 160) {
    // the first chunk of each stage, loaded by one thread per stage
    const int sidx = tid == 128 ? 0 : 1;
    if (sidx == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_g);
      tma_prefetch_desc(&tm_v);
    }
    const int c0 = helper ? hp + hpp * sidx : sidx;
    if (c0 < nchunks) {
      load_g(sidx, c0);
      load_k(sidx, c0);
      load_q(sidx, c0);
      if (!helper) load_v(sidx, c0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // Register split: the state side holds 64 fp32 state values per thread.  The launch
  // gives every thread 128 registers (512 x 128 = 65,536); the K-side warpgroups hand
  // 8 each back and the state side takes them: 256 x 120 + 256 x 136 = 65,536.
  if (warp < 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 120;" ::: "memory");
    // ------------------------------------------------------------ K-side
    // Two groups of 4 warps; group kw takes the chunks c = kw, kw + 2, ... and
    // owns stage kw, TP[kw] and TMEM columns [128 kw, 128 kw + 128), so the
    // dependent chain of one chunk overlaps the other group's chunk.  Kc rotates
    // over three slots (chunk % 3).
    // A helper's groups take c = hp + hpp kw + 2 hpp i, run the gate, a2 and the solve,
    // and publish [T; A^qk]; a tile fed by helpers runs the gate and takes [T; A^qk]
    // from the ring in place of a2 and the solve.
    const int kw = warp >> 2;
    const int t = tid & 127;            // thread within the group
    const int wq = warp & 3;            // TMEM lane quarter of this warp
    const int row = 32 * wq + (t & 31); // TMEM lane = row of an M = 128 result (== t)
    const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
    const uint32_t bar_id = kw ? 3u : 1u;
    const uint32_t tm = tmem + 128u * kw;  // G, then D1 (+0), then D2
    const uint32_t st = sbase + kw * L::kStageBytes;
    const uint32_t tp = sbase + L::kTP + kw * 16384;
    // compact fp32 solve layout in the stage's g area (after the cumsum product has read g)
    float *Sd = reinterpret_cast<float *>(smem + kw * L::kStageBytes + L::kG);  // [4][16][20]
    float *So = Sd + 4 * 16 * kSdLd;                                            // [2][16][20]
    float *Sl = So + 2 * 16 * kSdLd;                                            // [32][36]
    float *Ys = reinterpret_cast<float *>(smem + L::kTP + kw * 16384);          // TP rows 0-63
    const uint32_t mma_bar = ctx.bar(kMmaK0 + kw);
    // g per key channel (G by the cumsum product below): compiled in, or read from p.gate
    const bool chan = kChan || p.gate == 0;
    // g holds gate logits: each group turns its g tile into -c softplus(g) in place before
    // the cumsum product, which is then issued at the top of the chunk (not ahead)
    const bool gsp = kPrep && chan && (p.prep & kPrepGSoftplus);
    // a1: G = [Ltri; Ltri] g on the tensor cores, straight from the TMA'd g tile with
    // the constant operand in tensor memory: the chunk-local inclusive cumsum per
    // channel (rows 64-127 repeat rows 0-63)
    auto issue_cumsum = [&]() {
      tc_fence_after();
      constexpr uint32_t id = idesc_bf16(128, 128, false, true);
      const uint32_t bg = sdesc_lo(st + L::kG, 8192);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
        mma_ts(tm, tmem + kRLtri + 8u * k4, bg + 128 * k4, sdesc_hi(1024), id, k4 > 0);
      mma_commit(mma_bar);
    };
    if ((p.flags & 1) && tid == 0) {
      // test hook: a wait that can only time out
      if (!mbar_wait(ctx.bar(kNever), 0, 2000000LL)) {
        *abort_flag = 1;
        atomicCAS(p.status, 0u, kStatusTimeout);
      }
    }
    // The chunk loop, compiled once per role: a solve helper's and a tile's copies each
    // leave out the other's code (a helper schedule launch runs both kinds of CTA).
    auto kloop = [&](auto role) {
    constexpr bool helper = decltype(role)::value;
    constexpr bool fed = kSched && !helper;
    uint32_t kph = 0;
    // chunks of this group: c = kw, kw + 2, ...; in a helper c = hp + hpp kw + 2 hpp i
    for (int c = helper ? hp + hpp * kw : kw; c < nchunks; c += c_step) {
      const int s = kw;
      const int t0 = bos + c * C;
      const int len = min(C, eos - t0);
      const int kb = helper ? kw : c % 3;  // Kc slot (a helper's own two are read by its a2 only)
      const uint32_t kcb = sbase + L::kKc + kb * 16384;
      const int slot = c & (kRingSlots - 1);  // ring slot of this chunk's [T; A^qk]
      if (t == 0 && c + c_step < nchunks) {
        // the group's next chunk into L2: its stage loads, issued when each part is
        // released, then wait for L2 rather than HBM
        const int tn = bos + (c + c_step) * C;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          tma_prefetch_3d(&tm_k, 64 * x, h, tn);
          tma_prefetch_3d(&tm_q, 64 * x, h, tn);
          if (kChan || p.gate == 0) tma_prefetch_3d(&tm_g, 64 * x, h, tn);
          if (!helper) tma_prefetch_3d(&tm_v, 64 * x, h, tn);
        }
      }
      // beta of this thread's row (row t mod 64 of the chunk; 0 past the sequence end),
      // folded into Kb and Vb; loaded early to hide the global latency
      const int rb = t & 63;
      const float braw = rb < len ? __bfloat162float(p.beta[(size_t)(t0 + rb) * H + h]) : 0.f;
      // beta given as a logit: sigmoid (rows past the end keep 0)
      const float brow = kPrep && (p.prep & kPrepBetaSigmoid) && rb < len
                             ? fast_rcp(1.f + fast_exp2(-kLog2e * braw)) : braw;
      // one thread polls the mbarriers, the others park on the named barrier
      const int it = c >> c_shift;                // this group's it-th chunk
      const uint32_t cur = it & 1;                // parity of this chunk's loads
      // a1 with one log alpha per (token, head): G_r is one inclusive scan over the
      // chunk's rows (rows r and 32 + r of two per-warp scans), the same for every channel
      float g_row = 0.f;
      if (!kChan && p.gate == 1) {
        const int lane = t & 31;
        float ga = lane < len ? gate_log<kPrep>(__bfloat162float(p.g_tok[(size_t)(t0 + lane) * H + h]),
                                                p.prep, p.gate_scale) : 0.f;
        float gb = 32 + lane < len ? gate_log<kPrep>(__bfloat162float(p.g_tok[(size_t)(t0 + 32 + lane) * H + h]),
                                                     p.prep, p.gate_scale) : 0.f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float xa = __shfl_up_sync(0xffffffffu, ga, o), xb = __shfl_up_sync(0xffffffffu, gb, o);
          if (lane >= o) { ga += xa; gb += xb; }
        }
        g_row = (wq & 1) ? __shfl_sync(0xffffffffu, ga, 31) + gb : ga;  // row r = 32 (wq & 1) + lane
      }
      if (gsp) {
        // -c softplus of the chunk's gate logits, in place (bf16), then the cumsum product
        if (t == 0) ctx.wait(kFullG0 + s, cur);
        bar_sync(bar_id, 128);
        const uint32_t grow = st + L::kG + (t >> 6) * 8192;  // row t mod 64, channel half t / 64
#pragma unroll 2
        for (int j = 0; j < 8; ++j) {
          const uint32_t addr = grow + sw128(t & 63, j);
          float f[8];
          unpack8(ld_shared_v4(addr), f);
#pragma unroll
          for (int e = 0; e < 8; ++e) f[e] = neg_softplus(f[e], p.gate_scale);
          st8(addr, f);
        }
        fence_async_smem();
        bar_sync(bar_id, 128);
        if (t == 0) issue_cumsum();
      }
      if (t == 0) {
        if (chan) {
          if (it == 0 && !gsp) {  // later chunks had their cumsum product issued at the end of the previous one
            ctx.wait(kFullG0 + s, cur);
            issue_cumsum();
          }
          ctx.wait(kMmaK0 + kw, kph & 1);
        }
        ctx.wait(kFullK0 + s, cur);
        ctx.wait(kFullQ0 + s, cur);
        if (!helper) {
          if (c >= 3) ctx.wait(kKcFree0 + kb, ((c / 3) - 1) & 1);  // chunk c - 3 is done with Kc[kb]
          // chunk c - kGl is done with G_last[c % kGl]
          if (c >= kGl) ctx.wait(kGmRead0 + c % kGl, ((c / kGl) - 1) & 1);
        }
      } else if (fed && t == 32) {
        // meanwhile another thread acquires the chunk's ring slot (published by a helper);
        // the barrier below orders every thread's later reads of it after this
        ctx.wait_global(rflags + 2 * slot, static_cast<uint32_t>(c + 1));
      }
      if (chan) ++kph;
      bar_sync(bar_id, 128);
      tc_fence_after();

      // Each thread owns row r and 64 channels of the elementwise decay work.
      const int r = row & 63, half = row >> 6;
      const uint32_t kq = st + half * L::kKQ1;
      // Rows past the sequence end are zeroed and get unit factors (G log2 e taken
      // as 0), so no exp(-G) of the next sequence's decays can overflow there.
      const bool valid = r < len;
      const float lg2 = valid ? kLog2e : 0.f;
      // Optional input steps on the row's q and k: silu in place, then the norms.  With the
      // silu the sums of squares come from the values already in registers (the two halves
      // of a row meet in the stage's g area, read by the cumsum product already and written
      // by the solve only after the next barrier); without it, from the warp-level tensor
      // instructions (row_sumsq32x2), which needs no exchange.  1 / ||k|| goes into the
      // factors of Kb and Kc, 1 / ||q|| into those of Qh.
      const bool norm = kPrep && (p.prep & kPrepL2);
      float rk = 1.f, rq = 1.f, lk = 0.f;  // 1 / ||k_row||, 1 / ||q_row||, log2(rk)
      float ssk = 0.f, ssq = 0.f;
      if (kPrep && (p.prep & kPrepSilu)) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t addr = kq + sw128(r, j);
          const uint4 kw4 = ld_shared_v4(addr), qw4 = ld_shared_v4(addr + L::kQoff);
          const uint4 ks4 = make_uint4(silu_bf16x2(kw4.x), silu_bf16x2(kw4.y), silu_bf16x2(kw4.z),
                                       silu_bf16x2(kw4.w));
          const uint4 qs4 = make_uint4(silu_bf16x2(qw4.x), silu_bf16x2(qw4.y), silu_bf16x2(qw4.z),
                                       silu_bf16x2(qw4.w));
          st_shared_v4(addr, ks4.x, ks4.y, ks4.z, ks4.w);
          st_shared_v4(addr + L::kQoff, qs4.x, qs4.y, qs4.z, qs4.w);
          if (norm) {
            float fk[8], fq[8];
            unpack8(ks4, fk);
            unpack8(qs4, fq);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              ssk = fmaf(fk[e], fk[e], ssk);
              ssq = fmaf(fq[e], fq[e], ssq);
            }
          }
        }
        if (norm) {
          float *xch = Sd;
          xch[t] = ssk;
          xch[128 + t] = ssq;
          bar_sync(bar_id, 128);
          ssk += xch[t ^ 64];
          ssq += xch[128 + (t ^ 64)];
        }
      } else if (norm) {
        row_sumsq32x2(st, st + L::kQoff, 32 * (wq & 1), t & 31, ssk, ssq);  // row r = 32 (wq & 1) + lane
      }
      if (norm) {
        // 1 / max(||x||, 1e-12) = 2^(-log2(max(||x||^2, 1e-24)) / 2)
        lk = -0.5f * fast_log2(fmaxf(ssk, 1e-24f));
        rk = fast_exp2(lk);
        rq = fast_exp2(-0.5f * fast_log2(fmaxf(ssq, 1e-24f)));
      }
      const float bk = kPrep ? brow * rk : brow;  // Kb's row factor
      const uint32_t bb = pack_bf16x2(brow, brow);  // beta in bf16 pairs: Kb's factor is beta exp(G)
      // exp(G), beta exp(G) and exp(-G) of the row, when G is one per row
      uint32_t f_row = 0u, fk_row = 0u, fe_row = 0u;
      if (!chan) {
        const float dr = g_row * lg2;
        const float er = fast_exp2(dr), ier = fast_exp2(-dr);
        if constexpr (kPrep) {
          f_row = pack_bf16x2(rq * er, rq * er);
          fk_row = pack_bf16x2(bk * er, bk * er);
          fe_row = pack_bf16x2(rk * ier, rk * ier);
        } else {
          f_row = pack_bf16x2(er, er);
          fk_row = pack_bf16x2(brow * er, brow * er);
          fe_row = pack_bf16x2(ier, ier);
        }
      }
#pragma unroll 1
      for (int hh = 0; hh < 4; ++hh) {  // channels 64 half + 16 hh .. + 15
        float G[16];
        if (chan) {
          tmem_ld16(tm + lane_base + 64 * half + 16 * hh, G);
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) G[j] = g_row;
        }
        if (r == len - 1) {  // the chunk's last valid row: gamma = exp(G_last) for the state side
#pragma unroll
          for (int j = 0; j < 16; j += 4)
            *reinterpret_cast<float4 *>(glast + (c % kGl) * 128 + 64 * half + 16 * hh + j) =
                make_float4(fast_exp2(G[j] * kLog2e), fast_exp2(G[j + 1] * kLog2e),
                            fast_exp2(G[j + 2] * kLog2e), fast_exp2(G[j + 3] * kLog2e));
        }
        // bf16 pairs: exp(+-G) (and beta exp(G) for Kb) rounded to bf16, then one bf16
        // product per output pair.  With one G per row (a per-token gate, or none) the
        // factors are the row's own, formed once before the loop.
        auto products = [&](auto per_channel, auto normed) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const uint32_t addr = kq + sw128(r, 2 * hh + q);
            uint4 kw = ld_shared_v4(addr), qw = ld_shared_v4(addr + L::kQoff);
            if (!valid) kw = qw = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t kp[4] = {kw.x, kw.y, kw.z, kw.w}, qp[4] = {qw.x, qw.y, qw.z, qw.w};
            uint32_t kh[4], qh[4], kc[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t f = f_row, fk = fk_row, fe = fe_row;
              if constexpr (decltype(per_channel)::value) {
                const float d0 = G[8 * q + 2 * j] * lg2, d1 = G[8 * q + 2 * j + 1] * lg2;
                const float e0 = fast_exp2(d0), e1 = fast_exp2(d1);
                if constexpr (decltype(normed)::value) {
                  f = pack_bf16x2(rq * e0, rq * e1);
                  fk = pack_bf16x2(bk * e0, bk * e1);
                  fe = pack_bf16x2(fast_exp2(lk - d0), fast_exp2(lk - d1));
                } else {
                  f = pack_bf16x2(e0, e1);
                  fk = mul_bf16x2(f, bb);
                  fe = pack_bf16x2(fast_exp2(-d0), fast_exp2(-d1));
                }
              }
              kh[j] = mul_bf16x2(kp[j], fk);
              qh[j] = mul_bf16x2(qp[j], f);
              kc[j] = mul_bf16x2(kp[j], fe);
            }
            st_shared_v4(addr, kh[0], kh[1], kh[2], kh[3]);
            st_shared_v4(addr + L::kQoff, qh[0], qh[1], qh[2], qh[3]);
            st_shared_v4(kcb + half * 8192 + sw128(r, 2 * hh + q), kc[0], kc[1], kc[2], kc[3]);
          }
        };
        if (!chan) {
          products(std::false_type{}, std::false_type{});
        } else if constexpr (kPrep) {
          // one variant for every combination of steps (factors 1 and 0 without the
          // norm), which keeps a single copy of this loop in the instruction cache
          products(std::true_type{}, std::true_type{});
        } else {
          products(std::true_type{}, std::false_type{});
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_sync(bar_id, 128);

      if (fed) {
        // The chunk's [T; A^qk] comes from a helper through ring slot c % 4 (acquired
        // above): it is read into registers while TP[s] is still being read by chunk
        // c - 2's output product, then stored there.  The read is counted while the
        // W / U product runs.
        if (t == 0 && c + 2 < nchunks && !*abort_flag) load_g(s, c + 2);  // g was read by the cumsum product only
        const uint4 *src = reinterpret_cast<const uint4 *>(rdata + slot * kRingSlotBytes);
        uint4 w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = __ldcg(src + 128 * j + t);
        if (t == 0 && c >= 2) ctx.wait(kKcFree0 + (c - 2) % 3, ((c - 2) / 3) & 1);
        bar_sync(bar_id, 128);
#pragma unroll
        for (int j = 0; j < 8; ++j) st_shared_v4(tp + 16 * (128 * j + t), w[j].x, w[j].y, w[j].z, w[j].w);
      } else {
        // a2: [Kb; Qh] Kc^T -> D1 (rows 0-63: A^kk, rows 64-127: A^qk)
        if (t == 0) {
          tc_fence_after();
          constexpr uint32_t id = idesc_bf16(128, 64, false, false);
          const uint32_t akq = sdesc_lo(st, 16), bkc = sdesc_lo(kcb, 16);
#pragma unroll
          for (int k8 = 0; k8 < 8; ++k8)
            mma_ss(tm, akq + (k8 >> 2) * (L::kKQ1 >> 4) + 2 * (k8 & 3), sdesc_hi(1024),
                   bkc + (k8 >> 2) * 512 + 2 * (k8 & 3), sdesc_hi(1024), id, k8 > 0);
          mma_commit(mma_bar);
          ctx.wait(kMmaK0 + kw, kph & 1);
          if (helper) {  // Kb and Qh are read by a2 only in a helper: the next chunk's k and q
            if (c + c_step < nchunks && !*abort_flag) {
              load_k(s, c + c_step);
              load_q(s, c + c_step);
            }
          } else if (c >= 2) {
            // TP[s] was last read by chunk c - 2's output product, committed with its Kc release
            ctx.wait(kKcFree0 + (c - 2) % 3, ((c - 2) / 3) & 1);
          }
        }
        ++kph;
        bar_sync(bar_id, 128);
        tc_fence_after();
        // A^kk (fp32, strictly lower; beta is in Kb) goes to the stage's g area, which
        // the cumsum product has finished reading, in the compact solve layout
        // (diagonal 16-blocks, the two 16-wide sub-diagonal blocks, the lower-left
        // 32 x 32 block; the zero blocks above the diagonal are not stored).  T is
        // then computed in place there.
#pragma unroll 1
        for (int hh = 0; hh < 4; ++hh) {  // columns 16 hh .. 16 hh + 15
          float a[16];
          tmem_ld16(tm + lane_base + 16 * hh, a);
          if (row < 64) {  // A^kk row (strictly lower)
            // Entries on and above the diagonal of a diagonal block are stored unmasked:
            // the substitution below reads only the strictly lower ones and then
            // overwrites each block with its inverse.
            const int I = row >> 4, rl = row & 15;
            const int J = hh;  // block column
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int j = 16 * hh + 4 * q;  // global column of this float4
              const float4 v = make_float4(a[4 * q + 0], a[4 * q + 1], a[4 * q + 2], a[4 * q + 3]);
              if (J == I) *reinterpret_cast<float4 *>(Sd + sd_idx(I, rl, j & 15)) = v;
              if ((I == 1 && J == 0) || (I == 3 && J == 2))
                *reinterpret_cast<float4 *>(So + so_idx(I >> 1, rl, j & 15)) = v;
              if (row >= 32 && j < 32) *reinterpret_cast<float4 *>(Sl + sl_idx(row - 32, j)) = v;
            }
          } else {  // A^qk row (lower, diagonal included) -> bf16 TP rows 64-127
            const int i = row - 64;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              float v[8];
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const int j = 16 * hh + 8 * q + jj;
                v[jj] = j <= i ? a[8 * q + jj] : 0.f;
              }
              st8(tp + sw128(row, 2 * hh + q), v);
            }
          }
        }
        tc_fence_before();
        // The diagonal 16 x 16 blocks below are inverted by the warp that read their
        // rows out (warp 0: rows 0-31, warp 1: rows 32-63), so warps 0-1 go on after
        // a warp-level sync while warps 2-3 finish A^qk; the group meets again after.
        __syncwarp();

        // a3: T = (I + A^kk)^-1 in place, by recursive doubling of the block inverse
        //   [[L11, 0], [L21, L22]]^-1 = [[T11, 0], [-T22 L21 T11, T22]]
        // 16 x 16 diagonal blocks first (left-looking substitution, one column
        // per thread), then the 16-wide and the 32-wide off-diagonal blocks.
        if (t < 64) {
          float x[16];
          const int I = t >> 4, cc = t & 15;
          {
            // left-looking: x[r2] = -(row r2 of the block) . x[0 .. r2-1], rows read as
            // float4s, four partial sums per row (x[m] = 0 above column cc)
            const float *Ab = Sd + sd_idx(I, 0, 0);
#pragma unroll
            for (int r2 = 0; r2 < 16; ++r2) {
              float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int m4 = 0; m4 < r2; m4 += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(Ab + r2 * kSdLd + m4);
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                  if (m4 + e < r2) s4[e] = fmaf(av[e], x[m4 + e], s4[e]);
              }
              x[r2] = r2 == cc ? 1.f : (r2 > cc ? -((s4[0] + s4[1]) + (s4[2] + s4[3])) : 0.f);
            }
          }
          __syncwarp();  // every read of this warp's diagonal blocks is done
          float *Tb = Sd + sd_idx(I, 0, cc);
#pragma unroll
          for (int r2 = 0; r2 < 16; ++r2) Tb[r2 * kSdLd] = x[r2];
        }
        bar_sync(bar_id, 128);
        // The off-diagonal blocks are small dense products: warp-level TF32 MMAs
        // (16 x 8 tiles; fp32 operands enter as TF32, their low 13 mantissa bits
        // dropped: a relative error below 2^-10, under the bf16 rounding T gets next).
        const int lg = (t & 31) >> 2, lc = t & 3;  // fragment coordinates of this lane
        {  // T_10 and T_32: Y = L_{b+1,b} T_bb, then T_{b+1,b} = -T_{b+1,b+1} Y
          const int b = wq >> 1, n0 = 8 * (wq & 1);  // warp: block b, 8 output columns
          float y[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k0 = 0; k0 < 16; k0 += 8) {
            const uint32_t a[4] = {tf32_bits(So[so_idx(b, lg, k0 + lc)]),
                                   tf32_bits(So[so_idx(b, lg + 8, k0 + lc)]),
                                   tf32_bits(So[so_idx(b, lg, k0 + lc + 4)]),
                                   tf32_bits(So[so_idx(b, lg + 8, k0 + lc + 4)])};
            const uint32_t bb[2] = {tf32_bits(Sd[sd_idx(2 * b, k0 + lc, n0 + lg)]),
                                    tf32_bits(Sd[sd_idx(2 * b, k0 + lc + 4, n0 + lg)])};
            mma_tf32_16x8x8(y, a, bb);
          }
          // column n of T_{b+1,b} needs column n of Y only: this warp's own columns
          float *yb = Ys + b * 16 * 20;
          *reinterpret_cast<float2 *>(yb + lg * 20 + n0 + 2 * lc) = make_float2(y[0], y[1]);
          *reinterpret_cast<float2 *>(yb + (lg + 8) * 20 + n0 + 2 * lc) = make_float2(y[2], y[3]);
          __syncwarp();
          float z[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int k0 = 0; k0 < 16; k0 += 8) {
            const uint32_t a[4] = {tf32_bits(Sd[sd_idx(2 * b + 1, lg, k0 + lc)]),
                                   tf32_bits(Sd[sd_idx(2 * b + 1, lg + 8, k0 + lc)]),
                                   tf32_bits(Sd[sd_idx(2 * b + 1, lg, k0 + lc + 4)]),
                                   tf32_bits(Sd[sd_idx(2 * b + 1, lg + 8, k0 + lc + 4)])};
            const uint32_t bb[2] = {tf32_bits(yb[(k0 + lc) * 20 + n0 + lg]),
                                    tf32_bits(yb[(k0 + lc + 4) * 20 + n0 + lg])};
            mma_tf32_16x8x8(z, a, bb);
          }
          *reinterpret_cast<float2 *>(So + so_idx(b, lg, n0 + 2 * lc)) = make_float2(-z[0], -z[1]);
          *reinterpret_cast<float2 *>(So + so_idx(b, lg + 8, n0 + 2 * lc)) = make_float2(-z[2], -z[3]);
        }
        bar_sync(bar_id, 128);
        // rows 32-63, columns 0-31: Y = L[32:64, 0:32] T[0:32, 0:32], then -T[32:64, 32:64] Y.
        // Warp wq takes columns 8 wq .. 8 wq + 7 of all 32 rows, so the second product
        // reads only its own columns of Y; the result stays in registers until T is
        // converted to bf16 below (L[32:64, 0:32] is read by every warp meanwhile).
        const int n0 = 8 * wq;
        float z[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          float y[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
          // T[0:32, 0:16] = [T_00; T_10];  T[0:32, 16:32] = [0; T_11]
#pragma unroll
          for (int k0 = 0; k0 < 32; k0 += 8) {
            if (wq >= 2 && k0 < 16) continue;
            auto tlo = [&](int k, int cl) -> float {  // T[k][n0 + cl], k in 0..31, cl in 0..7
              if (wq < 2) return k < 16 ? Sd[sd_idx(0, k, n0 + cl)] : So[so_idx(0, k - 16, n0 + cl)];
              return Sd[sd_idx(1, k - 16, n0 - 16 + cl)];
            };
            const uint32_t bb[2] = {tf32_bits(tlo(k0 + lc, lg)), tf32_bits(tlo(k0 + lc + 4, lg))};
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              const int ra = 16 * mt + lg;
              const uint32_t a[4] = {tf32_bits(Sl[sl_idx(ra, k0 + lc)]), tf32_bits(Sl[sl_idx(ra + 8, k0 + lc)]),
                                     tf32_bits(Sl[sl_idx(ra, k0 + lc + 4)]),
                                     tf32_bits(Sl[sl_idx(ra + 8, k0 + lc + 4)])};
              mma_tf32_16x8x8(y[mt], a, bb);
            }
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            float *yr = Ys + (16 * mt + lg) * kYLd + n0 + 2 * lc;
            *reinterpret_cast<float2 *>(yr) = make_float2(y[mt][0], y[mt][1]);
            *reinterpret_cast<float2 *>(yr + 8 * kYLd) = make_float2(y[mt][2], y[mt][3]);
          }
          __syncwarp();
          // T[32:48, 32:64] = [T_22, 0];  T[48:64, 32:64] = [T_32, T_33]
#pragma unroll
          for (int k0 = 0; k0 < 32; k0 += 8) {
            const uint32_t bb[2] = {tf32_bits(Ys[(k0 + lc) * kYLd + n0 + lg]),
                                    tf32_bits(Ys[(k0 + lc + 4) * kYLd + n0 + lg])};
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              if (mt == 0 && k0 >= 16) continue;
              auto thi = [&](int r2, int k) -> float {  // T[32 + 16 mt + r2][32 + k]
                if (mt == 0) return Sd[sd_idx(2, r2, k)];
                return k < 16 ? So[so_idx(1, r2, k)] : Sd[sd_idx(3, r2, k - 16)];
              };
              const uint32_t a[4] = {tf32_bits(thi(lg, k0 + lc)), tf32_bits(thi(lg + 8, k0 + lc)),
                                     tf32_bits(thi(lg, k0 + lc + 4)), tf32_bits(thi(lg + 8, k0 + lc + 4))};
              mma_tf32_16x8x8(z[mt], a, bb);
            }
          }
        }
        bar_sync(bar_id, 128);
        {  // T -> TP rows 0-63 (bf16), 32 columns per thread; rows 32-63, columns 0-31
           // come from the fragments above
          const int i = t & 63, hh = t >> 6, I = i >> 4, il = i & 15;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j0 = 32 * hh + 8 * q, J = j0 >> 4, jl = j0 & 15;
            if (I >= 2 && J <= 1) continue;
            const float *src = nullptr;  // 8 consecutive T entries of row i, or zeros
            if (J == I) src = Sd + sd_idx(I, il, jl);
            else if ((I == 1 && J == 0) || (I == 3 && J == 2)) src = So + so_idx(I >> 1, il, jl);
            float tv[8];
            if (src) {
              const float4 t0v = *reinterpret_cast<const float4 *>(src);
              const float4 t1v = *reinterpret_cast<const float4 *>(src + 4);
              tv[0] = t0v.x; tv[1] = t0v.y; tv[2] = t0v.z; tv[3] = t0v.w;
              tv[4] = t1v.x; tv[5] = t1v.y; tv[6] = t1v.z; tv[7] = t1v.w;
            } else {
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) tv[jj] = 0.f;
            }
            st8(tp + sw128(i, 4 * hh + q), tv);  // T is exactly lower triangular
          }
          uint8_t *tpg = smem + L::kTP + kw * 16384;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int ri = 32 + 16 * mt + lg + 8 * e, cj = n0 + 2 * lc;
              *reinterpret_cast<uint32_t *>(tpg + sw128(ri, cj >> 3) + 2 * (cj & 7)) =
                  pack_bf16x2(-z[mt][2 * e], -z[mt][2 * e + 1]);
            }
        }

        if (helper) {
          // publish: once the tile has read chunk c - 4 out of the slot, copy TP (16 KiB,
          // the shared-memory image) there and release chunk c + 1
          fence_async_smem();  // the solve scratch in the g area is rewritten by the next load
          bar_sync(bar_id, 128);
          if (t == 0) {
            if (c + c_step < nchunks && !*abort_flag) load_g(s, c + c_step);
            ctx.wait_global(rflags + 2 * slot + 1, static_cast<uint32_t>(c >> 2));
          }
          bar_sync(bar_id, 128);
          uint4 *dst = reinterpret_cast<uint4 *>(rdata + slot * kRingSlotBytes);
#pragma unroll
          for (int j = 0; j < 8; ++j) __stcg(dst + 128 * j + t, ld_shared_v4(tp + 16 * (128 * j + t)));
          __threadfence();
          bar_sync(bar_id, 128);
          if (t == 0) {
            st_release_gpu(rflags + 2 * slot, static_cast<uint32_t>(c + 1));
            if (chan && !gsp && c + c_step < nchunks) {  // a1 of the group's next chunk
              ctx.wait(kFullG0 + s, cur ^ 1);
              issue_cumsum();
            }
          }
          continue;
        }
      }  // !fed

      // With the solve helpers (where the state side is the longer chain) the K-side forms
      // Vb = diag(beta) V in place once the v tile has landed: thread t scales the d_v half
      // t / 64 of row t mod 64, whose beta it holds.  In the plain schedule the state side
      // does it (only the state side reads Vb).
      if constexpr (kSched) {
        ctx.wait(kFullV0 + s, cur);
        const uint32_t fb = pack_bf16x2(brow, brow);
        const uint32_t vrow = st + L::kV + (t >> 6) * 8192;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t addr = vrow + sw128(rb, q);
          const uint4 w = ld_shared_v4(addr);
          st_shared_v4(addr, mul_bf16x2(w.x, fb), mul_bf16x2(w.y, fb), mul_bf16x2(w.z, fb),
                       mul_bf16x2(w.w, fb));
        }
      }
      fence_async_smem();  // also orders the solve's scratch writes before the g reload
      bar_sync(bar_id, 128);

      // [T; A^qk] Kb -> D2, rows 0-63: W = T Kb, issued before the state side's first
      // products (which need [T; A^qk] and Vb only) so that it goes ahead of them
      if (t == 0) {
        tc_fence_after();
        constexpr uint32_t id_k = idesc_bf16(128, 128, false, true);
        const uint32_t atp = sdesc_lo(tp, 16), bkb = sdesc_lo(st, L::kKQ1);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_ss(tm, atp + 2 * k4, sdesc_hi(1024), bkb + 128 * k4, sdesc_hi(1024), id_k, k4 > 0);
        mma_commit(mma_bar);
        mbar_arrive(ctx.bar(kTPReady0 + s));
        // the g area (solve scratch) is free: the group's next chunk's g tile
        if (!fed && c + 2 < nchunks && !*abort_flag) load_g(s, c + 2);
        ctx.wait(kMmaK0 + kw, kph & 1);
      } else if (fed && t == 32) {
        // every thread's ring loads have completed (their values are in TP[s]): count
        // the read (a gpu-scope release, kept off the issuing thread)
        red_release_gpu_add(rflags + 2 * slot + 1, 1u);
      }
      ++kph;
      bar_sync(bar_id, 128);
      tc_fence_after();
      if (row < 64) {
        // -W in bf16 over the row's Kb: rows 0-63 of the state product's B operand
        // [-W; Qh] (its rows 64-127 are Qh in the q area)
#pragma unroll 1
        for (int hq = 0; hq < 8; ++hq) {  // channels 16 hq .. 16 hq + 15
          float a[16];
          tmem_ld16(tm + lane_base + 16 * hq, a);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float w8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w8[e] = -a[8 * j + e];
            st8(st + (hq >> 2) * L::kKQ1 + sw128(row, 2 * (hq & 3) + j), w8);
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_sync(bar_id, 128);
      if (t == 0) {
        mbar_arrive(ctx.bar(kReady0 + s));
        if (chan && !gsp && c + 2 < nchunks) {  // a1 of chunk c + 2: the group's TMEM columns are free again
          ctx.wait(kFullG0 + s, cur ^ 1);
          issue_cumsum();
        }
      }
    }
    };
    if (kSched && helper)
      kloop(std::true_type{});
    else
      kloop(std::false_type{});
    if (t == 0) {  // all of this group's MMAs retired before TMEM is released
      mma_commit(ctx.bar(kFinK0 + kw));
      mbar_wait(ctx.bar(kFinK0 + kw), 0, kWaitCycles);
    }
  } else if (!helper) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 136;" ::: "memory");
    // ------------------------------------------------------------ state side
    // Thread (d_v row v = 32 (warp % 4) + lane, key-channel half hs = (warp - 8) / 4)
    // holds S[64 hs + j][v], j = 0..63, in fp32: column v of the state, which is row v
    // of S^T and TMEM lane v of every state-side product.
    const int st_id = tid - 256;
    const int qd = warp & 3, hs = (warp - 8) >> 2;
    const int v = 32 * qd + (tid & 31);
    const uint32_t lane_base = static_cast<uint32_t>(32 * qd) << 16;
    const size_t soff = (size_t)pair * DK * DV + (size_t)(64 * hs) * DV + v;
    float S[64];
    if (p.init_state) {
#pragma unroll
      for (int j = 0; j < 64; ++j) S[j] = p.init_state[soff + (size_t)j * DV];
    } else {
#pragma unroll
      for (int j = 0; j < 64; ++j) S[j] = 0.f;
    }
    uint32_t sph = 0;
    int pend_v = -1;  // chunk whose v tile (stage pend_v & 1) is loaded once the outputs left it
    for (int c = 0; c < nchunks; ++c) {
      const int s = c & 1;
      const int t0 = bos + c * C;
      const int len = min(C, eos - t0);
      const int kb = c % 3, gb = c % kGl;
      const uint32_t st = sbase + s * L::kStageBytes;
      const uint32_t tps = sbase + L::kTP + s * 16384;
      const uint32_t kcb = sbase + L::kKc + kb * 16384;
      // plain schedule: this thread's share of Vb = diag(beta) V, row vr and d_v columns
      // 32 (st_id / 64) .. + 31; its beta is loaded first
      const int vr = st_id & 63;
      float vbeta = 0.f;
      if constexpr (!kSched) {
        if (vr < len) {
          vbeta = __bfloat162float(p.beta[(size_t)(t0 + vr) * H + h]);
          if (kPrep && (p.prep & kPrepBetaSigmoid)) vbeta = fast_rcp(1.f + fast_exp2(-kLog2e * vbeta));
        }
      }
      // S^T in bf16 pairs -> columns [kRA + 32 hs, +32) of lane v: the state product's A operand
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) pk[jj] = pack_bf16x2(S[32 * hh + 2 * jj], S[32 * hh + 2 * jj + 1]);
        tmem_st16(tmem + lane_base + kRA + 32 * hs + 16 * hh, pk);
      }
      if constexpr (!kSched) {
        ctx.wait(kFullV0 + s, (c >> 1) & 1);
        const uint32_t fb = pack_bf16x2(vbeta, vbeta);
        const uint32_t vrow = st + L::kV + (st_id >> 7) * 8192;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t addr = vrow + sw128(vr, 4 * ((st_id >> 6) & 1) + q);
          const uint4 w = ld_shared_v4(addr);
          st_shared_v4(addr, mul_bf16x2(w.x, fb), mul_bf16x2(w.y, fb), mul_bf16x2(w.z, fb),
                       mul_bf16x2(w.w, fb));
        }
        fence_async_smem();  // Vb is read by the state products
      }
      tc_fence_before();
      bar_sync(2, 256);
      if (st_id == 0) {
        if (pend_v >= 0) {
          // the previous chunk's outputs have been read out of its v area: the next v tile
          bulk_wait_read();
          if (!*abort_flag) load_v(pend_v & 1, pend_v);
          pend_v = -1;
        }
        ctx.wait(kTPReady0 + s, (c >> 1) & 1);
        tc_fence_after();
        // [(E - Vb)^T | X^T] = Vb^T [T; A^qk]^T - Vb^T [I | 0] + S^T [-W; Qh]^T, one commit:
        // the first two terms as soon as [T; A^qk] is there, the state product once -W is
        constexpr uint32_t id_init = idesc_bf16(128, 128, true, false);
        constexpr uint32_t id_negi = idesc_bf16(128, 64, true, false);
        const uint32_t avb = sdesc_lo(st + L::kV, 8192);  // Vb^T (MN-major)
        const uint32_t btp = sdesc_lo(tps, 16);           // [T; A^qk] rows
        const uint32_t bni = sdesc_lo(sbase + L::kNegI, 16);  // -I rows
        const uint32_t bwq = sdesc_lo(st, 16);            // [-W; Qh]
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_ss(tmem + kRD1, avb + 128 * k4, sdesc_hi(1024), btp + 2 * k4, sdesc_hi(1024), id_init, k4 > 0);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_ss(tmem + kRD1, avb + 128 * k4, sdesc_hi(1024), bni + 2 * k4, sdesc_hi(1024), id_negi, 1);
        ctx.wait(kReady0 + s, (c >> 1) & 1);
        tc_fence_after();
        constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);
#pragma unroll
        for (int k8 = 0; k8 < 8; ++k8)
          mma_ts(tmem + kRD1, tmem + kRA + 8u * k8, bwq + (k8 >> 2) * (L::kKQ1 >> 4) + 2 * (k8 & 3),
                 sdesc_hi(1024), id_s, 1);
        mma_commit(ctx.bar(kMmaS));
        ctx.wait(kMmaS, sph & 1);
        // the stage's k and q tiles ([-W; Qh]) have been read: the group's next chunk's
        if (c + 2 < nchunks && !*abort_flag) {
          load_k(s, c + 2);
          load_q(s, c + 2);
        }
      }
      ++sph;
      bar_sync(2, 256);
      tc_fence_after();
      if (st_id < 128) {
        // gamma = exp(G_last) of key channel st_id (written before Ready, which thread 0
        // waited on before the barrier above).  A chunk whose total log decay is beyond
        // the range the factors exp(+-G) are formed in marks the pair for the exact
        // recomputation (or is reported without the flags): from here on this CTA stores
        // nothing for it; the pipeline itself runs on unchanged
        const float gam = glast[gb * 128 + st_id];
        if (!(gam >= kMinGamma) && !(*skip_flag & 1)) {
          *skip_flag = 1;
          if (p.pair_flags) {
            // (a segment run marks its sequence's pair, the sequence taken from its table entry)
            const int fp = p.seq_stride == 4 ? p.cu_seqlens[4 * (pair / H) + 3] * H + h : pair;
            if (atomicExch(p.pair_flags + fp, 1u) == 0u) atomicAdd(p.status + 3, 1u);
          } else {
            atomicCAS(p.status, 0u, kStatusGateRange);
          }
        }
      }
      {  // (E - Vb)^T of tokens 32 hs .. 32 hs + 31, bf16 pairs -> columns [kREV + 16 hs, +16)
        uint32_t pk[16];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float a[16];
          tmem_ld16(tmem + lane_base + kRD1 + 32 * hs + 16 * hh, a);
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) pk[8 * hh + jj] = pack_bf16x2(a[2 * jj], a[2 * jj + 1]);
        }
        tmem_st16(tmem + lane_base + kREV + 16 * hs, pk);
      }
      tc_fence_before();
      bar_sync(2, 256);
      if (st_id == 0) {
        tc_fence_after();
        // (Kc^T E)^T = (E - Vb)^T Kc + Vb^T Kc over S^T and the first half of the above
        // (both read by now); O^T / s = X^T + (E - Vb)^T A^qk^T
        constexpr uint32_t id_e = idesc_bf16(128, 128, false, true);
        constexpr uint32_t id_v = idesc_bf16(128, 128, true, true);
        constexpr uint32_t id_o = idesc_bf16(128, 64, false, false);
        const uint32_t bkc = sdesc_lo(kcb, 8192), avb = sdesc_lo(st + L::kV, 8192);
        const uint32_t baq = sdesc_lo(tps + 8192, 16);  // A^qk rows
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_ts(tmem + kRD4, tmem + kREV + 8u * k4, bkc + 128 * k4, sdesc_hi(1024), id_e, k4 > 0);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_ss(tmem + kRD4, avb + 128 * k4, sdesc_hi(1024), bkc + 128 * k4, sdesc_hi(1024), id_v, 1);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_ts(tmem + kRD1 + 64, tmem + kREV + 8u * k4, baq + 2 * k4, sdesc_hi(1024), id_o, 1);
        mma_commit(ctx.bar(kMmaS));
        ctx.wait(kMmaS, sph & 1);
        mbar_arrive(ctx.bar(kKcFree0 + kb));  // Kc[kb] and TP[s] have been read
      }
      ++sph;
      bar_sync(2, 256);
      tc_fence_after();
      // read after the barrier that follows every setter of the skip flag
      const bool store = !*skip_flag;
      {  // S <- gamma (S + Kc^T E), elementwise per key channel
        const float4 *g4 = reinterpret_cast<const float4 *>(glast + gb * 128 + 64 * hs);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          float a[16];
          tmem_ld16(tmem + lane_base + kRD4 + 64 * hs + 16 * hh, a);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 gm = g4[4 * hh + q];
            const float gv[4] = {gm.x, gm.y, gm.z, gm.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float &sv = S[16 * hh + 4 * q + e];
              sv = gv[e] * (sv + a[4 * q + e]);
            }
          }
        }
      }
      // outputs: row v of O^T / s, tokens 32 hs .. 32 hs + 31, into the chunk's v area (Vb
      // has been read) laid out as the two 64-channel output boxes (128-byte swizzle: token
      // row r, 16-byte piece j at r * 128 + ((j ^ (r & 7)) << 4)).  A full chunk leaves by
      // TMA; a sequence's partial last chunk is copied out row by row (a box would pass its
      // end).
      const bool full = len == C;
      const uint32_t obase = st + L::kV + (v >> 6) * 8192 + 2 * (v & 7);
      const uint32_t opiece = ((v & 63) >> 3) << 4;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float a[16];
        tmem_ld16(tmem + lane_base + kRD1 + 64 + 32 * hs + 16 * hh, a);
        if (store) {
          const uint32_t ob = obase + (32 * hs + 16 * hh) * 128;  // first token of these columns
#pragma unroll
          for (int i = 0; i < 16; ++i)
            st_shared_u16(ob + i * 128 + (opiece ^ ((i & 7) << 4)),
                          __bfloat16_as_ushort(__float2bfloat16_rn(p.scale * a[i])));
        }
      }
      fence_async_smem();
      tc_fence_before();
      bar_sync(2, 256);  // every thread has read kRD4, kRD1 and G_last[gb], and staged its outputs
      if (!full && store) {
#pragma unroll 1
        for (int idx = st_id; idx < len * 16; idx += 256) {
          const int r = idx >> 4, box = (idx >> 3) & 1, j = idx & 7;  // token r, channels 64 box + 8 j
          const uint4 w = ld_shared_v4(st + L::kV + box * 8192 + r * 128 + ((j ^ (r & 7)) << 4));
          *reinterpret_cast<uint4 *>(p.out + ((size_t)(t0 + r) * H + h) * DV + 64 * box + 8 * j) = w;
        }
      }
      if (st_id == 0) {
        mbar_arrive(ctx.bar(kGmRead0 + gb));
        if (store && full && !*abort_flag) {
          tma_store_3d(&tm_o, st + L::kV, 0, h, t0);
          tma_store_3d(&tm_o, st + L::kV + 8192, 64, h, t0);
        }
        bulk_commit();
        // the v area is reloaded (for chunk c + 2) once the store has read it: next chunk
        if (c + 2 < nchunks) pend_v = c + 2;
      }
    }
    bar_sync(2, 256);  // every setter of the skip flag is done
    if (p.final_state && !(*skip_flag & 1)) {
#pragma unroll
      for (int j = 0; j < 64; ++j) p.final_state[soff + (size_t)j * DV] = S[j];
    }
    if (st_id == 0) {
      bulk_wait();  // the last outputs' stores are complete
      mma_commit(ctx.bar(kFinS));
      mbar_wait(ctx.bar(kFinS), 0, kWaitCycles);
    }
  }

  // no TMA load may still be in flight when the CTA leaves (possible only after a
  // timeout stopped its consumer): wait (bounded) for the last load of every part
  __syncthreads();
  if (tid == 0) {
    constexpr uint32_t kFull[4] = {kFullQ0, kFullG0, kFullK0, kFullV0};
    for (int sidx = 0; sidx < 2; ++sidx)
      for (int part = 0; part < 4; ++part) {
        const int c = issued[4 * sidx + part];
        if (c >= 0) mbar_wait(ctx.bar(kFull[part] + sidx), (c >> c_shift) & 1, kWaitCycles);
      }
  }
  if (tid == 0 && *abort_flag) atomicCAS(p.status, 0u, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
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

// Launch order of the plain schedule when it needs more than one wave: the sequences
// sorted longest first (ties by index), so the longest chains start first and the last
// wave holds the short ones.  One CTA ranks the (length, index) keys in shared memory
// (all threads read the same key at a time); offsets out of order count as length 0
// (the prefill kernel skips and reports them).
constexpr int kOrderMaxSeqs = 2048;
__global__ void __launch_bounds__(1024) kda_tc_order_kernel(const int32_t *cu_seqlens, int N, int T,
                                                            int32_t *order) {
  extern __shared__ unsigned long long okeys[];
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const int a = cu_seqlens[i], b = cu_seqlens[i + 1];
    const int len = (0 <= a && a <= b && b <= T) ? b - a : 0;
    okeys[i] = (static_cast<unsigned long long>(0x7FFFFFFF - len) << 32) | static_cast<unsigned>(i);
  }
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    const unsigned long long ki = okeys[i];
    int rank = 0;
    for (int j = 0; j < N; ++j) rank += okeys[j] < ki;
    order[rank] = i;
  }
}
size_t order_bytes(long long num_seqs) { return (static_cast<size_t>(num_seqs) * 4 + 255) / 256 * 256; }

// Segment-parallel scan of a few long sequences ("Kimi Delta Attention (KDA)", the state
// recurrence is affine in the start state: S_end = M S_start + B over any stretch of
// tokens, M the product of the per-token transitions (I - beta k k^T) Diag(alpha)).
// With few sequence-heads the helpers still leave most SMs idle, so every sequence is cut
// into P segments of whole chunks:
//   pass 1  segment 0 from the true start (its outputs are final); every middle segment
//           p = 1 .. P - 2 twice, from zero (its end state B_p) and from the identity with
//           V taken as zero (its transfer matrix M_p, as d_k = d_v);
//   combine S_1 = end of segment 0, S_{p+1} = M_p S_p + B_p (fp32, column blocks apart);
//   pass 2  segments 1 .. P - 1 from S_p, storing their outputs; the last one's end state
//           is the sequence's final state.
// Runs of sequence n: pass 1 n (2P - 3) + k, pass 2 n (P - 1) + q - 1.  The first pass runs
// N H (2P - 3) CTAs in one wave: at least 3 segments of at least 32 chunks of the average
// sequence, otherwise the other schedules run.
constexpr int kSegMinChunks = 32;
int seg_count(int N, long long T, int H, int sms) {
  if (N < 1 || H < 1 || sms < 1 || T >= (1LL << 30)) return 0;  // (zero V tiles are read below token 0)
  const long long NH = static_cast<long long>(N) * H;
  if (NH > sms) return 0;
  const long long nch = (T / N + C - 1) / C;  // chunks of the average sequence
  const long long P = std::min<long long>((sms / NH + 3) / 2, nch / kSegMinChunks);
  return P >= 3 ? static_cast<int>(P) : 0;
}
// run tables (3P slots per sequence) and the (sequence, head) pairs the second pass skips
size_t seg_table_bytes(int P, int N, int H) {
  return (static_cast<size_t>(3 * P) * N * sizeof(int4) + static_cast<size_t>(N) * H * 4 + 255) / 256 * 256;
}
// The pairs of the larger pass that can take solve helpers (at most kHelperMaxPairs), or 0.
long long seg_ring_pairs(int P, long long NH) {
  const long long r1 = (2 * P - 3) * NH, r2 = (P - 1) * NH;
  return std::max(r1 <= kHelperMaxPairs ? r1 : 0, r2 <= kHelperMaxPairs ? r2 : 0);
}
size_t ring_bytes(long long pairs);
// run tables, pass-1 end states, start states, pass-2 end states, the helpers' ring
size_t seg_bytes(int P, int N, int H) {
  const long long NH = static_cast<long long>(N) * H;
  return seg_table_bytes(P, N, H) + static_cast<size_t>(4 * P - 5) * NH * DK * DV * sizeof(float) +
         ring_bytes(seg_ring_pairs(P, NH));
}
int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 152;  // no device: size for a GB300
  }
  return sms;
}

// The run tables of both passes, block n for sequence n, from its offsets as the device
// holds them (checked like every other kernel does: out of order or range, the sequence's
// runs are skipped and KDA_ERR_SEQLENS recorded).  Segment q takes chunks q m / P ..
// (q + 1) m / P - 1 of the sequence's m chunks (sizes differ by one chunk at most); the last
// one ends at the sequence's end.
__global__ void kda_seg_table_kernel(const int32_t *cu_seqlens, int T, int P, int4 *runs1, int4 *runs2,
                                     uint32_t *status) {
  const int n = blockIdx.x;
  const int b = cu_seqlens[n], e = cu_seqlens[n + 1];
  const bool ok = 0 <= b && b <= e && e <= T;
  if (!ok && threadIdx.x == 0) atomicCAS(status, 0u, kStatusSeqlens);
  const int skip = ok ? 0 : kRunSkip;
  const long long m = ok ? (static_cast<long long>(e) - b + C - 1) / C : 0;
  int4 *r1 = runs1 + n * (2 * P - 3), *r2 = runs2 + n * (P - 1);
  for (int q = threadIdx.x; q < P; q += blockDim.x) {
    const int sb = ok ? static_cast<int>(std::min<long long>(b + q * m / P * C, e)) : b;
    const int se = ok ? static_cast<int>(std::min<long long>(b + (q + 1) * m / P * C, e)) : b;
    if (q == 0) {
      r1[0] = make_int4(sb, se, skip, n);
    } else {
      r2[q - 1] = make_int4(sb, se, skip, n);
      if (q < P - 1) {
        r1[2 * q - 1] = make_int4(sb, se, kRunNoOut | skip, n);
        r1[2 * q] = make_int4(sb, se, kRunZeroV | kRunNoOut | skip, n);
      }
    }
  }
}

// The start states of the pass-1 runs, in the buffer their end states then overwrite (each
// thread of the chunk kernel reads and later writes the same elements): each sequence's
// run 0 its given initial state (zero without one), runs 2p - 1 zero, runs 2p the identity.
__global__ void __launch_bounds__(256) kda_seg_init_kernel(float *F1, const float *init, int P, int H) {
  const size_t i = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;  // < N (2P-3) H d_k d_v
  const size_t per_run = static_cast<size_t>(H) * DK * DV;
  const int run = static_cast<int>(i / per_run), k = run % (2 * P - 3), n = run / (2 * P - 3);
  const size_t e = i % per_run;  // element of head e / (d_k d_v)
  float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
  if (k == 0) {
    if (init) x = *reinterpret_cast<const float4 *>(init + static_cast<size_t>(n) * per_run + e);
  } else if (k % 2 == 0) {
    const int r = static_cast<int>(e % (DK * DV)) / DV, c = static_cast<int>(e % DV);  // c .. c + 3
    x = make_float4(r == c ? 1.f : 0.f, r == c + 1 ? 1.f : 0.f, r == c + 2 ? 1.f : 0.f, r == c + 3 ? 1.f : 0.f);
  }
  *reinterpret_cast<float4 *>(F1 + i) = x;
}

// S_1 = the end state of segment 0 (pass-1 run 0); S_{p+1} = M_p S_p + B_p with M_p, B_p
// the end states of pass-1 runs 2p and 2p - 1, in fp32.  CTA (n, h, cb) keeps columns
// 4 cb .. 4 cb + 3 of sequence n's state of head h in shared memory (the columns do not
// mix).  Warp w forms rows 8 w .. 8 w + 7: lane l multiplies keys 4 l .. 4 l + 3 (its
// part of each row of M_p, read as one float4 per row, the warp's loads coalesced, and
// loaded while the CTA still works on the step before), and the lanes' 32 partial sums
// are reduced by a butterfly that leaves row 8 w + l / 4, column l mod 4 in lane l.  The
// CTAs with cb = 0 also copy the recomputation marks the first pass left, for the second
// pass to skip those sequence-heads.
constexpr int kCombThreads = 512;
__global__ void __launch_bounds__(kCombThreads) kda_seg_combine_kernel(const float *F1, float *starts, int P,
                                                                       int H, const uint32_t *pair_flags,
                                                                       uint32_t *head_skip) {
  __shared__ float4 Ssh[DK];  // S_p[j][4 cb .. 4 cb + 3]
  const int nh = blockIdx.x / (DV / 4), cb = blockIdx.x % (DV / 4), n = nh / H, h = nh % H;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (cb == 0 && threadIdx.x == 0) head_skip[nh] = pair_flags ? pair_flags[nh] : 0u;
  const size_t stride = static_cast<size_t>(H) * DK * DV;
  // sequence n's pass-1 runs and start states, head h
  F1 += static_cast<size_t>(n) * (2 * P - 3) * stride;
  starts += static_cast<size_t>(n) * (P - 1) * stride;
  const size_t hoff = static_cast<size_t>(h) * DK * DV;
  if (threadIdx.x < DK) {  // run 0: segment 0's end
    const size_t o = hoff + static_cast<size_t>(threadIdx.x) * DV + 4 * cb;
    const float4 s1 = *reinterpret_cast<const float4 *>(F1 + o);
    *reinterpret_cast<float4 *>(starts + o) = s1;
    Ssh[threadIdx.x] = s1;
  }
  const int orow = 8 * w + (l >> 2), ocol = 4 * cb + (l & 3);  // the element lane l forms
  const size_t ooff = hoff + static_cast<size_t>(orow) * DV + ocol;
  // row part of M_q (rows 8 w + rr, keys 4 l .. 4 l + 3) and lane l's element of B_q
  auto load = [&](int q, float4 (&m)[8], float &b) {
    const float *M = F1 + 2 * q * stride + hoff + static_cast<size_t>(8 * w) * DV + 4 * l;
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) m[rr] = *reinterpret_cast<const float4 *>(M + rr * DV);
    b = F1[(2 * q - 1) * stride + ooff];
  };
  auto step = [&](int q, float4 (&mc)[8], float bc, float4 (&mn)[8], float &bn) {
    __syncthreads();  // Ssh holds S_q
    if (q + 1 <= P - 2) load(q + 1, mn, bn);
    float4 sv[4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) sv[jj] = Ssh[4 * l + jj];
    float v[32];  // v[4 rr + c]: this lane's part of row 8 w + rr, column c
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const float mj[4] = {mc[rr].x, mc[rr].y, mc[rr].z, mc[rr].w};
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        a0 = fmaf(mj[jj], sv[jj].x, a0);
        a1 = fmaf(mj[jj], sv[jj].y, a1);
        a2 = fmaf(mj[jj], sv[jj].z, a2);
        a3 = fmaf(mj[jj], sv[jj].w, a3);
      }
      v[4 * rr] = a0, v[4 * rr + 1] = a1, v[4 * rr + 2] = a2, v[4 * rr + 3] = a3;
    }
    // butterfly over the lanes: at offset o each lane keeps the half of its values its
    // bit o selects and adds the partner's copy of that half; lane l ends with v[l]
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const bool up = l & o;
#pragma unroll
      for (int i = 0; i < o; ++i) {
        const float send = up ? v[i] : v[i + o], keep = up ? v[i + o] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    const float sn = v[0] + bc;
    __syncthreads();  // every thread has read S_q
    reinterpret_cast<float *>(Ssh)[4 * orow + (l & 3)] = sn;
    starts[q * stride + ooff] = sn;
  };
  float4 mA[8], mB[8];
  float bA = 0.f, bB = 0.f;
  if (P >= 3) load(1, mA, bA);
  for (int q = 1; q <= P - 2; q += 2) {
    step(q, mA, bA, mB, bB);
    if (q + 1 <= P - 2) step(q + 1, mB, bB, mA, bA);
  }
}

// Each sequence's final state from its last segment's end state, for every (sequence, head)
// whose runs all went through (not skipped, not marked for the exact recomputation, which
// writes it from the untouched initial state instead).
__global__ void __launch_bounds__(256) kda_seg_final_kernel(const float *F2, float *final_state, const int4 *runs2,
                                                            const uint32_t *pair_flags, int P, int H) {
  const size_t i = (static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;  // < N H d_k d_v
  const int nh = static_cast<int>(i / (DK * DV)), n = nh / H;
  const int last = n * (P - 1) + P - 2;  // sequence n's last pass-2 run
  if ((runs2[last].z & kRunSkip) || (pair_flags && pair_flags[nh])) return;
  const size_t src = (static_cast<size_t>(last) * H + nh % H) * DK * DV + i % (DK * DV);
  *reinterpret_cast<float4 *>(final_state + i) = *reinterpret_cast<const float4 *>(F2 + src);
}

// Ring of the helper schedule: [P][kRingSlots] slot images, then [P][kRingSlots][2] words.
size_t ring_bytes(long long pairs) {
  return static_cast<size_t>(pairs) * kRingSlots * (kRingSlotBytes + 2 * sizeof(uint32_t));
}

}  // namespace

bool chunk_tc_supported(int d_k, int d_v, bool bf16) { return bf16 && d_k == 128 && d_v == 128; }
size_t chunk_tc_scratch_bytes(int num_seqs, int total_tokens, int num_heads, int, int) {
  const long long pairs = (long long)num_seqs * num_heads;
  size_t bytes = 0;
  if (pairs >= 1 && pairs <= kHelperMaxPairs) bytes = ring_bytes(pairs);  // solve helpers
  else if (num_seqs >= 2 && num_seqs <= kOrderMaxSeqs) bytes = order_bytes(num_seqs);  // launch order
  // a few long sequences: the segment-parallel scan, when it applies
  const int P = seg_count(num_seqs, total_tokens, num_heads, device_sms());
  if (P) bytes = std::max(bytes, seg_bytes(P, num_seqs, num_heads));
  return bytes;
}

// The solve-helper schedule over `pairs` pairs in one cooperative launch, every CTA resident
// as the hand-over through global memory needs: cudaSuccess once enqueued, cudaErrorNotReady
// when it does not apply or does not fit (nothing launched: the plain schedule runs).
template <bool kPrep, bool kChan>
static cudaError_t launch_helpers(const ChunkArgs &a, cudaStream_t stream, CUtensorMap &mq, CUtensorMap &mk,
                                  CUtensorMap &mg, CUtensorMap &mv, CUtensorMap &mo, TcParams prm,
                                  long long pairs, uint8_t *ring, size_t ring_avail) {
  // one or two helpers per pair, all CTAs in one wave
  const int hpp = 3 * pairs <= a.num_sms ? 2 : (2 * pairs <= a.num_sms ? 1 : 0);
  int dev = 0, coop = 0;
  if (hpp == 0 || pairs > kHelperMaxPairs || !ring || ring_avail < ring_bytes(pairs)) return cudaErrorNotReady;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) {
    (void)cudaGetLastError();
    return cudaErrorNotReady;
  }
  cudaError_t err = cudaFuncSetAttribute(kda_chunk_tc_kernel<true, kPrep, kChan>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (err != cudaSuccess) return err;
  prm.npairs = static_cast<int>(pairs);  // the tiles; CTAs from here on are helpers
  prm.ring = ring;
  prm.ring_flags = reinterpret_cast<uint32_t *>(ring + pairs * kRingSlots * kRingSlotBytes);
  prm.helpers_per_pair = hpp;
  err = cudaMemsetAsync(prm.ring_flags, 0, pairs * kRingSlots * 2 * sizeof(uint32_t), stream);
  if (err != cudaSuccess) return err;
  void *args[] = {&mq, &mk, &mg, &mv, &mo, &prm};
  err = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kda_chunk_tc_kernel<true, kPrep, kChan>),
                                    dim3(static_cast<unsigned>((1 + hpp) * pairs)), dim3(kThreads), args,
                                    L::kAlloc, stream);
  if (err != cudaErrorCooperativeLaunchTooLarge) return err;
  (void)cudaGetLastError();  // not all resident (SMs taken)
  return cudaErrorNotReady;
}

// The launch of one instantiation: the segment-parallel scan for a few long sequences with few
// heads, else the solve-helper schedule when it fits, else the plain one.
template <bool kPrep, bool kChan>
static cudaError_t launch_tc(const ChunkArgs &a, cudaStream_t stream, CUtensorMap &mq, CUtensorMap &mk,
                             CUtensorMap &mg, CUtensorMap &mv, CUtensorMap &mo, TcParams &prm,
                             long long pairs) {
  cudaError_t err = cudaFuncSetAttribute(kda_chunk_tc_kernel<false, kPrep, kChan>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (err != cudaSuccess) return err;
  // A few long sequences with few heads: the segment-parallel scan (two passes and a combine)
  const int P = seg_count(a.num_seqs, a.total_tokens, a.num_heads, a.num_sms);
  if (P && a.scratch && a.scratch_bytes >= seg_bytes(P, a.num_seqs, a.num_heads)) {
    const int N = a.num_seqs, H = a.num_heads;
    const long long NH = static_cast<long long>(N) * H;
    const size_t st = static_cast<size_t>(H) * DK * DV;  // floats of one run's states
    unsigned char *base = static_cast<unsigned char *>(a.scratch);
    int4 *runs1 = reinterpret_cast<int4 *>(base);
    int4 *runs2 = runs1 + static_cast<size_t>(N) * (2 * P - 3);
    uint32_t *head_skip = reinterpret_cast<uint32_t *>(runs1 + static_cast<size_t>(N) * 3 * P);
    float *F1 = reinterpret_cast<float *>(base + seg_table_bytes(P, N, H));
    float *starts = F1 + static_cast<size_t>(N) * (2 * P - 3) * st;
    float *F2 = starts + static_cast<size_t>(N) * (P - 1) * st;
    uint8_t *ring = reinterpret_cast<uint8_t *>(F2 + static_cast<size_t>(N) * (P - 1) * st);
    const size_t ring_avail = ring_bytes(seg_ring_pairs(P, NH));
    // a pass through the helper schedule when it fits, else the plain one
    auto pass = [&](TcParams &pp, long long np) -> cudaError_t {
      pp.npairs = static_cast<int>(np);  // (run, head) pairs of this pass
      cudaError_t e = launch_helpers<kPrep, kChan>(a, stream, mq, mk, mg, mv, mo, pp, np, ring, ring_avail);
      if (e != cudaErrorNotReady) return e;
      kda_chunk_tc_kernel<false, kPrep, kChan><<<(unsigned)np, kThreads, L::kAlloc, stream>>>(mq, mk, mg, mv, mo,
                                                                                                pp);
      return cudaGetLastError();
    };
    kda_seg_table_kernel<<<N, 128, 0, stream>>>(a.cu_seqlens, a.total_tokens, P, runs1, runs2, a.status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const size_t n1 = static_cast<size_t>(N) * (2 * P - 3) * st;  // floats, a multiple of 1024
    kda_seg_init_kernel<<<(unsigned)(n1 / 1024), 256, 0, stream>>>(F1, a.init_state, P, H);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    TcParams p1 = prm;
    p1.cu_seqlens = reinterpret_cast<const int32_t *>(runs1);
    p1.seq_stride = 4;
    p1.init_state = F1;  // in place
    p1.final_state = F1;
    if ((err = pass(p1, (2 * P - 3) * NH)) != cudaSuccess) return err;
    kda_seg_combine_kernel<<<(unsigned)(NH * (DV / 4)), kCombThreads, 0, stream>>>(F1, starts, P, H,
                                                                                  a.pair_flags, head_skip);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    TcParams p2 = prm;
    p2.cu_seqlens = reinterpret_cast<const int32_t *>(runs2);
    p2.seq_stride = 4;
    p2.head_skip = head_skip;
    p2.init_state = starts;
    p2.final_state = F2;
    if ((err = pass(p2, (P - 1) * NH)) != cudaSuccess || !a.final_state) return err;
    kda_seg_final_kernel<<<(unsigned)(NH * DK * DV / 1024), 256, 0, stream>>>(F2, a.final_state, runs2,
                                                                              a.pair_flags, P, H);
    return cudaGetLastError();
  }
  // Few sequence-heads leave most SMs idle: with room for the ring, one or two solve
  // helpers per sequence-head join its tile in one cooperative launch.
  err = launch_helpers<kPrep, kChan>(a, stream, mq, mk, mg, mv, mo, prm, pairs,
                                     static_cast<uint8_t *>(a.scratch), a.scratch ? a.scratch_bytes : 0);
  if (err != cudaErrorNotReady) return err;
  // More than one wave: start the longest sequences first (when the workspace has room)
  if (pairs > a.num_sms && a.num_seqs >= 2 && a.num_seqs <= kOrderMaxSeqs && a.scratch &&
      a.scratch_bytes >= order_bytes(a.num_seqs)) {
    int32_t *order = static_cast<int32_t *>(a.scratch);
    kda_tc_order_kernel<<<1, 1024, a.num_seqs * sizeof(unsigned long long), stream>>>(
        a.cu_seqlens, a.num_seqs, a.total_tokens, order);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    prm.order = order;
  }
  kda_chunk_tc_kernel<false, kPrep, kChan><<<(unsigned)pairs, kThreads, L::kAlloc, stream>>>(mq, mk, mg, mv,
                                                                                                 mo, prm);
  return cudaGetLastError();
}

cudaError_t launch_chunk_tc(const ChunkArgs &a, cudaStream_t stream) {
  if (!chunk_tc_supported(a.d_k, a.d_v, a.bf16)) return cudaErrorInvalidValue;
  if (!encode_fn()) return cudaErrorNotSupported;
  CUtensorMap mq, mk, mg, mv, mo;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mg, 0, sizeof(mg));
  memset(&mv, 0, sizeof(mv));
  memset(&mo, 0, sizeof(mo));
  if (a.total_tokens > 0) {
    if (!make_map(&mq, a.q, a.total_tokens, a.num_heads) ||
        !make_map(&mk, a.k, a.total_tokens, a.num_heads) ||
        !make_map(&mg, a.gate == 0 ? a.g : a.q, a.total_tokens, a.num_heads) ||
        !make_map(&mv, a.v, a.total_tokens, a.num_heads) ||
        !make_map(&mo, a.out, a.total_tokens, a.num_heads))
      return cudaErrorInvalidValue;
  }
  TcParams prm;
  prm.beta = static_cast<const __nv_bfloat16 *>(a.beta);
  prm.g_tok = a.gate == 1 ? static_cast<const __nv_bfloat16 *>(a.g) : nullptr;
  prm.gate = a.gate;
  prm.prep = a.prep;
  prm.gate_scale = a.gate_scale;
  prm.helpers_per_pair = 1;
  prm.init_state = a.init_state;
  prm.cu_seqlens = a.cu_seqlens;
  prm.out = static_cast<__nv_bfloat16 *>(a.out);
  prm.final_state = a.final_state;
  prm.status = a.status;
  prm.pair_flags = a.pair_flags;
  prm.T = a.total_tokens;
  prm.H = a.num_heads;
  prm.scale = a.scale;
  prm.flags = a.test_flags;
  prm.ring = nullptr;
  prm.ring_flags = nullptr;
  prm.order = nullptr;
  prm.seq_stride = 1;
  prm.head_skip = nullptr;
  const long long pairs = (long long)a.num_seqs * a.num_heads;
  prm.npairs = static_cast<int>(pairs);
  if (pairs == 0) return cudaSuccess;
  // one instantiation per gate family (one log alpha per key channel, or the others),
  // with or without the input steps
  if (a.prep)
    return a.gate == 0 ? launch_tc<true, true>(a, stream, mq, mk, mg, mv, mo, prm, pairs)
                       : launch_tc<true, false>(a, stream, mq, mk, mg, mv, mo, prm, pairs);
  return a.gate == 0 ? launch_tc<false, true>(a, stream, mq, mk, mg, mv, mo, prm, pairs)
                     : launch_tc<false, false>(a, stream, mq, mk, mg, mv, mo, prm, pairs);
}

}  // namespace kda
