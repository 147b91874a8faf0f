/*
 * kda_oracle.c -- plain, slow, sequential fp64 CPU oracle for the Kimi Delta
 * Attention (KDA) forward recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this.  It shares no code, header,
 * table or helper with the CUDA library; it is the definition written out.
 *
 * What it computes ("Kimi Delta Attention (KDA)", brain.bigb.es, opening
 * equation and the five-line reference recurrence in the transposed d_k x d_v
 * layout; "K3 架构图解", Ch.08, the four-line column-vector form):
 *
 *   per sequence, per head, state S in R^{d_k x d_v}, for t = 1..T:
 *     alpha_t = exp(g_t)                     g_t = log(alpha_t) <= 0, per key channel
 *     S~_t    = Diag(alpha_t) S_{t-1}        forget (before predict)
 *     vhat_t  = S~_t^T k_t                   predict
 *     e_t     = beta_t (v_t - vhat_t)        correct (beta_t scalar per token and head)
 *     S_t     = S~_t + k_t e_t^T             rank-one write
 *     o_t     = scale * S_t^T q_t            read after write
 *
 * Layouts (row-major, contiguous):
 *   q, k, g : [T_total, H, d_k]      v, out : [T_total, H, d_v]
 *   beta    : [T_total, H]           state  : [N, H, d_k, d_v]
 *   cu_seqlens : [N + 1], sequence n owns tokens [cu[n], cu[n+1]).
 *
 * Each (sequence, head) pair is an independent recurrence; pairs are spread
 * over POSIX threads.  Within a pair the arithmetic order is fixed, so the
 * result does not depend on the thread count.  Build with -ffp-contract=off so
 * that x86 and Arm hosts give bit-identical results.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
  int num_seqs, H, dk, dv;
  const int64_t *cu;
  double scale;
  const double *q, *k, *v, *g, *beta, *init_state;
  double *out, *final_state;
  int64_t next_pair; /* work counter, (seq, head) pairs handed out in order */
} kda_oracle_job;

/* One (sequence, head) recurrence, token by token. */
static void kda_oracle_pair(const kda_oracle_job *J, int n, int h, double *S,
                            double *e) {
  const int H = J->H, dk = J->dk, dv = J->dv;
  const int64_t bos = J->cu[n], eos = J->cu[n + 1];
  const size_t state_off = ((size_t)n * H + h) * (size_t)dk * dv;

  if (J->init_state)
    memcpy(S, J->init_state + state_off, sizeof(double) * (size_t)dk * dv);
  else
    memset(S, 0, sizeof(double) * (size_t)dk * dv);

  for (int64_t t = bos; t < eos; ++t) {
    const double *qt = J->q + ((size_t)t * H + h) * dk;
    const double *kt = J->k + ((size_t)t * H + h) * dk;
    const double *gt = J->g + ((size_t)t * H + h) * dk;
    const double *vt = J->v + ((size_t)t * H + h) * dv;
    const double bt = J->beta[(size_t)t * H + h];
    double *ot = J->out + ((size_t)t * H + h) * dv;

    /* forget: scale key channel (row) i of S by alpha_t[i] */
    for (int i = 0; i < dk; ++i) {
      const double a = exp(gt[i]);
      for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;
    }
    /* predict + correct: e = beta (v - S~^T k) */
    for (int j = 0; j < dv; ++j) {
      double pred = 0.0;
      for (int i = 0; i < dk; ++i) pred += S[(size_t)i * dv + j] * kt[i];
      e[j] = bt * (vt[j] - pred);
    }
    /* write: S += k e^T */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += kt[i] * e[j];
    /* read after write: o = scale * S^T q */
    for (int j = 0; j < dv; ++j) {
      double acc = 0.0;
      for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qt[i];
      ot[j] = J->scale * acc;
    }
  }
  if (J->final_state)
    memcpy(J->final_state + state_off, S, sizeof(double) * (size_t)dk * dv);
}

static void *kda_oracle_worker(void *arg) {
  kda_oracle_job *J = (kda_oracle_job *)arg;
  const int64_t pairs = (int64_t)J->num_seqs * J->H;
  double *S = (double *)malloc(sizeof(double) * (size_t)J->dk * J->dv);
  double *e = (double *)malloc(sizeof(double) * (size_t)J->dv);
  for (;;) {
    const int64_t p = __atomic_fetch_add(&J->next_pair, 1, __ATOMIC_RELAXED);
    if (p >= pairs) break;
    kda_oracle_pair(J, (int)(p / J->H), (int)(p % J->H), S, e);
  }
  free(S);
  free(e);
  return NULL;
}

/* Number of host threads the oracle uses when asked for "all cores". */
int kda_oracle_default_threads(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Runs the recurrence for every (sequence, head) pair.
 * init_state may be NULL (zeros); final_state may be NULL (not written).
 * threads <= 0 means one thread per online core.  Returns the thread count
 * used, or -1 on a bad argument.
 */
int kda_oracle_fwd(int num_seqs, const int64_t *cu_seqlens, int H, int dk,
                   int dv, double scale, const double *q, const double *k,
                   const double *v, const double *g, const double *beta,
                   const double *init_state, double *out, double *final_state,
                   int threads) {
  if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
  for (int n = 0; n < num_seqs; ++n)
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
  kda_oracle_job J;
  J.num_seqs = num_seqs;
  J.H = H;
  J.dk = dk;
  J.dv = dv;
  J.cu = cu_seqlens;
  J.scale = scale;
  J.q = q;
  J.k = k;
  J.v = v;
  J.g = g;
  J.beta = beta;
  J.init_state = init_state;
  J.out = out;
  J.final_state = final_state;
  J.next_pair = 0;

  if (threads <= 0) threads = kda_oracle_default_threads();
  const int64_t pairs = (int64_t)num_seqs * H;
  if (threads > pairs) threads = pairs > 0 ? (int)pairs : 1;
  if (threads <= 1) {
    kda_oracle_worker(&J);
    return 1;
  }
  pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)threads);
  int started = 0;
  for (int i = 0; i < threads; ++i)
    if (pthread_create(&tid[i], NULL, kda_oracle_worker, &J) == 0) ++started;
  if (started == 0) kda_oracle_worker(&J);
  for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
  free(tid);
  return started > 0 ? started : 1;
}
