/*
 * kda_host_decode.c -- single-token KDA decode on the host's CPU cores.
 *
 * A separate host tool, not part of the GPU library: libkda_gb300.so neither links
 * nor calls it, and it calls nothing of the GPU library.  It serves a decode step
 * where no GPU is at hand, as the pages' pure-PyTorch shim runs the recurrence on a
 * CPU ("Kimi Delta Attention (KDA)", brain.bigb.es, the last section: the same
 * state and outputs from the chunked and the recurrent schedule, on a laptop CPU).
 *
 * One step of the recurrence per (sequence, head), in fp32, the state d_k x d_v
 * row-major and updated in place ("Kimi Delta Attention (KDA)", the five-line
 * recurrence; "K3 架构图解" Ch.08, the column-vector form):
 *   S~ = Diag(alpha) S,  e = beta (v - S~^T k),  S <- S~ + k e^T,  o = scale S^T q
 * Two passes over the state: decay and predict (S~ and S~^T k), then write and read
 * (S <- S~ + k e^T and S^T q); the inner loops run over d_v, so they vectorise.
 * The (sequence, head) pairs are split over POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include "kda_host_decode.h"

typedef struct {
  int pairs, begin, end, d_k, d_v, gate;
  float scale;
  const float *q, *k, *v, *g, *beta;
  float *state, *out;
} job_t;

static void step_pair(const job_t *j, int p, float *pred) {
  const int dk = j->d_k, dv = j->d_v;
  const float *q = j->q + (size_t)p * dk, *k = j->k + (size_t)p * dk;
  const float *v = j->v + (size_t)p * dv;
  float *S = j->state + (size_t)p * dk * dv, *o = j->out + (size_t)p * dv;
  const float a_tok = j->gate == KDA_HOST_GATE_SCALAR ? expf(j->g[p]) : 1.0f;
  memset(pred, 0, sizeof(float) * (size_t)dv);
  /* pass 1: S~ = Diag(alpha) S and pred = S~^T k */
  for (int i = 0; i < dk; ++i) {
    const float a = j->gate == KDA_HOST_GATE_CHANNEL ? expf(j->g[(size_t)p * dk + i]) : a_tok;
    const float ki = k[i];
    float *row = S + (size_t)i * dv;
    for (int c = 0; c < dv; ++c) {
      row[c] *= a;
      pred[c] += ki * row[c];
    }
  }
  /* e = beta (v - pred), kept in pred */
  const float b = j->beta[p];
  for (int c = 0; c < dv; ++c) pred[c] = b * (v[c] - pred[c]);
  /* pass 2: S <- S~ + k e^T and o = scale S^T q */
  memset(o, 0, sizeof(float) * (size_t)dv);
  for (int i = 0; i < dk; ++i) {
    const float ki = k[i], qi = q[i];
    float *row = S + (size_t)i * dv;
    for (int c = 0; c < dv; ++c) {
      row[c] += ki * pred[c];
      o[c] += qi * row[c];
    }
  }
  for (int c = 0; c < dv; ++c) o[c] *= j->scale;
}

static void *run_jobs(void *arg) {
  const job_t *j = (const job_t *)arg;
  float *pred = (float *)malloc(sizeof(float) * (size_t)j->d_v);
  if (!pred) return (void *)1;
  for (int p = j->begin; p < j->end; ++p) step_pair(j, p, pred);
  free(pred);
  return NULL;
}

int kda_host_decode_default_threads(void) {
  const long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

int kda_host_decode_step(int num_seqs, int num_heads, int d_k, int d_v, float scale, int gate,
                         const float *q, const float *k, const float *v, const float *g,
                         const float *beta, float *state, float *out, int threads) {
  if (num_seqs < 0 || num_heads < 1 || d_k < 1 || d_v < 1) return KDA_HOST_ERR_SHAPE;
  if (gate < KDA_HOST_GATE_CHANNEL || gate > KDA_HOST_GATE_NONE) return KDA_HOST_ERR_SHAPE;
  const long long pairs = (long long)num_seqs * num_heads;
  if (pairs > (1LL << 30)) return KDA_HOST_ERR_SHAPE;
  if (pairs == 0) return KDA_HOST_OK;
  if (!q || !k || !v || !beta || !state || !out || (gate != KDA_HOST_GATE_NONE && !g))
    return KDA_HOST_ERR_NULL;
  if (!(scale > 0.0f)) scale = 1.0f / sqrtf((float)d_k);
  if (threads < 1) threads = kda_host_decode_default_threads();
  if (threads > pairs) threads = (int)pairs;
  job_t *jobs = (job_t *)calloc((size_t)threads, sizeof(job_t));
  pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return KDA_HOST_ERR_MEMORY;
  }
  int rc = KDA_HOST_OK, started = 0;
  for (int t = 0; t < threads; ++t) {
    job_t *j = &jobs[t];
    j->pairs = (int)pairs;
    j->begin = (int)(pairs * t / threads);
    j->end = (int)(pairs * (t + 1) / threads);
    j->d_k = d_k;
    j->d_v = d_v;
    j->gate = gate;
    j->scale = scale;
    j->q = q; j->k = k; j->v = v; j->g = g; j->beta = beta;
    j->state = state;
    j->out = out;
  }
  /* thread 0's share runs on the calling thread */
  for (int t = 1; t < threads; ++t) {
    if (pthread_create(&tids[t], NULL, run_jobs, &jobs[t]) != 0) {
      rc = KDA_HOST_ERR_THREAD;
      break;
    }
    started = t;
  }
  if (rc == KDA_HOST_OK && run_jobs(&jobs[0]) != NULL) rc = KDA_HOST_ERR_MEMORY;
  for (int t = 1; t <= started; ++t) {
    void *res = NULL;
    pthread_join(tids[t], &res);
    if (res != NULL && rc == KDA_HOST_OK) rc = KDA_HOST_ERR_MEMORY;
  }
  if (rc == KDA_HOST_ERR_THREAD) {
    /* the shares of the threads that did not start run here */
    for (int t = started + 1; t < threads; ++t) run_jobs(&jobs[t]);
    run_jobs(&jobs[0]);
    rc = KDA_HOST_OK;
  }
  free(jobs);
  free(tids);
  return rc;
}
