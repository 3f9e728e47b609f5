/*
 * Host build of the seeded input generator (see synth_core.h for the
 * definition).  Fills caller-owned host arrays; element i of a fill is the
 * generator's element (offset + i) of stream (seed, tid).  Large fills are
 * split over threads; the result does not depend on the thread count.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#include "synth_core.h"

typedef struct {
  int kind;
  uint64_t key, key2;
  uint64_t offset;
  int64_t lo, hi;
  float scale;
  float hot_prob;
  const float* hotvec;
  int32_t dim;
  void* out;
} syn_job;

enum { K_NORMAL_F32 = 0, K_NORMAL_BF16 = 1, K_UNIFORM_F32 = 2, K_E4M3 = 3, K_KEYS = 4 };

static void run_range(const syn_job* j) {
  for (int64_t i = j->lo; i < j->hi; ++i) {
    uint64_t g = j->offset + (uint64_t)i;
    switch (j->kind) {
      case K_NORMAL_F32:
        ((float*)j->out)[i] = syn_normal(j->key, g) * j->scale;
        break;
      case K_NORMAL_BF16:
        ((uint16_t*)j->out)[i] = syn_bf16_rne(syn_normal(j->key, g) * j->scale);
        break;
      case K_UNIFORM_F32:
        ((float*)j->out)[i] = syn_uniform(j->key, g);
        break;
      case K_E4M3:
        ((uint8_t*)j->out)[i] = syn_e4m3_rne(syn_normal(j->key, g) * j->scale);
        break;
      case K_KEYS: {
        /* element g of a [rows, dim] key tensor; row r = g / dim is "hot" with
         * probability hot_prob and then gets hotvec added along its row. */
        uint64_t r = g / (uint64_t)j->dim;
        uint64_t d = g % (uint64_t)j->dim;
        float v = syn_normal(j->key, g);
        if (j->hotvec && syn_uniform(j->key2, r) < j->hot_prob) v = v + j->hotvec[d];
        ((float*)j->out)[i] = v;
        break;
      }
    }
  }
}

static void* worker(void* p) {
  run_range((const syn_job*)p);
  return NULL;
}

static void run(syn_job base, int64_t n, int nthreads) {
  if (n <= 0) return;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < 65536 || nthreads == 1) {
    base.lo = 0;
    base.hi = n;
    run_range(&base);
    return;
  }
  pthread_t th[256];
  syn_job jobs[256];
  int64_t per = (n + nthreads - 1) / nthreads;
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = base;
    jobs[t].lo = (int64_t)t * per;
    jobs[t].hi = jobs[t].lo + per < n ? jobs[t].lo + per : n;
    if (jobs[t].lo >= jobs[t].hi) break;
    if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) {
      run_range(&jobs[t]);
      th[t] = 0;
    }
    started = t + 1;
  }
  for (int t = 0; t < started; ++t)
    if (th[t]) pthread_join(th[t], NULL);
}

uint64_t syn_stream_key(uint64_t seed, uint64_t tid) { return syn_key(seed, tid); }

void syn_host_normal_f32(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float scale,
                         float* out, int nthreads) {
  syn_job j = {K_NORMAL_F32, syn_key(seed, tid), 0, offset, 0, 0, scale, 0.f, NULL, 1, out};
  run(j, n, nthreads);
}

void syn_host_normal_bf16(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float scale,
                          uint16_t* out, int nthreads) {
  syn_job j = {K_NORMAL_BF16, syn_key(seed, tid), 0, offset, 0, 0, scale, 0.f, NULL, 1, out};
  run(j, n, nthreads);
}

void syn_host_uniform_f32(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float* out,
                          int nthreads) {
  syn_job j = {K_UNIFORM_F32, syn_key(seed, tid), 0, offset, 0, 0, 1.f, 0.f, NULL, 1, out};
  run(j, n, nthreads);
}

void syn_host_e4m3_normal(uint64_t seed, uint64_t tid, uint64_t offset, int64_t n, float scale,
                          uint8_t* out, int nthreads) {
  syn_job j = {K_E4M3, syn_key(seed, tid), 0, offset, 0, 0, scale, 0.f, NULL, 1, out};
  run(j, n, nthreads);
}

void syn_host_keys(uint64_t seed, uint64_t tid, uint64_t tid_hot, uint64_t offset, int64_t n,
                   int32_t dim, float hot_prob, const float* hotvec, float* out, int nthreads) {
  syn_job j = {K_KEYS, syn_key(seed, tid), syn_key(seed, tid_hot), offset, 0, 0, 1.f, hot_prob,
               hotvec, dim, out};
  run(j, n, nthreads);
}
