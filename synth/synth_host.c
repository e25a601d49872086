/*
 * Host filler for the seeded synthetic inputs (see synth_arith.h for the
 * definition). Multithreaded with POSIX threads; every element depends only on
 * (seed, tensor_id, offset + i), so the split across threads does not change
 * any value.
 */
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "synth_arith.h"

typedef struct {
  void *dst;
  uint64_t begin, end;
  uint64_t key, offset;
  double sigma;
  int kind; /* 0 = bf16, 1 = fp32 */
} synth_job;

static void *synth_worker(void *arg) {
  synth_job *j = (synth_job *)arg;
  if (j->kind == 0) {
    uint16_t *d = (uint16_t *)j->dst;
    for (uint64_t i = j->begin; i < j->end; ++i) d[i] = synth_bf16(j->key, j->offset + i, j->sigma);
  } else {
    uint32_t *d = (uint32_t *)j->dst;
    for (uint64_t i = j->begin; i < j->end; ++i) d[i] = synth_f32(j->key, j->offset + i, j->sigma);
  }
  return NULL;
}

static void synth_fill(void *dst, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t offset,
                       double sigma, int kind, int nthreads) {
  enum { MAXT = 256 };
  if (nthreads < 1) nthreads = 1;
  if (nthreads > MAXT) nthreads = MAXT;
  if ((uint64_t)nthreads > n / 65536 + 1) nthreads = (int)(n / 65536 + 1);
  synth_job jobs[MAXT];
  pthread_t th[MAXT];
  const uint64_t key = synth_key(seed, tensor_id);
  for (int t = 0; t < nthreads; ++t) {
    jobs[t].dst = dst;
    jobs[t].begin = n * (uint64_t)t / (uint64_t)nthreads;
    jobs[t].end = n * (uint64_t)(t + 1) / (uint64_t)nthreads;
    jobs[t].key = key;
    jobs[t].offset = offset;
    jobs[t].sigma = sigma;
    jobs[t].kind = kind;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, synth_worker, &jobs[t]) != 0) break;
    started = t;
  }
  synth_worker(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  for (int t = started + 1; t < nthreads; ++t) synth_worker(&jobs[t]); /* threads that failed to start */
}

/* dst[i] = bf16 bits of sigma * normal(seed, tensor_id, offset + i), i < n. */
void synth_fill_bf16(uint16_t *dst, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t offset,
                     double sigma, int nthreads) {
  synth_fill(dst, n, seed, tensor_id, offset, sigma, 0, nthreads);
}

/* dst[i] = fp32 bits of sigma * normal(seed, tensor_id, offset + i), i < n. */
void synth_fill_f32(uint32_t *dst, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t offset,
                    double sigma, int nthreads) {
  synth_fill(dst, n, seed, tensor_id, offset, sigma, 1, nthreads);
}

/* The raw unscaled draw as a double (for statistical checks of the stream). */
void synth_normals_f64(double *dst, uint64_t n, uint64_t seed, uint64_t tensor_id, uint64_t offset) {
  const uint64_t key = synth_key(seed, tensor_id);
  for (uint64_t i = 0; i < n; ++i) dst[i] = synth_normal(key, offset + i);
}

/* Exposed for tests of the rounding routine against an independent reference. */
uint32_t synth_round_bits(double v, int mbits) { return synth_round_e8(v, mbits); }

uint64_t synth_stream_u64(uint64_t key, uint64_t n) { return synth_stream(key, n); }
