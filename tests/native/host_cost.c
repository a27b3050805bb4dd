/*
 * host_cost.c - host time of back-to-back launches through the C ABI.
 *
 * Built by tests/test_gpu_host_cost.py into a small shared object linked
 * against libpa.so.  Each function issues n calls of one entry point with
 * the same arguments (device buffers prepared by the test) and returns the
 * mean host time per call in nanoseconds, or minus the status of the first
 * call that did not return PA_OK.  The calls only queue work; the test
 * synchronizes before and after.
 */
#include <stdint.h>
#include <time.h>

#include "pa.h"

static double now_ns(void) {
  struct timespec t;
  clock_gettime(CLOCK_MONOTONIC, &t);
  return (double)t.tv_sec * 1e9 + (double)t.tv_nsec;
}

double host_cost_decode(int n, void *out, const void *q, const void *k, const void *v,
                        const int32_t *bt, int32_t mb, const int32_t *sl, int32_t b,
                        int32_t hq, int32_t hkv, int32_t d, int32_t bs, int32_t np,
                        float scale, int32_t dt) {
  const double t0 = now_ns();
  for (int i = 0; i < n; ++i) {
    pa_status st = pa_decode(out, q, k, v, bt, mb, sl, b, hq, hkv, d, bs, np, scale,
                             (pa_dtype)dt, 0, 0);
    if (st != PA_OK) return -(double)st;
  }
  return (now_ns() - t0) / n;
}

double host_cost_splitkv(int n, float *po, float *pl, const void *q, const void *k,
                         const void *v, const int32_t *bt, int32_t mb, const int32_t *sl,
                         int32_t b, int32_t hq, int32_t hkv, int32_t d, int32_t bs, int32_t np,
                         float scale, int32_t pps, int32_t ms, int32_t dt) {
  const double t0 = now_ns();
  for (int i = 0; i < n; ++i) {
    pa_status st = pa_decode_splitkv(po, pl, q, k, v, bt, mb, sl, b, hq, hkv, d, bs, np, scale,
                                     pps, ms, (pa_dtype)dt, 0, 0);
    if (st != PA_OK) return -(double)st;
  }
  return (now_ns() - t0) / n;
}

double host_cost_chunk(int n, void *out, const void *q, const void *k, const void *v,
                       const int32_t *bt, int32_t mb, const int32_t *sl, int32_t b, int32_t nq,
                       int32_t hq, int32_t hkv, int32_t d, int32_t bs, int32_t np, float scale,
                       int32_t dt) {
  const double t0 = now_ns();
  for (int i = 0; i < n; ++i) {
    pa_status st = pa_decode_chunk(out, q, k, v, bt, mb, sl, b, nq, hq, hkv, d, bs, np, scale,
                                   (pa_dtype)dt, 0, 0);
    if (st != PA_OK) return -(double)st;
  }
  return (now_ns() - t0) / n;
}
