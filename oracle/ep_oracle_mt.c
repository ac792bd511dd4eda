/*
 * Multi-threaded driver of the CPU oracle, for the timed CPU baseline.
 *
 * TEST INFRASTRUCTURE ONLY (like ep_oracle.c): the benchmark's CPU-baseline
 * leg and the tests are its only callers.
 *
 * It adds no arithmetic.  Dispatch and combine define every output row from
 * one token's data alone ("GPU Microarchitecture: DeepEP from First
 * Principles", 1.1 and 1.2: each token's rows go to, and come back from, its
 * selected experts independently of other tokens), so the tokens are split
 * into contiguous slices and each POSIX thread runs the single-threaded
 * oracle function itself on its slice.  Rows of different tokens are
 * disjoint (a valid layout gives each (t, k) its own row), so the output is
 * the single-threaded oracle's, bit for bit.  The layout stays sequential:
 * it is a global count and prefix sum.  Alignment padding rows are cleared
 * once, after the slices, by the same oracle function over zero tokens.
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#include "ep_oracle.h"

enum { OP_DISPATCH_BF16, OP_DISPATCH_FP8, OP_COMBINE };

typedef struct {
  int op;
  int32_t t0, t1;             /* token slice [t0, t1) */
  int32_t H, K, E;
  const uint16_t *x;          /* dispatch input / combine expert rows */
  const float *w;
  const int32_t *slot_of, *expert_start, *expert_end;
  void *out;                  /* recv_x, recv_q or y */
  float *recv_scale, *recv_w;
} slice_t;

static void *run_slice(void *arg) {
  const slice_t *s = (const slice_t *)arg;
  const int32_t n = s->t1 - s->t0;
  const float *w = s->w ? s->w + (int64_t)s->t0 * s->K : NULL;
  const int32_t *so = s->slot_of + (int64_t)s->t0 * s->K;
  switch (s->op) {
    case OP_DISPATCH_BF16:
      oracle_dispatch_bf16(n, s->H, s->K, s->E, s->x + (int64_t)s->t0 * s->H, w, so,
                           s->expert_start, s->expert_end, 0, (uint16_t *)s->out,
                           s->recv_w);
      break;
    case OP_DISPATCH_FP8:
      oracle_dispatch_fp8(n, s->H, s->K, s->E, s->x + (int64_t)s->t0 * s->H, w, so,
                          s->expert_start, s->expert_end, 0, (uint8_t *)s->out,
                          s->recv_scale, s->recv_w);
      break;
    default:
      /* combine: x is the expert rows (all of them), out the token rows */
      oracle_combine(n, s->H, s->K, s->x, w, so,
                     (uint16_t *)s->out + (int64_t)s->t0 * s->H);
      break;
  }
  return NULL;
}

/* Runs `proto` over [0, T) in nthreads contiguous slices; returns 0, or -1 if
 * a thread could not be started (the slices already started are joined and
 * the rest run on the calling thread, so the result is complete either way). */
static int run_sliced(const slice_t *proto, int32_t T, int32_t nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > T) nthreads = T > 0 ? T : 1;
  slice_t *sl = (slice_t *)malloc(sizeof(slice_t) * (size_t)nthreads);
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  int *started = (int *)calloc((size_t)nthreads, sizeof(int));
  int rc = 0;
  if (!sl || !th || !started) {
    free(sl); free(th); free(started);
    slice_t one = *proto;
    one.t0 = 0;
    one.t1 = T;
    run_slice(&one);
    return -1;
  }
  for (int32_t i = 0; i < nthreads; ++i) {
    sl[i] = *proto;
    sl[i].t0 = (int32_t)((int64_t)T * i / nthreads);
    sl[i].t1 = (int32_t)((int64_t)T * (i + 1) / nthreads);
    started[i] = i > 0 && pthread_create(&th[i], NULL, run_slice, &sl[i]) == 0;
    if (i > 0 && !started[i]) rc = -1;
  }
  run_slice(&sl[0]);
  for (int32_t i = 1; i < nthreads; ++i) {
    if (started[i])
      pthread_join(th[i], NULL);
    else
      run_slice(&sl[i]);
  }
  free(sl); free(th); free(started);
  return rc;
}

int oracle_dispatch_bf16_mt(int32_t T, int32_t H, int32_t K, int32_t E,
                            const uint16_t *x, const float *w,
                            const int32_t *slot_of, const int32_t *expert_start,
                            const int32_t *expert_end, int zero_padding,
                            uint16_t *recv_x, float *recv_w, int32_t nthreads) {
  slice_t p = {OP_DISPATCH_BF16, 0, 0, H, K, E, x, w, slot_of, expert_start,
               expert_end, recv_x, NULL, recv_w};
  int rc = run_sliced(&p, T, nthreads);
  if (zero_padding)
    oracle_dispatch_bf16(0, H, K, E, x, w, slot_of, expert_start, expert_end, 1,
                         recv_x, recv_w);
  return rc;
}

int oracle_dispatch_fp8_mt(int32_t T, int32_t H, int32_t K, int32_t E,
                           const uint16_t *x, const float *w,
                           const int32_t *slot_of, const int32_t *expert_start,
                           const int32_t *expert_end, int zero_padding,
                           uint8_t *recv_q, float *recv_scale, float *recv_w,
                           int32_t nthreads) {
  slice_t p = {OP_DISPATCH_FP8, 0, 0, H, K, E, x, w, slot_of, expert_start,
               expert_end, recv_q, recv_scale, recv_w};
  int rc = run_sliced(&p, T, nthreads);
  if (zero_padding)
    oracle_dispatch_fp8(0, H, K, E, x, w, slot_of, expert_start, expert_end, 1,
                        recv_q, recv_scale, recv_w);
  return rc;
}

int oracle_combine_mt(int32_t T, int32_t H, int32_t K, const uint16_t *Y,
                      const float *w, const int32_t *slot_of, uint16_t *y,
                      int32_t nthreads) {
  slice_t p = {OP_COMBINE, 0, 0, H, K, 0, Y, w, slot_of, NULL, NULL, y, NULL, NULL};
  return run_sliced(&p, T, nthreads);
}
