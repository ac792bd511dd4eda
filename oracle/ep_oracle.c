/*
 * CPU oracle for the MoE dispatch / combine layout path -- implementation.
 *
 * TEST INFRASTRUCTURE ONLY (see ep_oracle.h).  Plain C99, one thread, built
 * with -ffp-contract=off so that every fused multiply-add below is the
 * explicit fmaf() it is written as and nothing else is contracted.
 *
 * The layout is computed from its definition with a comparison sort, on
 * purpose unlike the GPU's counting sort.
 */
#include "ep_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16: the upper 16 bits of an IEEE binary32.                              */
/* ------------------------------------------------------------------------ */

float oracle_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Round to nearest, ties to even, as "Deep Dive - DeepEP", "Combine: reverse
 * routing plus reduction" states it for finite values: add 0x7FFF plus the
 * lowest kept bit, then truncate.  That formula is also right for infinities
 * and overflows to infinity; a NaN is returned as a quiet NaN of its sign. */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
    return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
  uint32_t r = (u + 0x7FFFu + ((u >> 16) & 1u)) & 0xFFFF0000u;
  return (uint16_t)(r >> 16);
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 (OCP 8-bit floating point, "E4M3FN"): 1 sign bit, 4 exponent     */
/* bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN, so   */
/* the largest finite magnitude is 1.75 * 2^8 = 448; subnormals are m*2^-9.  */
/* ------------------------------------------------------------------------ */

float oracle_e4m3_to_f32(uint8_t c) {
  int sign = (c & 0x80) != 0;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  double v;
  if (e == 0xF && m == 0x7)
    return sign ? -NAN : NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return (float)(sign ? -v : v);
}

/* n >= 0: nearest integer, halfway cases to the even integer. */
static double round_half_even(double n) {
  double fl = floor(n);
  double d = n - fl;
  if (d > 0.5) return fl + 1.0;
  if (d < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Round to the nearest E4M3 value, ties to the even mantissa; magnitudes
 * that round beyond 448 (and infinities) saturate to +-448 ("satfinite");
 * NaN maps to the NaN code of its sign.  All steps are exact in double: a
 * binary32 value scaled by a power of two. */
uint8_t oracle_f32_to_e4m3(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  if (isnan(v)) return (uint8_t)(sign | 0x7F);
  double a = fabs((double)v);
  if (isinf(a)) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {
    /* subnormal binade: quantum 2^-9; n = 8 is the smallest normal (code 8) */
    double n = round_half_even(a * 512.0);
    return (uint8_t)(sign | (uint8_t)n);
  }
  int ex;
  (void)frexp(a, &ex);          /* a = f * 2^ex, f in [0.5, 1) */
  int E = ex - 1;               /* a in [2^E, 2^(E+1)) */
  if (E > 8) return (uint8_t)(sign | 0x7E);
  double n = round_half_even(ldexp(a, 3 - E));   /* in [8, 16] */
  int code = ((E + 7) << 3) + ((int)n - 8);      /* n == 16 carries */
  if (code > 0x7E) code = 0x7E;                  /* satfinite */
  return (uint8_t)(sign | (uint8_t)code);
}

void oracle_f32_to_bf16_n(int64_t n, const float *in, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(in[i]);
}
void oracle_bf16_to_f32_n(int64_t n, const uint16_t *in, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f32(in[i]);
}
void oracle_f32_to_e4m3_n(int64_t n, const float *in, uint8_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_e4m3(in[i]);
}
void oracle_e4m3_to_f32_n(int64_t n, const uint8_t *in, float *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f32(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Layout                                                                    */
/* ------------------------------------------------------------------------ */

int64_t oracle_recv_capacity(int32_t max_tokens, int32_t num_topk,
                             int32_t num_experts, int32_t alignment) {
  return (int64_t)max_tokens * num_topk +
         (int64_t)num_experts * (alignment - 1);
}

typedef struct {
  int32_t e, t, k;
} entry_t;

/* Order within an expert: source-global order.  Source ranks own contiguous
 * token blocks, so (source rank, token) order is token order, then k. */
static int entry_cmp(const void *pa, const void *pb) {
  const entry_t *a = (const entry_t *)pa, *b = (const entry_t *)pb;
  if (a->e != b->e) return a->e < b->e ? -1 : 1;
  if (a->t != b->t) return a->t < b->t ? -1 : 1;
  if (a->k != b->k) return a->k < b->k ? -1 : 1;
  return 0;
}

int oracle_layout(int32_t T, int32_t K, int32_t E, int32_t R, int32_t A,
                  const int64_t *topk_idx, int64_t cap,
                  int32_t *expert_count, int32_t *expert_start,
                  int32_t *expert_end, int32_t *rank_start,
                  int32_t *tokens_per_rank, uint8_t *is_token_in_rank,
                  int32_t *slot_of, int32_t *src_info) {
  if (T < 0 || K < 1 || E < 1 || R < 1 || A < 1 || E % R != 0)
    return ORACLE_ERR_INVALID_ARG;
  const int32_t Eg = E / R;

  /* 1. validate: -1 is "unused", anything else outside [0, E) is an error
   *    (never Python's last expert); an expert may appear once per token. */
  for (int64_t p = 0; p < (int64_t)T * K; ++p)
    if (topk_idx[p] < -1 || topk_idx[p] >= E) return ORACLE_ERR_EXPERT_RANGE;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k)
      for (int32_t k2 = k + 1; k2 < K; ++k2) {
        int64_t a = topk_idx[(int64_t)t * K + k];
        if (a >= 0 && a == topk_idx[(int64_t)t * K + k2])
          return ORACLE_ERR_DUP_EXPERT;
      }

  /* 2. count per expert */
  for (int32_t e = 0; e < E; ++e) expert_count[e] = 0;
  for (int64_t p = 0; p < (int64_t)T * K; ++p)
    if (topk_idx[p] >= 0) expert_count[topk_idx[p]] += 1;

  /* 3. aligned prefix sum: each segment rounded up to A rows; the end of
   *    expert e's valid rows is its aligned start plus its real count. */
  expert_start[0] = 0;
  for (int32_t e = 0; e < E; ++e) {
    int32_t padded = ((expert_count[e] + A - 1) / A) * A;
    expert_start[e + 1] = expert_start[e] + padded;
    expert_end[e] = expert_start[e] + expert_count[e];
  }
  if ((int64_t)expert_start[E] > cap) return ORACLE_ERR_CAPACITY;
  for (int32_t r = 0; r <= R; ++r) rank_start[r] = expert_start[r * Eg];

  /* 4. per destination rank: a token travels once to each rank that owns at
   *    least one of its experts (owner rank = expert / experts per rank). */
  for (int32_t r = 0; r < R; ++r) tokens_per_rank[r] = 0;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t r = 0; r < R; ++r) {
      uint8_t in = 0;
      for (int32_t k = 0; k < K; ++k) {
        int64_t e = topk_idx[(int64_t)t * K + k];
        if (e >= 0 && e / Eg == r) in = 1;
      }
      is_token_in_rank[(int64_t)t * R + r] = in;
      tokens_per_rank[r] += in;
    }

  /* 5. slots: sort the unmasked (t, k) by (expert, token, k); the i-th entry
   *    of expert e lands at expert_start[e] + i. */
  int64_t n = 0;
  for (int64_t p = 0; p < (int64_t)T * K; ++p) n += topk_idx[p] >= 0;
  entry_t *ent = (entry_t *)malloc((size_t)(n > 0 ? n : 1) * sizeof(entry_t));
  if (!ent) return ORACLE_ERR_INVALID_ARG;
  int64_t j = 0;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) {
      int64_t e = topk_idx[(int64_t)t * K + k];
      if (e >= 0) {
        ent[j].e = (int32_t)e;
        ent[j].t = t;
        ent[j].k = k;
        ++j;
      }
    }
  qsort(ent, (size_t)n, sizeof(entry_t), entry_cmp);

  for (int64_t p = 0; p < (int64_t)T * K; ++p) slot_of[p] = -1;
  for (int64_t s = 0; s < 2 * cap; ++s) src_info[s] = -1;
  int32_t prev_e = -1, rank_in_e = 0;
  for (int64_t i = 0; i < n; ++i) {
    if (ent[i].e != prev_e) {
      prev_e = ent[i].e;
      rank_in_e = 0;
    }
    int32_t slot = expert_start[ent[i].e] + rank_in_e++;
    slot_of[(int64_t)ent[i].t * K + ent[i].k] = slot;
    src_info[2 * (int64_t)slot] = ent[i].t;
    src_info[2 * (int64_t)slot + 1] = ent[i].k;
  }
  free(ent);
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Dispatch                                                                  */
/* ------------------------------------------------------------------------ */

void oracle_dispatch_bf16(int32_t T, int32_t H, int32_t K, int32_t E,
                          const uint16_t *x, const float *w,
                          const int32_t *slot_of, const int32_t *expert_start,
                          const int32_t *expert_end, int zero_padding,
                          uint16_t *recv_x, float *recv_w) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) {
      int32_t s = slot_of[(int64_t)t * K + k];
      if (s < 0) continue;
      memcpy(recv_x + (int64_t)s * H, x + (int64_t)t * H,
             (size_t)H * sizeof(uint16_t));
      if (w && recv_w) recv_w[s] = w[(int64_t)t * K + k];
    }
  if (zero_padding)
    for (int32_t e = 0; e < E; ++e)
      for (int32_t s = expert_end[e]; s < expert_start[e + 1]; ++s) {
        memset(recv_x + (int64_t)s * H, 0, (size_t)H * sizeof(uint16_t));
        if (recv_w) recv_w[s] = 0.0f;
      }
}

/* One fp32 scale per 128 consecutive channels.  amax is the exact maximum of
 * |x|; the scale is amax / 448 (fp32, round to nearest) and is the dequant
 * multiplier (x ~ q * scale); q = E4M3(x / scale) with an fp32 division.  An
 * all-zero block has scale 0 and payload 0. */
static void quantize_row(int32_t H, const uint16_t *xrow, uint8_t *q,
                         float *scale) {
  for (int32_t c = 0; c < H / 128; ++c) {
    float amax = 0.0f;
    for (int32_t i = 0; i < 128; ++i) {
      float a = fabsf(oracle_bf16_to_f32(xrow[c * 128 + i]));
      if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
      scale[c] = 0.0f;
      memset(q + c * 128, 0, 128);
      continue;
    }
    float s = amax / 448.0f;
    scale[c] = s;
    for (int32_t i = 0; i < 128; ++i)
      q[c * 128 + i] = oracle_f32_to_e4m3(oracle_bf16_to_f32(xrow[c * 128 + i]) / s);
  }
}

void oracle_dispatch_fp8(int32_t T, int32_t H, int32_t K, int32_t E,
                         const uint16_t *x, const float *w,
                         const int32_t *slot_of, const int32_t *expert_start,
                         const int32_t *expert_end, int zero_padding,
                         uint8_t *recv_q, float *recv_scale, float *recv_w) {
  const int32_t nb = H / 128;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) {
      int32_t s = slot_of[(int64_t)t * K + k];
      if (s < 0) continue;
      /* recomputed for every slot from x[t]: each copy is defined alone */
      quantize_row(H, x + (int64_t)t * H, recv_q + (int64_t)s * H,
                   recv_scale + (int64_t)s * nb);
      if (w && recv_w) recv_w[s] = w[(int64_t)t * K + k];
    }
  if (zero_padding)
    for (int32_t e = 0; e < E; ++e)
      for (int32_t s = expert_end[e]; s < expert_start[e + 1]; ++s) {
        memset(recv_q + (int64_t)s * H, 0, (size_t)H);
        for (int32_t c = 0; c < nb; ++c) recv_scale[(int64_t)s * nb + c] = 0.0f;
        if (recv_w) recv_w[s] = 0.0f;
      }
}

/* ------------------------------------------------------------------------ */
/* Combine                                                                   */
/* ------------------------------------------------------------------------ */

/* Reverse route plus reduction: each output element is one fp32 fold over the
 * token's unmasked selections in ascending k, applying each gate weight
 * exactly once, then a single cast to bf16 (no bf16 subtotal). */
void oracle_combine(int32_t T, int32_t H, int32_t K, const uint16_t *Y,
                    const float *w, const int32_t *slot_of, uint16_t *y) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t i = 0; i < H; ++i) {
      float acc = 0.0f;
      for (int32_t k = 0; k < K; ++k) {
        int32_t s = slot_of[(int64_t)t * K + k];
        if (s < 0) continue;
        float wk = w ? w[(int64_t)t * K + k] : 1.0f;
        acc = fmaf(wk, oracle_bf16_to_f32(Y[(int64_t)s * H + i]), acc);
      }
      y[(int64_t)t * H + i] = oracle_f32_to_bf16(acc);
    }
}

/* ------------------------------------------------------------------------ */
/* Combine epilogue                                                          */
/* ------------------------------------------------------------------------ */

void oracle_combine_epilogue(int32_t T, int32_t H, int32_t K, const uint16_t *Y,
                             const float *w, const int32_t *slot_of,
                             const uint16_t *b0, const uint16_t *b1,
                             const float *recv_w, uint16_t *y, float *combined_w) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t i = 0; i < H; ++i) {
      float acc = 0.0f;
      for (int32_t k = 0; k < K; ++k) {
        int32_t s = slot_of[(int64_t)t * K + k];
        if (s < 0) continue;
        float wk = w ? w[(int64_t)t * K + k] : 1.0f;
        acc = fmaf(wk, oracle_bf16_to_f32(Y[(int64_t)s * H + i]), acc);
      }
      if (b0) acc = acc + oracle_bf16_to_f32(b0[(int64_t)t * H + i]);
      if (b1) acc = acc + oracle_bf16_to_f32(b1[(int64_t)t * H + i]);
      y[(int64_t)t * H + i] = oracle_f32_to_bf16(acc);
    }
  if (combined_w && recv_w)
    for (int32_t t = 0; t < T; ++t)
      for (int32_t k = 0; k < K; ++k) {
        int32_t s = slot_of[(int64_t)t * K + k];
        combined_w[(int64_t)t * K + k] = s >= 0 ? recv_w[s] : 0.0f;
      }
}

/* ------------------------------------------------------------------------ */
/* FP8 scale layouts, pre-quantised input                                    */
/* ------------------------------------------------------------------------ */

int64_t oracle_scale_ld(int64_t cap) { return (cap + 3) / 4 * 4; }

void oracle_scales_to_col_major(int64_t cap, int32_t nb, const float *row_major,
                                int64_t ld, float *col_major) {
  for (int64_t r = 0; r < cap; ++r)
    for (int32_t c = 0; c < nb; ++c)
      col_major[(int64_t)c * ld + r] = row_major[r * nb + c];
}

void oracle_dispatch_fp8_prequant(int32_t T, int32_t H, int32_t K, int32_t E,
                                  const uint8_t *x_q, const float *x_scale,
                                  const float *w, const int32_t *slot_of,
                                  const int32_t *expert_start,
                                  const int32_t *expert_end, int zero_padding,
                                  uint8_t *recv_q, float *recv_scale,
                                  float *recv_w) {
  const int32_t nb = H / 128;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) {
      int32_t s = slot_of[(int64_t)t * K + k];
      if (s < 0) continue;
      memcpy(recv_q + (int64_t)s * H, x_q + (int64_t)t * H, (size_t)H);
      memcpy(recv_scale + (int64_t)s * nb, x_scale + (int64_t)t * nb,
             (size_t)nb * sizeof(float));
      if (w && recv_w) recv_w[s] = w[(int64_t)t * K + k];
    }
  if (zero_padding)
    for (int32_t e = 0; e < E; ++e)
      for (int32_t s = expert_end[e]; s < expert_start[e + 1]; ++s) {
        memset(recv_q + (int64_t)s * H, 0, (size_t)H);
        for (int32_t c = 0; c < nb; ++c) recv_scale[(int64_t)s * nb + c] = 0.0f;
        if (recv_w) recv_w[s] = 0.0f;
      }
}

/* ------------------------------------------------------------------------ */
/* Backward                                                                  */
/* ------------------------------------------------------------------------ */

void oracle_dispatch_backward(int32_t T, int32_t H, int32_t K,
                              const uint16_t *grad_recv, const float *grad_recv_w,
                              const int32_t *slot_of, uint16_t *grad_x,
                              float *grad_w) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t i = 0; i < H; ++i) {
      float acc = 0.0f;
      for (int32_t k = 0; k < K; ++k) {
        int32_t s = slot_of[(int64_t)t * K + k];
        if (s >= 0) acc = acc + oracle_bf16_to_f32(grad_recv[(int64_t)s * H + i]);
      }
      grad_x[(int64_t)t * H + i] = oracle_f32_to_bf16(acc);
    }
  if (grad_w && grad_recv_w)
    for (int32_t t = 0; t < T; ++t)
      for (int32_t k = 0; k < K; ++k) {
        int32_t s = slot_of[(int64_t)t * K + k];
        grad_w[(int64_t)t * K + k] = s >= 0 ? grad_recv_w[s] : 0.0f;
      }
}

void oracle_combine_backward(int32_t T, int32_t H, int32_t K, const uint16_t *dy,
                             const float *w, const int32_t *slot_of,
                             const uint16_t *Y, uint16_t *grad_Y, float *grad_w) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) {
      int32_t s = slot_of[(int64_t)t * K + k];
      if (s < 0) {
        if (grad_w) grad_w[(int64_t)t * K + k] = 0.0f;
        continue;
      }
      float wk = w ? w[(int64_t)t * K + k] : 1.0f;
      double dot = 0.0;
      for (int32_t i = 0; i < H; ++i) {
        float g = oracle_bf16_to_f32(dy[(int64_t)t * H + i]);
        float prod = wk * g;
        grad_Y[(int64_t)s * H + i] = oracle_f32_to_bf16(prod);
        if (grad_w && Y)
          dot += (double)g * (double)oracle_bf16_to_f32(Y[(int64_t)s * H + i]);
      }
      if (grad_w) grad_w[(int64_t)t * K + k] = Y ? (float)dot : 0.0f;
    }
}

/* ------------------------------------------------------------------------ */
/* Non-expanded (destination-major) stage                                    */
/* ------------------------------------------------------------------------ */

void oracle_rank_layout(int32_t T, int32_t R, const uint8_t *is_token_in_rank,
                        int32_t *rank_row_start, int32_t *rank_slot_of,
                        int32_t *rank_src) {
  rank_row_start[0] = 0;
  for (int32_t r = 0; r < R; ++r) {
    int32_t n = 0;
    for (int32_t t = 0; t < T; ++t) n += is_token_in_rank[(int64_t)t * R + r] != 0;
    rank_row_start[r + 1] = rank_row_start[r] + n;
  }
  for (int32_t r = 0; r < R; ++r) {
    int32_t row = rank_row_start[r];
    for (int32_t t = 0; t < T; ++t) {
      if (is_token_in_rank[(int64_t)t * R + r]) {
        rank_slot_of[(int64_t)t * R + r] = row;
        rank_src[row] = t;
        ++row;
      } else {
        rank_slot_of[(int64_t)t * R + r] = -1;
      }
    }
  }
}

void oracle_dispatch_ranks(int32_t T, int32_t H, int32_t K, int32_t E, int32_t R,
                           const uint16_t *x, const int64_t *topk_idx,
                           const float *w, const int32_t *rank_slot_of,
                           uint16_t *rank_x, int32_t *rank_topk_idx,
                           float *rank_topk_w) {
  const int32_t Eg = E / R;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t r = 0; r < R; ++r) {
      int32_t row = rank_slot_of[(int64_t)t * R + r];
      if (row < 0) continue;
      memcpy(rank_x + (int64_t)row * H, x + (int64_t)t * H, (size_t)H * sizeof(uint16_t));
      for (int32_t k = 0; k < K; ++k) {
        int64_t e = topk_idx[(int64_t)t * K + k];
        int on_rank = e >= 0 && e / Eg == r;
        rank_topk_idx[(int64_t)row * K + k] = on_rank ? (int32_t)(e - (int64_t)r * Eg) : -1;
        if (w && rank_topk_w)
          rank_topk_w[(int64_t)row * K + k] = on_rank ? w[(int64_t)t * K + k] : 0.0f;
      }
    }
}

void oracle_expand(int32_t T, int32_t H, int32_t K, int32_t E, int32_t R,
                   const int64_t *topk_idx, const int32_t *slot_of,
                   const int32_t *rank_slot_of, const uint16_t *rank_x,
                   const float *rank_topk_w, uint16_t *recv_x, float *recv_w) {
  const int32_t Eg = E / R;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t k = 0; k < K; ++k) {
      int64_t e = topk_idx[(int64_t)t * K + k];
      int32_t s = slot_of[(int64_t)t * K + k];
      if (e < 0 || s < 0) continue;
      int32_t row = rank_slot_of[(int64_t)t * R + e / Eg];
      memcpy(recv_x + (int64_t)s * H, rank_x + (int64_t)row * H, (size_t)H * sizeof(uint16_t));
      if (rank_topk_w && recv_w) recv_w[s] = rank_topk_w[(int64_t)row * K + k];
    }
}

void oracle_reduce_ranks(int32_t T, int32_t H, int32_t K, int32_t E, int32_t R,
                         const int64_t *topk_idx, const int32_t *slot_of,
                         const int32_t *rank_slot_of, const uint16_t *Y,
                         const float *w, uint16_t *rank_y) {
  const int32_t Eg = E / R;
  for (int32_t t = 0; t < T; ++t)
    for (int32_t r = 0; r < R; ++r) {
      int32_t row = rank_slot_of[(int64_t)t * R + r];
      if (row < 0) continue;
      for (int32_t i = 0; i < H; ++i) {
        float acc = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
          int64_t e = topk_idx[(int64_t)t * K + k];
          int32_t s = slot_of[(int64_t)t * K + k];
          if (e < 0 || s < 0 || e / Eg != r) continue;
          float wk = w ? w[(int64_t)t * K + k] : 1.0f;
          acc = fmaf(wk, oracle_bf16_to_f32(Y[(int64_t)s * H + i]), acc);
        }
        rank_y[(int64_t)row * H + i] = oracle_f32_to_bf16(acc);
      }
    }
}

void oracle_combine_ranks(int32_t T, int32_t H, int32_t R,
                          const int32_t *rank_slot_of, const uint16_t *rank_y,
                          uint16_t *y) {
  for (int32_t t = 0; t < T; ++t)
    for (int32_t i = 0; i < H; ++i) {
      float acc = 0.0f;
      for (int32_t r = 0; r < R; ++r) {
        int32_t row = rank_slot_of[(int64_t)t * R + r];
        if (row >= 0) acc = acc + oracle_bf16_to_f32(rank_y[(int64_t)row * H + i]);
      }
      y[(int64_t)t * H + i] = oracle_f32_to_bf16(acc);
    }
}
