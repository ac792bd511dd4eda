/*
 * CPU oracle for the MoE dispatch / combine layout path.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-threaded
 * restatement of what the method computes, used to check the CUDA library.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it.  It shares no code, header, table or constant with the CUDA path.
 *
 * Sources (page title, section):
 *  - "GPU Microarchitecture: DeepEP from First Principles", 1.1 (dispatch:
 *    token-major -> destination-major -> expert-major), 1.2 (combine:
 *    Output(T0) = 0.73 x Expert2(T0) + 0.27 x Expert7(T0)), 6.1 (layout
 *    metadata: count, prefix sum, offset), 6.2 (identity metadata),
 *    7.1 (count -> prefix sum -> scatter).
 *  - "Deep Dive - DeepEP": "Dispatch: layout, move, and epilogue" (input
 *    contract, -1 = unused, expanded mode, expert alignment, psum semantics),
 *    "Combine: reverse routing plus reduction" (fp32 accumulation, one final
 *    bf16 cast, the bf16 rounding formula), "Precision: FP8 on the wire, BF16
 *    for the reduction" (one fp32 scale per 128 values), "A four-token routing
 *    ledger" / "A runnable routing ledger" (owner rank = expert / experts per
 *    rank, per-rank dedup, masked selections, padding), "EPHandle: route
 *    metadata with a lifetime" (deterministic order by source-global order).
 *
 * Every function is pinned by the CPU test-suite against worked examples,
 * closed forms, exhaustive codec checks and brute force; none is
 * "parity unpinned".
 */
#ifndef EP_ORACLE_H
#define EP_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_INVALID_ARG = 1,
  ORACLE_ERR_EXPERT_RANGE = 2,
  ORACLE_ERR_DUP_EXPERT = 3,
  ORACLE_ERR_CAPACITY = 4
};

/* ---- number formats ---------------------------------------------------- */
float oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16(float f);   /* round to nearest even */
float oracle_e4m3_to_f32(uint8_t c);
uint8_t oracle_f32_to_e4m3(float v);    /* round to nearest even, satfinite */
/* element-wise array forms of the four codecs above */
void oracle_f32_to_bf16_n(int64_t n, const float *in, uint16_t *out);
void oracle_bf16_to_f32_n(int64_t n, const uint16_t *in, float *out);
void oracle_f32_to_e4m3_n(int64_t n, const float *in, uint8_t *out);
void oracle_e4m3_to_f32_n(int64_t n, const uint8_t *in, float *out);

/* ---- layout ------------------------------------------------------------ */
/* Worst-case rows of the expert-major buffer: every (token, k) unmasked and
 * every expert segment padded by alignment - 1 rows. */
int64_t oracle_recv_capacity(int32_t max_tokens, int32_t num_topk,
                             int32_t num_experts, int32_t alignment);

/* topk_idx [T*K] int64 row-major.  Outputs (all caller-allocated):
 * expert_count[E], expert_start[E+1], expert_end[E], rank_start[R+1],
 * tokens_per_rank[R], is_token_in_rank[T*R], slot_of[T*K],
 * src_info[2*cap] as (token, k) pairs; rows that carry no token are (-1,-1).
 * Returns an ORACLE_* status; on error the outputs are unspecified. */
int oracle_layout(int32_t T, int32_t K, int32_t E, int32_t R, int32_t A,
                  const int64_t *topk_idx, int64_t cap,
                  int32_t *expert_count, int32_t *expert_start,
                  int32_t *expert_end, int32_t *rank_start,
                  int32_t *tokens_per_rank, uint8_t *is_token_in_rank,
                  int32_t *slot_of, int32_t *src_info);

/* ---- dispatch ---------------------------------------------------------- */
/* recv_x[slot_of[t,k]] = x[t] (raw bf16 bits); recv_w[slot] = w[t,k].
 * With zero_padding, rows [expert_end[e], expert_start[e+1]) are zeroed and
 * their recv_w set to 0.  w and recv_w may be NULL (then recv_w untouched). */
void oracle_dispatch_bf16(int32_t T, int32_t H, int32_t K, int32_t E,
                          const uint16_t *x, const float *w,
                          const int32_t *slot_of, const int32_t *expert_start,
                          const int32_t *expert_end, int zero_padding,
                          uint16_t *recv_x, float *recv_w);

/* Fused 1x128 FP8 E4M3 quantisation of each dispatched row:
 * recv_q[slot, H] bytes, recv_scale[slot, H/128] fp32 (dequant multiplier). */
void oracle_dispatch_fp8(int32_t T, int32_t H, int32_t K, int32_t E,
                         const uint16_t *x, const float *w,
                         const int32_t *slot_of, const int32_t *expert_start,
                         const int32_t *expert_end, int zero_padding,
                         uint8_t *recv_q, float *recv_scale, float *recv_w);

/* ---- combine ----------------------------------------------------------- */
/* y[t,i] = bf16( fold over k ascending, slot_of[t,k] >= 0, of
 *               acc = fmaf(w[t,k], Y[slot_of[t,k], i], acc) ), acc0 = +0.
 * w == NULL means every weight is 1 (plain sum of caller-weighted rows). */
void oracle_combine(int32_t T, int32_t H, int32_t K, const uint16_t *Y,
                    const float *w, const int32_t *slot_of, uint16_t *y);

/* ---- combine epilogue ("Deep Dive - DeepEP", "Combine: reverse routing
 * plus reduction": zero, one or two bf16 bias tensors in the combine
 * epilogue; optional return of top-k weights) ------------------------- */
/* y[t,i] = bf16( (fold + b0[t,i]) + b1[t,i] ), fold as in oracle_combine, the
 * bias terms added in fp32 after it (b0/b1 may be NULL: no term).
 * combined_w[t,k] = recv_w[slot_of[t,k]], 0 for a masked selection (NULL:
 * not computed). */
void oracle_combine_epilogue(int32_t T, int32_t H, int32_t K, const uint16_t *Y,
                             const float *w, const int32_t *slot_of,
                             const uint16_t *b0, const uint16_t *b1,
                             const float *recv_w, uint16_t *y, float *combined_w);

/* ---- FP8 scale layouts and pre-quantised input ("Deep Dive - DeepEP",
 * "Precision: FP8 on the wire, BF16 for the reduction": input may be FP8
 * values plus scale factors; a column-major scale layout for TMA paths) -- */
/* Leading dimension of the column-major scale array: cap rounded up to a
 * multiple of 4 fp32 (16 bytes). */
int64_t oracle_scale_ld(int64_t cap);
/* Row-major scales [cap][nb] -> column-major [nb][ld]; entries of rows that
 * are not copied keep their value in col. */
void oracle_scales_to_col_major(int64_t cap, int32_t nb, const float *row_major,
                                int64_t ld, float *col_major);
/* Pre-quantised input: recv_q[slot] = x_q[t] and recv_scale[slot] = x_scale[t]
 * (bit copies), recv_w as in the other dispatches. */
void oracle_dispatch_fp8_prequant(int32_t T, int32_t H, int32_t K, int32_t E,
                                  const uint8_t *x_q, const float *x_scale,
                                  const float *w, const int32_t *slot_of,
                                  const int32_t *expert_start,
                                  const int32_t *expert_end, int zero_padding,
                                  uint8_t *recv_q, float *recv_scale,
                                  float *recv_w);

/* ---- backward ("Deep Dive - DeepEP", combine section, backward duality:
 * for the unweighted route operators dispatch and combine are transposes --
 * copying rows forward becomes summing their gradients backward -- and the
 * gate multiplication needs its own gradient) -------------------------- */
/* Dispatch backward: grad_x[t,i] = bf16( sum over k ascending, slot_of >= 0,
 * of grad_recv[slot, i] ), fp32 from +0.  grad_w[t,k] = grad_recv_w[slot],
 * 0 for a masked selection (both gradient-of-weight pointers may be NULL). */
void oracle_dispatch_backward(int32_t T, int32_t H, int32_t K,
                              const uint16_t *grad_recv, const float *grad_recv_w,
                              const int32_t *slot_of, uint16_t *grad_x,
                              float *grad_w);
/* Combine backward for y[t] = sum_k w[t,k] * Y[slot_of[t,k]] (+ biases):
 * grad_Y[slot, i] = bf16( w[t,k] * dy[t,i] ) (fp32 product, then one bf16
 * rounding; w == NULL: weight 1, a bit copy of dy); rows of masked or
 * padding slots are not written.  grad_w[t,k] = sum_i dy[t,i] * Y[slot, i]
 * evaluated in double and rounded once to fp32, 0 for a masked selection
 * (grad_w and Y may be NULL). */
void oracle_combine_backward(int32_t T, int32_t H, int32_t K, const uint16_t *dy,
                             const float *w, const int32_t *slot_of,
                             const uint16_t *Y, uint16_t *grad_Y, float *grad_w);

/* ---- non-expanded (destination-major) stage ("Deep Dive - DeepEP",
 * "Why expert parallelism needs a communication layer": a token travels
 * once to each selected destination rank, an optional expansion then makes
 * one slot per expert; "Dispatch: layout, move, and epilogue": in
 * non-expanded mode one received row is a source token with its top-k
 * metadata; "GPU Microarchitecture: DeepEP from First Principles" 2.1 and
 * 1.2: receive buffer -> expert buffer, and expert-major -> destination-
 * major -> token-major on the way back) ------------------------------- */
/* Rank rows: rank r owns rows [rank_row_start[r], rank_row_start[r+1]),
 * one per token sent to it, in token order.  rank_slot_of[t*R + r] = row or
 * -1; rank_src[row] = t.  Uses the flags of oracle_layout. */
void oracle_rank_layout(int32_t T, int32_t R, const uint8_t *is_token_in_rank,
                        int32_t *rank_row_start, int32_t *rank_slot_of,
                        int32_t *rank_src);
/* rank_x[row(t,r)] = x[t] (bf16 bits); per row, for each k: local expert id
 * (e - r*E/R) when expert e of (t,k) is on rank r, else -1; its weight there,
 * else 0 (w may be NULL: weights not written). */
void oracle_dispatch_ranks(int32_t T, int32_t H, int32_t K, int32_t E, int32_t R,
                           const uint16_t *x, const int64_t *topk_idx,
                           const float *w, const int32_t *rank_slot_of,
                           uint16_t *rank_x, int32_t *rank_topk_idx,
                           float *rank_topk_w);
/* Expansion: recv_x[slot_of[t,k]] = rank_x[rank_slot_of[t, r(e)]] for every
 * unmasked (t,k), r(e) = e / (E/R); recv_w[slot] = rank_topk_w[row, k]. */
void oracle_expand(int32_t T, int32_t H, int32_t K, int32_t E, int32_t R,
                   const int64_t *topk_idx, const int32_t *slot_of,
                   const int32_t *rank_slot_of, const uint16_t *rank_x,
                   const float *rank_topk_w, uint16_t *recv_x, float *recv_w);
/* Per-rank reduction (the destination rank's partial sum before sending
 * back): rank_y[row(t,r), i] = bf16( fold over k ascending with r(e_k) = r of
 * acc = fmaf(w[t,k], Y[slot_of[t,k], i], acc) ), acc0 = +0, w NULL -> 1. */
void oracle_reduce_ranks(int32_t T, int32_t H, int32_t K, int32_t E, int32_t R,
                         const int64_t *topk_idx, const int32_t *slot_of,
                         const int32_t *rank_slot_of, const uint16_t *Y,
                         const float *w, uint16_t *rank_y);
/* Token-major sum over destination ranks: y[t,i] = bf16( fold over r
 * ascending with rank_slot_of[t,r] >= 0 of acc += rank_y[row, i] ). */
void oracle_combine_ranks(int32_t T, int32_t H, int32_t R,
                          const int32_t *rank_slot_of, const uint16_t *rank_y,
                          uint16_t *y);

/* ---- multi-threaded driver (ep_oracle_mt.c) ------------------------------
 * The functions above, run by nthreads POSIX threads on contiguous token
 * slices (no arithmetic of their own; results equal the single-threaded
 * calls bit for bit).  Return 0, or -1 if a thread could not be started (the
 * work is then finished on the calling thread). */
int oracle_dispatch_bf16_mt(int32_t T, int32_t H, int32_t K, int32_t E,
                            const uint16_t *x, const float *w,
                            const int32_t *slot_of, const int32_t *expert_start,
                            const int32_t *expert_end, int zero_padding,
                            uint16_t *recv_x, float *recv_w, int32_t nthreads);
int oracle_dispatch_fp8_mt(int32_t T, int32_t H, int32_t K, int32_t E,
                           const uint16_t *x, const float *w,
                           const int32_t *slot_of, const int32_t *expert_start,
                           const int32_t *expert_end, int zero_padding,
                           uint8_t *recv_q, float *recv_scale, float *recv_w,
                           int32_t nthreads);
int oracle_combine_mt(int32_t T, int32_t H, int32_t K, const uint16_t *Y,
                      const float *w, const int32_t *slot_of, uint16_t *y,
                      int32_t nthreads);

#ifdef __cplusplus
}
#endif
#endif /* EP_ORACLE_H */
