/*
 * ep.h -- C ABI of the GB300 MoE dispatch / combine layout library
 * (libep_gb300.so, CUDA sm_103a).
 *
 * The library implements the data-parallel hot path of expert-parallel MoE
 * communication as a layout transformation on ONE GPU: expert-parallel ranks
 * are logical destination partitions of a single HBM buffer.
 *
 *   ep_get_layout : topk_idx            -> counts, aligned offsets, slots
 *   ep_dispatch   : token-major x       -> expert-major rows (bf16 or FP8)
 *   ep_combine    : expert-major rows   -> token-major y (gate-weighted)
 *
 * Sources (page title, section):
 *  "GPU Microarchitecture: DeepEP from First Principles" -- 1.1 and 1.2
 *  (dispatch token-major -> destination-major -> expert-major; combine back,
 *  Output(T0) = 0.73 x Expert2(T0) + 0.27 x Expert7(T0)), 6.1 / 6.2 (layout
 *  and identity metadata), 7.1 (count -> prefix sum -> scatter).
 *  "Deep Dive - DeepEP" -- "V2's single interface: ElasticBuffer" (problem
 *  statement: max tokens, hidden, top-k, FP8 dispatch), "Dispatch: layout,
 *  move, and epilogue" (topk_idx / topk_weights contract, -1 = unused,
 *  expanded mode, expert alignment, psum semantics, zero padding, CPU sync),
 *  "Combine: reverse routing plus reduction" (fp32 accumulation, one bf16
 *  cast), "Precision: FP8 on the wire, BF16 for the reduction" (one fp32
 *  scale per 128 values), "EPHandle: route metadata with a lifetime" (the
 *  handle carries route metadata, not gate values; deterministic order).
 *
 * Conventions for every entry point
 *  - Pointers named d_* or documented "device" are CUDA device pointers; all
 *    buffers are allocated and owned by the CALLER.  The library never
 *    allocates or frees memory and keeps no pointer after a call returns.
 *    (The host-buffer entry points, when they copy in chunks, create two
 *    copy streams -- one a direction -- and a few events per device on
 *    first use, kept until exit.)
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued asynchronously on it; a call returns before
 *    the GPU has finished unless documented otherwise.
 *  - Calls that do not synchronise can be recorded into a CUDA graph by
 *    stream capture: the device entry points, and the host-buffer entry
 *    points in both modes (in chunked mode the library's copy streams join
 *    the capture through events; make one chunked call outside any capture
 *    first, which creates them).  ep_get_layout with h_expert_count,
 *    ep_check_error and the self-tests synchronise and cannot be captured.
 *  - Argument errors are detected on the host before anything is launched
 *    and returned synchronously (EP_ERR_INVALID_ARG).  Errors in the routing
 *    data (an expert id outside [-1, E), an expert repeated within a token)
 *    can only be seen on the GPU: they are recorded in the layout's device
 *    error word and reported by ep_check_error (or by ep_get_layout when it
 *    is asked to synchronise).  Kernels never trap.
 *  - Every device pointer must be 16-byte aligned.
 *  - Row-major layouts throughout.  T = num_tokens of the ep_get_layout call
 *    (<= cfg.max_tokens), H = hidden, K = num_topk, E = num_experts,
 *    R = num_ranks, A = expert_alignment, cap = ep_recv_capacity(cfg).
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point (int32_t). */
enum {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1,   /* bad config, pointer, alignment or size      */
  EP_ERR_EXPERT_RANGE = 2,  /* a topk_idx entry outside [-1, E)            */
  EP_ERR_DUP_EXPERT = 3,    /* an expert selected twice by one token       */
  EP_ERR_CAPACITY = 4,      /* a buffer or built-in scratch is too small   */
  EP_ERR_CUDA = 5,          /* a CUDA runtime call failed                  */
  EP_ERR_TIMEOUT = 6,       /* a bounded on-chip wait gave up (no hang)    */
  EP_ERR_TIMEOUT_PENDING = 7 /* as EP_ERR_TIMEOUT, and a bulk copy the
                                waiting CTA had issued was still not done
                                when it returned: it may still write that
                                SM's shared memory, so treat the CUDA
                                context as unreliable                     */
};

/* Problem statement, as in the pages' buffer constructor: max tokens,
 * hidden size, top-k, expert count, FP8 dispatch; plus the logical rank
 * count, the expert alignment and the zero-padding switch of dispatch. */
typedef struct {
  int32_t max_tokens;        /* tokens a layout may hold (capacity planning)   */
  int32_t hidden;            /* H: bf16 channels per row, H <= 2^20; H % 8
                                == 0 for bf16 rows, H % 128 == 0 when
                                use_fp8_dispatch                              */
  int32_t num_topk;          /* K in [1, 32], K <= E                           */
  int32_t num_experts;       /* E in [1, 2048]                                  */
  int32_t num_ranks;         /* R logical ranks, E % R == 0; rank r owns the
                                experts [r*E/R, (r+1)*E/R)                     */
  int32_t expert_alignment;  /* A in [1, 1024]: every expert segment starts
                                at a multiple of A rows                        */
  int32_t use_fp8_dispatch;  /* 0: bf16 rows; 1: E4M3 rows + 1x128 fp32 scales */
  int32_t zero_padding;      /* 1: dispatch clears the alignment gap rows      */
} ep_config;

/* The layout handle: route metadata only (no gate values).  Every pointer is
 * a caller-allocated DEVICE buffer of the size given; ep_get_layout fills
 * them and sets num_tokens.  The handle stays valid, and may be reused by
 * any number of dispatch / combine calls, while the route is unchanged. */
typedef struct {
  int32_t *expert_count;     /* [E]   rows routed to each expert (unaligned)   */
  int32_t *expert_start;     /* [E+1] aligned start row of each expert segment;
                                expert_start[E] = rows in use                  */
  int32_t *expert_end;       /* [E]   expert_start[e] + expert_count[e]: the
                                end of expert e's valid rows (psum semantics)  */
  int32_t *rank_start;       /* [R+1] first row of each logical rank's range
                                (= expert_start[r*E/R])                        */
  int32_t *tokens_per_rank;  /* [R]   tokens sent to each rank, counted once
                                per (token, rank)                              */
  uint8_t *is_token_in_rank; /* [max_tokens*R] 1 if token t has an expert
                                on rank r                                      */
  int32_t *slot_of;          /* [max_tokens*K] row of (t,k) in the expert-major
                                buffer, -1 for an unused (-1) selection        */
  int32_t *src_info;         /* [cap*2] (token, k) of each row in use;
                                (-1,-1) for alignment padding rows             */
  int32_t *err;              /* [1]   device error word                        */
  void *workspace;           /* ep_layout_workspace_bytes(cfg) bytes           */
  /* Optional destination-major rows (all three set, or all NULL): rank r
   * owns rows [rank_row_start[r], rank_row_start[r+1]), one per token sent
   * to it (a token is sent once to every rank owning one of its experts),
   * in token order. */
  int32_t *rank_row_start;   /* [R+1]                                          */
  int32_t *rank_slot_of;     /* [max_tokens*R] rank row of (t, r), or -1       */
  int32_t *rank_src;         /* [max_tokens*min(K,R)] token of each rank row   */
  int32_t num_tokens;        /* set by ep_get_layout                           */
  int32_t reserved;
} ep_layout;

/* Rows the expert-major buffer needs in the worst case:
 * max_tokens*K + E*(A-1).  Returns -1 if the config is invalid. */
EP_API int64_t ep_recv_capacity(const ep_config *cfg);

/* Bytes of device scratch memory ep_get_layout needs in layout->workspace
 * (per-tile expert and rank counts, per-tile error bits); layouts of at
 * most 4096 (t, k) pairs do not touch it.  Returns -1 if the config is
 * invalid. */
EP_API int64_t ep_layout_workspace_bytes(const ep_config *cfg);

/* Layout ("GPU Microarchitecture: DeepEP from First Principles", 6.1 and 7.1;
 * "Deep Dive - DeepEP", "Dispatch: layout, move, and epilogue").
 *
 * d_topk_idx: device int64 [num_tokens, K]; -1 marks an unused selection.
 * Counts rows per expert and per destination rank (a token counts once per
 * rank), lays the experts out contiguously with every segment rounded up to
 * A rows, and assigns each (t, k) its row: within an expert, rows follow
 * source-global order (source rank, token, k) -- the pages' deterministic
 * mode, produced directly.  Logical source ranks own contiguous token
 * blocks, so that order is (t, k) order.  Runs one kernel on `stream` when
 * num_tokens * K <= 4096, else two.  The layout's error word is cleared by
 * the call itself before anything is recorded in it.
 *
 * h_expert_count: NULL for a fully asynchronous call.  If non-NULL (host
 * memory, E int32), the call synchronises `stream`, copies the per-expert
 * counts there and returns the device error status (the pages' CPU-sync
 * path).  Without it, consumers must use only rows [expert_start[e],
 * expert_end[e]) and call ep_check_error to see routing errors.
 * num_tokens may be 0.  Returns EP_OK or an error. */
EP_API int32_t ep_get_layout(const ep_config *cfg, int32_t num_tokens,
                      const int64_t *d_topk_idx, ep_layout *layout,
                      int32_t *h_expert_count, void *stream);

/* Dispatch, expanded mode ("GPU Microarchitecture: DeepEP from First
 * Principles", 1.1; "Deep Dive - DeepEP", "Dispatch: layout, move, and
 * epilogue" and "Precision: FP8 on the wire, BF16 for the reduction").
 *
 * d_x: device bf16 [T, H] (raw 16-bit patterns).
 * d_topk_weights: device fp32 [T, K] or NULL.
 * d_recv_x: device [cap, H]: bf16 rows, or E4M3 bytes when use_fp8_dispatch.
 *   Row slot_of[t,k] receives token t.  bf16 rows are bit copies.  FP8 rows:
 *   per 128-channel block, amax = max|x| (exact), scale = amax / 448 (fp32,
 *   round to nearest), q = E4M3(x / scale) rounded to nearest even with
 *   saturation to +-448; an all-zero block has scale 0 and q = 0.
 * d_recv_scale: device fp32 [cap, H/128] (FP8 only, else ignored; may be
 *   NULL for bf16): the dequantisation multipliers, x ~ q * scale.
 * d_recv_w: device fp32 [cap] or NULL: recv_w[slot_of[t,k]] = w[t,k], one
 *   gate weight per expert row (requires d_topk_weights).
 * With cfg->zero_padding, rows [expert_end[e], expert_start[e+1]) get
 * zero payload, zero scales and zero weight.  Rows at or past
 * expert_start[E] are never written.  Returns EP_OK or an error. */
EP_API int32_t ep_dispatch(const ep_config *cfg, const ep_layout *layout,
                    const void *d_x, const float *d_topk_weights,
                    void *d_recv_x, float *d_recv_scale, float *d_recv_w,
                    void *stream);

/* Combine ("GPU Microarchitecture: DeepEP from First Principles", 1.2;
 * "Deep Dive - DeepEP", "Combine: reverse routing plus reduction").
 *
 * d_expert_out: device bf16 [cap, H] in the layout's row order (the expert
 *   outputs of the dispatched rows).
 * d_topk_weights: device fp32 [T, K], or NULL.  For each token and channel,
 *   acc = +0.0f; for k = 0..K-1 with slot_of[t,k] >= 0:
 *   acc = fmaf(w[t,k], expert_out[slot_of[t,k], i], acc); y = bf16(acc),
 *   round to nearest even.  Each gate weight is applied exactly once; with
 *   NULL every weight is 1, i.e. the plain sum of rows the caller already
 *   weighted (the pages' V2 contract).  Unused selections contribute
 *   nothing and the remaining weights are not renormalised; padding rows
 *   are never read.
 * d_y: device bf16 [T, H].  Returns EP_OK or an error. */
EP_API int32_t ep_combine(const ep_config *cfg, const ep_layout *layout,
                   const void *d_expert_out, const float *d_topk_weights,
                   void *d_y, void *stream);

/* Layout and dispatch in one call ("Deep Dive - DeepEP", "Dispatch: layout,
 * move, and epilogue": a dispatch counts and lays out rows by rank and
 * expert, then moves them -- conceptual stages that kernels can overlap).
 *
 * Same arguments and results as ep_get_layout (with h_expert_count NULL)
 * followed by ep_dispatch of the same num_tokens tokens, and the same errors
 * for the same arguments.  For inputs of at most 4096 (t, k) pairs whose
 * one-launch layout gives each of its CTAs at most 64 pairs, one kernel does
 * both: each CTA of the layout copies the x rows of its own tokens into
 * shared memory while it computes the layout (when they fit beside its
 * other arrays), then dispatches them as soon as their rows are known, so
 * the dispatch costs no second launch.  Larger inputs run the two paths in
 * turn.  (Column-major scales and pre-quantised input are ep_dispatch_fp8's
 * and are not offered here.)  Returns EP_OK or an error. */
EP_API int32_t ep_layout_and_dispatch(const ep_config *cfg, int32_t num_tokens,
                                      const int64_t *d_topk_idx, ep_layout *layout,
                                      const void *d_x, const float *d_topk_weights,
                                      void *d_recv_x, float *d_recv_scale,
                                      float *d_recv_w, void *stream);

/* Allocation-free layout.  The pages have no counterpart: this entry point
 * exists for callers that cannot allocate device memory -- code inside a
 * framework that owns all device memory and has no spare buffer to give, a
 * serving loop that must not allocate after warm-up (cudaMalloc can
 * synchronise the device and fragment a sized pool), or a plugin that only
 * receives the tensors it computes on.
 *
 * Same arguments and results as ep_get_layout, except that
 * layout->workspace is ignored (it may be NULL): the per-tile scratch lives
 * in a 1 MiB array in the library's own device memory, which every GPU that
 * loads the library holds until the process exits.  Only layouts of more
 * than 4096 (t, k) pairs (num_tokens * K > 4096, which take two launches)
 * use scratch; of those, configurations whose ep_layout_workspace_bytes
 * exceeds 1 MiB (152 * 4 * (E rounded up to 4 + R rounded up to 4) + 608
 * bytes) are rejected with EP_ERR_CAPACITY before anything is launched.
 * Smaller layouts are accepted whatever E and R.  Nothing is allocated or
 * freed, by this call or by any routine it calls.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it; make that first call before any
 * stream capture.  All calls share the one array and it keeps the last
 * call's contents; every call writes the scratch it reads before reading
 * it, so nothing has to start at zero.  Calls whose work overlaps on the GPU
 * (e.g. on two streams at once) race on the array: order them. */
EP_API int32_t ep_get_layout_noalloc(const ep_config *cfg, int32_t num_tokens,
                                     const int64_t *d_topk_idx,
                                     ep_layout *layout,
                                     int32_t *h_expert_count, void *stream);

/* Leading dimension (in fp32 entries) of column-major FP8 scales:
 * ep_recv_capacity(cfg) rounded up to a multiple of 4, so that every
 * block's column starts on a 16-byte boundary.  -1 if the config is
 * invalid. */
EP_API int64_t ep_scale_ld(const ep_config *cfg);

/* FP8 dispatch with options ("Deep Dive - DeepEP", "Precision: FP8 on the
 * wire, BF16 for the reduction": the input may arrive as FP8 values plus
 * scale factors; a column-major scale layout serves TMA-fed consumers).
 *
 * Input, exactly one of:
 *   d_x       device bf16 [T, H], quantised as in ep_dispatch (1x128 blocks,
 *             scale = amax / 448, E4M3 round to nearest even, saturating);
 *   d_x_q + d_x_scale  device E4M3 bytes [T, H] and fp32 scales [T, H/128]
 *             of pre-quantised rows, copied bit for bit.
 * d_recv_q: device [cap, H] E4M3 rows (row slot_of[t,k] gets token t).
 * d_recv_scale: device fp32; scale_col_major = 0: [cap, H/128] row-major;
 *   1: [H/128, ep_scale_ld(cfg)] column-major (entry (row, block) at
 *   block * ld + row).
 * d_topk_weights / d_recv_w: as in ep_dispatch.  cfg->zero_padding clears
 * the alignment gap rows (payload, scales in the chosen layout, weights).
 * H % 128 == 0 is required; cfg->use_fp8_dispatch is not consulted.
 * Returns EP_OK or an error. */
EP_API int32_t ep_dispatch_fp8(const ep_config *cfg, const ep_layout *layout,
                               const void *d_x, const uint8_t *d_x_q,
                               const float *d_x_scale,
                               const float *d_topk_weights, uint8_t *d_recv_q,
                               float *d_recv_scale, int32_t scale_col_major,
                               float *d_recv_w, void *stream);

/* Combine with its epilogue ("Deep Dive - DeepEP", "Combine: reverse routing
 * plus reduction": zero, one or two bf16 bias tensors in the combine
 * epilogue; optional return of the top-k weights).
 *
 * As ep_combine, then in fp32 and in this order: acc += bias0[t,i] (if
 * d_bias0), acc += bias1[t,i] (if d_bias1), then one bf16 rounding.  Biases
 * are device bf16 [T, H]; a NULL bias is no term.
 * d_combined_w (device fp32 [T, K], optional; needs d_recv_w, the per-row
 * weights dispatch wrote): combined_w[t,k] = recv_w[slot_of[t,k]], 0 for an
 * unused selection.  With both biases and d_combined_w NULL this is exactly
 * ep_combine.  Returns EP_OK or an error. */
EP_API int32_t ep_combine_epilogue(const ep_config *cfg, const ep_layout *layout,
                                   const void *d_expert_out,
                                   const float *d_topk_weights,
                                   const void *d_bias0, const void *d_bias1,
                                   const float *d_recv_w, void *d_y,
                                   float *d_combined_w, void *stream);

/* Backward of dispatch ("Deep Dive - DeepEP", combine section, backward
 * duality: dispatch and combine are transposes -- copying rows forward
 * becomes summing their gradients backward).
 * d_grad_recv: device bf16 [cap, H], the gradient of the dispatched rows.
 * d_grad_x: device bf16 [T, H]; grad_x[t,i] = bf16( sum over k ascending,
 *   slot_of[t,k] >= 0, of grad_recv[slot_of[t,k], i] ), fp32 from +0.
 * d_grad_recv_w / d_grad_w (both or neither; device fp32 [cap] / [T, K]):
 *   the weights rode along as copies, so grad_w[t,k] =
 *   grad_recv_w[slot_of[t,k]], 0 for an unused selection.
 * Returns EP_OK or an error. */
EP_API int32_t ep_dispatch_backward(const ep_config *cfg, const ep_layout *layout,
                                    const void *d_grad_recv,
                                    const float *d_grad_recv_w, void *d_grad_x,
                                    float *d_grad_w, void *stream);

/* Backward of combine (same source: the transpose of the weighted row sum,
 * and the gate gradient the surrounding autograd needs).
 * d_dy: device bf16 [T, H], the gradient of y.
 * d_grad_expert_out: device bf16 [cap, H]; grad[slot_of[t,k], i] =
 *   bf16( w[t,k] * dy[t,i] ) (fp32 product, one rounding); with
 *   d_topk_weights NULL the weight is 1 and the rows are bit copies of dy
 *   (a dispatch of dy).  Rows of unused selections are not written;
 *   alignment gap rows are zeroed when cfg->zero_padding.
 * d_grad_w (optional, device fp32 [T, K]; needs d_expert_out, the forward
 *   expert rows): grad_w[t,k] = sum_i dy[t,i] * Y[slot_of[t,k], i] in fp32 in
 *   a fixed order (deterministic run to run), 0 for an unused selection.
 * Gradients of the combine biases are dy itself.  Returns EP_OK or an
 * error. */
EP_API int32_t ep_combine_backward(const ep_config *cfg, const ep_layout *layout,
                                   const void *d_dy, const float *d_topk_weights,
                                   const void *d_expert_out,
                                   void *d_grad_expert_out, float *d_grad_w,
                                   void *stream);

/* ---- Non-expanded (destination-major) stage ------------------------------
 * ("Deep Dive - DeepEP", "Why expert parallelism needs a communication
 * layer": a token travels once to each selected destination rank and an
 * optional expansion then makes one slot per expert; "Dispatch: layout,
 * move, and epilogue": in non-expanded mode a received row is a source token
 * with its top-k metadata; "GPU Microarchitecture: DeepEP from First
 * Principles" 2.1 and 1.2: receive buffer -> expert buffer, and on the way
 * back expert-major -> destination-major -> token-major.)
 * All four need a layout computed with the rank-row pointers set
 * (layout->rank_row_start / rank_slot_of / rank_src); rows = rank_row_start[R]
 * <= ep_rank_rows_capacity(cfg).  bf16 rows; d_topk_idx is the int64 [T, K]
 * routing the layout was computed from. */

/* Rows the destination-major buffer may need: max_tokens * min(K, R). */
EP_API int64_t ep_rank_rows_capacity(const ep_config *cfg);

/* rank_x[row(t,r)] = x[t] for every rank r that owns one of token t's
 * experts.  Per rank row, K entries of metadata: d_rank_topk_idx (int32) =
 * local expert id e - r*E/R where the token's k-th expert is on rank r, -1
 * elsewhere; d_rank_topk_w (fp32, optional) = that selection's weight, 0
 * elsewhere.  Returns EP_OK or an error. */
EP_API int32_t ep_dispatch_ranks(const ep_config *cfg, const ep_layout *layout,
                                 const void *d_x, const int64_t *d_topk_idx,
                                 const float *d_topk_weights, void *d_rank_x,
                                 int32_t *d_rank_topk_idx, float *d_rank_topk_w,
                                 void *stream);

/* Expansion: recv_x[slot_of[t,k]] = rank_x[row(t, rank of expert k)] for
 * every (t,k) that is not an unused (-1) selection; d_recv_w[slot] = d_rank_topk_w[row, k] (both or
 * neither).  expand(dispatch_ranks(x)) equals ep_dispatch(x) row for row.
 * cfg->zero_padding clears the alignment gap rows.  Returns EP_OK or an
 * error. */
EP_API int32_t ep_expand(const ep_config *cfg, const ep_layout *layout,
                         const int64_t *d_topk_idx, const void *d_rank_x,
                         const float *d_rank_topk_w, void *d_recv_x,
                         float *d_recv_w, void *stream);

/* Per-rank reduction, the destination rank's partial sum before the rows go
 * back: rank_y[row(t,r), i] = bf16( fold over k ascending whose expert is on
 * rank r of acc = fmaf(w[t,k], expert_out[slot_of[t,k], i], acc) ), acc from
 * +0, weight 1 when d_topk_weights is NULL.  The bf16 partial is the extra
 * rounding of a two-stage reduction ("Combine: reverse routing plus
 * reduction": 256 + 1 rounds to 256, then 256 - 256 = 0).  Returns EP_OK or
 * an error. */
EP_API int32_t ep_reduce_ranks(const ep_config *cfg, const ep_layout *layout,
                               const int64_t *d_topk_idx, const void *d_expert_out,
                               const float *d_topk_weights, void *d_rank_y,
                               void *stream);

/* Token-major sum over destination ranks: y[t,i] = bf16( fold over r
 * ascending with a row for (t, r) of acc += rank_y[row, i] ), fp32 from +0.
 * Needs R <= 64.  Returns EP_OK or an error. */
EP_API int32_t ep_combine_ranks(const ep_config *cfg, const ep_layout *layout,
                                const void *d_rank_y, void *d_y, void *stream);

/* ---- Host buffers ---------------------------------------------------------
 * For callers whose token rows live in host memory (CPU-resident activations,
 * a serving loop that stages batches on the host).  Results equal
 * ep_dispatch / ep_combine bit for bit.  num_chunks selects how the rows
 * cross the host link:
 *  - 0 (direct): no copy and no staging buffer.  The kernel reads
 *    (dispatch) or writes (combine) the host rows in place, each byte once
 *    over the link, on `stream` alone.  The host buffer must be page-locked
 *    memory the device can address (cudaHostAlloc, or cudaHostRegister with
 *    mapping) whose device address is 16-byte aligned, else
 *    EP_ERR_INVALID_ARG; the staging pointer is not used and may be NULL.
 *    Where kernels reach the link's rate, this saves the staging traffic
 *    and the chunk hand-offs.
 *  - 1..64 (chunked): the rows move in token chunks on a copy stream the
 *    library owns, and each chunk's dispatch or combine waits only for its
 *    own chunk's copy ("Deep Dive - DeepEP", "EventOverlap: a stream
 *    contract": streams let data movement and compute overlap; readiness is
 *    a stream dependency on an event, not a host wait).  num_chunks is an
 *    upper bound: a chunk carries at least 4 MiB of rows (T rows of 2H
 *    bytes split into n = min(num_chunks, max(1, floor(2HT / 4 MiB)))
 *    chunks of ceil(T / n) tokens, the last ragged); a single chunk is
 *    copied on `stream` itself, with no copy stream involved.  The first
 *    chunked call on a device creates that device's two copy streams, one
 *    for rows coming in (ep_dispatch_from_host) and one for rows going out
 *    (ep_combine_to_host), and their events (kept until exit).  Calls of
 *    one direction on one device share its stream, so their copies run in
 *    call order; the two directions run at once, so a combine's rows going
 *    out can overlap the next batch's rows coming in when the two calls
 *    are on different streams.  Calls are made from one host thread at a
 *    time.  Host buffers should be pinned (page-locked): pageable memory
 *    works but its copies do not overlap. */

/* As ep_dispatch with x in host memory (h_x: host bf16 [T, H]).  Direct
 * (num_chunks = 0): the dispatch kernel reads h_x in place; d_x is unused.
 * Chunked: h_x is copied into d_x (device bf16 [T, H], a staging buffer the
 * caller owns and that holds x afterwards) chunk by chunk, overlapped with
 * the dispatch of the chunks already copied; the copies start once the work
 * enqueued on `stream` before this call is done (so d_x may still be read
 * by it).  cfg->use_fp8_dispatch and cfg->zero_padding act as in
 * ep_dispatch.  Returns EP_OK or an error. */
EP_API int32_t ep_dispatch_from_host(const ep_config *cfg, const ep_layout *layout,
                                     const void *h_x, void *d_x,
                                     const float *d_topk_weights, void *d_recv_x,
                                     float *d_recv_scale, float *d_recv_w,
                                     int32_t num_chunks, void *stream);

/* As ep_combine with y returned to host memory (h_y: host bf16 [T, H]).
 * Direct (num_chunks = 0): the combine kernel writes h_y in place; d_y is
 * unused.  Chunked: each chunk of tokens is combined into d_y (device bf16
 * [T, H], staging owned by the caller) and then copied to h_y while later
 * chunks combine.  Either way, work enqueued on `stream` after this call
 * starts after the last row reached h_y, so a synchronisation of `stream`
 * makes h_y readable.  Returns EP_OK or an error. */
EP_API int32_t ep_combine_to_host(const ep_config *cfg, const ep_layout *layout,
                                  const void *d_expert_out, const float *d_topk_weights,
                                  void *d_y, void *h_y, int32_t num_chunks, void *stream);

/* Synchronises `stream` and returns the status recorded in the layout's
 * device error word by the last layout call (EP_OK if none): routing errors,
 * else EP_ERR_TIMEOUT_PENDING or EP_ERR_TIMEOUT if one of its bounded
 * on-chip waits gave up.  Each layout call clears the word before its
 * kernels record anything, so a status never carries over from an earlier
 * call.  After a timeout, part of the layout was not written: do not use it
 * for dispatch or combine. */
EP_API int32_t ep_check_error(const ep_layout *layout, void *stream);

/* Self-test of the FP8 dispatch arithmetic ("Deep Dive - DeepEP",
 * "Precision: FP8 on the wire, BF16 for the reduction": one fp32 scale per
 * 128 values; the scale here is amax / 448 and each value is quantised from
 * x / scale rounded to nearest).  The dispatch forms x / scale as a product
 * with the block's reciprocal plus one fused multiply-add correction, which
 * may differ from the IEEE quotient in its last bit (blocks whose scale is
 * below 2^-100 or infinite divide); this runs the dispatch's quotient for
 * every positive bf16 block maximum, finite or +inf, and every bf16 value x
 * with |x| <= amax (about 2^31 pairs: the whole non-NaN input domain)
 * beside the IEEE division and compares the E4M3 codes.
 * d_counts: device uint64 [3], 16-byte aligned: [0] = pairs whose E4M3
 * codes differ (0: the dispatch's codes equal those of the IEEE division),
 * [1] = pairs whose fp32 quotients differ, [2] = those of them whose IEEE
 * quotient is a normal fp32 number (information only).  d_first: device
 * int32, -1 or (amax bits << 16 | x bits) of one code mismatch.
 * Asynchronous on `stream`.  Returns EP_OK or an error. */
EP_API int32_t ep_selftest_fp8_quotient(uint64_t *d_counts, int32_t *d_first,
                                        void *stream);

/* Self-test of the bounded on-chip wait (the layout kernel's wait for its
 * bulk copies):
 * launches one CTA that waits on a shared-memory barrier nothing will ever
 * complete, with a limit of timeout_ns nanoseconds.  The wait gives up, the
 * kernel records EP_ERR_TIMEOUT in d_err (device int32, OR-ed in) and
 * returns; the GPU context stays usable.  Synchronises `stream` and returns
 * the recorded status (EP_ERR_TIMEOUT when the mechanism works).
 * timeout_ns must be in [1000, 10^9]. */
EP_API int32_t ep_selftest_wait_timeout(int64_t timeout_ns, int32_t *d_err,
                                        void *stream);

/* Self-test of the layout's own bounded wait ("Deep Dive - DeepEP",
 * "Benchmark and failure-mode checklist": a timeout is a failure boundary,
 * reported, never a hang).  Runs the two-launch layout of ep_get_layout
 * (same arguments; num_tokens * K above 4096 or E above 2048, so that the
 * layout takes two launches) except that CTA `stall_tile` of its second
 * kernel issues no copy of the per-tile counts and waits for it with a
 * limit of timeout_ns nanoseconds (in [1000, 10^9]).  That wait gives up,
 * the CTA records EP_ERR_TIMEOUT in the layout's error word and returns
 * without writing its rows; the other CTAs finish.  stall_tile must be in
 * [0, CTAs of that kernel): 0 .. max(tiles, min(E, 152)) - 1, where tiles
 * is the number of token tiles (at most 152).  Synchronises `stream` and
 * returns the recorded status (EP_ERR_TIMEOUT when the mechanism works);
 * the layout it leaves is incomplete and must not be used. */
EP_API int32_t ep_selftest_layout_timeout(const ep_config *cfg, int32_t num_tokens,
                                          const int64_t *d_topk_idx, ep_layout *layout,
                                          int32_t stall_tile, int64_t timeout_ns,
                                          void *stream);

/* The cudaError_t of the last CUDA runtime call of this library that failed
 * in the calling thread (0 if none since the previous query); reading it
 * clears it.  Explains an EP_ERR_CUDA status. */
EP_API int32_t ep_last_cuda_error(void);

/* Static, human-readable name of a status code. */
EP_API const char *ep_status_str(int32_t status);

#ifdef __cplusplus
}
#endif
#endif /* EP_GB300_H */
