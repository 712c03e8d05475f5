/*
 * ep.h -- C ABI of the single-GPU MoE dispatch / combine library (libep.so).
 *
 * One GPU, logical ranks: the experts 0..E-1 are owned by R logical ranks in
 * contiguous blocks of L = E / R; token t comes from logical rank t / M
 * (M = num_max_tokens_per_rank).  The three steps of the hot path are
 *
 *   ep_layout    routing layout from topk_idx: counts, prefix sums, the
 *                destination row of every (token, slot) and per-row source
 *                metadata;
 *   ep_dispatch  copy epilogue: the rows of x (BF16, or FP8 e4m3 with 1x128
 *                fp32 scales) land in the rank layout or in the expert-
 *                expanded, alignment-padded layout;
 *   ep_combine   per-token weighted gather-reduce of the expert outputs back
 *                to source-token order, fp32 accumulation, BF16 result;
 *
 * plus the backward pair (ep_dispatch_backward, ep_combine_backward) and
 * ep_handle_free.  The arguments follow the dispatch / combine / handle
 * contract described in "DeepEP V2 notes, ch. 7: how V2 dispatch builds
 * expert inputs" (§7.1 input contract, §7.2 layout metadata and allocation,
 * §7.3 copy epilogue, §7.5 handle reuse) and "DeepEP V2 notes, ch. 8:
 * combine, handle and async overlap" (§8.1 combine along the handle, §8.2
 * streams).  There is no communication: every "rank" lives in this GPU's HBM.
 *
 * Conventions for every entry point
 *   - All pointers named x, y, recv_*, out, bias*, topk_* are DEVICE pointers
 *     owned by the caller; `cfg`, `info`, `out_handle`, `rows` are HOST
 *     pointers.  Matrices are dense row-major with no padding between rows.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and is ordered after earlier work on that stream.  Nothing is
 *     synchronised with the host except the count wait of do_cpu_sync.
 *   - Errors are returned as ep_status; no exception crosses the ABI.  On any
 *     status other than EP_OK (and EP_ERR_BAD_TOPK_IDX, see ep_layout)
 *     nothing is allocated and no output is defined.
 *   - The calling thread's current CUDA device must be the device that owns
 *     the pointers.
 */
#ifndef EP_H_
#define EP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

/* Same type as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *ep_stream_t;

typedef enum ep_status {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1,   /* bad config value, NULL or misaligned pointer */
  EP_ERR_UNSUPPORTED = 2,   /* valid but outside this build's limits */
  EP_ERR_BAD_TOPK_IDX = 3,  /* a topk_idx value outside [-1, num_experts) */
  EP_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  EP_ERR_OOM = 5,           /* device or pinned host allocation failed */
  EP_ERR_TIMEOUT = 6,       /* do_cpu_sync: counts not ready before the deadline */
  EP_ERR_OVERFLOW = 7       /* upper-bound allocation exceeded (repeated experts) */
} ep_status;

/* Bits of the device error word (ep_layout_info.error_word). */
#define EP_ERRBIT_BAD_TOPK_IDX 1u  /* value outside [-1, E): the slot is treated as empty */
#define EP_ERRBIT_OVERFLOW 2u      /* rows at or past rows_alloc (or past an expert's
                                      fixed capacity) were dropped */
#define EP_ERRBIT_TIMEOUT 4u       /* a bounded device-side wait gave up (output undefined) */

/* Build limits (checked by ep_validate_config). */
#define EP_MAX_TOPK 32
#define EP_MAX_EXPERTS 2048
#define EP_MAX_HIDDEN 32768

/*
 * Parameters of one layout; copied into the handle.  Field meaning follows
 * the dispatch arguments of §7.2 (num_experts, expert_alignment,
 * num_max_tokens_per_rank, do_cpu_sync, do_expand, do_zero_padding,
 * use_tma_aligned_col_major_sf) and §7.1 (topk).
 */
typedef struct ep_config {
  int32_t num_tokens;               /* T >= 0 */
  int32_t num_topk;                 /* K in [1, EP_MAX_TOPK] */
  int32_t num_experts;              /* E in [1, EP_MAX_EXPERTS], E % R == 0 */
  int32_t num_ranks;                /* R >= 1 logical ranks */
  int32_t hidden;                   /* H, multiple of 8 (of 128 with use_fp8) */
  int32_t num_max_tokens_per_rank;  /* M >= 1, T <= M * R */
  int32_t expert_alignment;         /* A >= 1 */
  int32_t topk_idx_is_int64;        /* 1: topk_idx is int64 (torch default), 0: int32 */
  uint8_t do_expand;                /* 1: expert-expanded layout, 0: rank layout */
  uint8_t do_zero_padding;          /* expanded only: zero the alignment padding rows */
  uint8_t do_cpu_sync;              /* 1: wait for the counts, exact allocation */
  uint8_t use_fp8;                  /* dispatch quantises to e4m3 + fp32 scales */
  uint8_t use_tma_aligned_col_major_sf; /* FP8 scales column-major, 16 B aligned */
  uint8_t fixed_capacity;           /* 1: fixed-capacity per-expert layout (below) */
  uint8_t reserved0[2];             /* must be 0 */
  int32_t num_sms;                  /* 0 = all SMs; otherwise cap on the SMs used */
  int32_t cpu_sync_timeout_ms;      /* do_cpu_sync deadline; 0 = 10000 ms */
} ep_config;

/*
 * Fixed-capacity per-expert layout (fixed_capacity = 1; DeepEP README,
 * "Interfaces and examples", low_latency_dispatch: a per-rank
 * [local experts, max tokens per rank * ranks, hidden] receive tensor and a
 * per-expert count, usable under CUDA graphs).  Requires do_expand = 1,
 * expert_alignment = 1, do_zero_padding = 0 and E * M * R < 2^31.  With
 * capacity = M * R, expert e owns rows [e * capacity, (e + 1) * capacity):
 * its i-th slot in (token, slot) order lands at row e * capacity + i, and
 * rows past cnt_expert[e] are not written.  rows_alloc = E * capacity in
 * both sync modes.  A slot whose position reaches the capacity (only when a
 * token repeats an expert) is dropped and sets EP_ERRBIT_OVERFLOW.  FP8
 * scales: row-major [E * capacity, H/128], or, with
 * use_tma_aligned_col_major_sf, one column-major slab per expert --
 * sf[e * sf_expert_stride + j * sf_hidden_stride + i], sf_hidden_stride =
 * align(capacity, 4), sf_expert_stride = (H/128) * sf_hidden_stride.
 */

/*
 * Filled by ep_layout.  Device pointers are owned by the handle and stay
 * valid until ep_handle_free; they are stream-ordered on the layout stream.
 */
typedef struct ep_layout_info {
  int64_t num_recv_tokens;      /* rank-layout rows; exact with do_cpu_sync, else -1 */
  int64_t num_expanded_tokens;  /* aligned expanded rows; exact with do_cpu_sync, else -1 */
  int64_t rows_alloc;           /* rows the caller allocates for recv_x and friends:
                                   the exact total (do_cpu_sync) or the upper bound */
  int64_t sf_numel;             /* fp32 elements of recv_sf (FP8 only, else 0) */
  int64_t sf_token_stride;      /* recv_sf[row * sf_token_stride + j * sf_hidden_stride] */
  int64_t sf_hidden_stride;
  const int32_t *topk_idx;            /* [T, K] int32 copy, invalid values -> -1 */
  const int32_t *cnt_expert;          /* [E] valid slots per expert (unaligned) */
  const int32_t *cnt_expert_aligned;  /* [E] counts rounded up to A */
  const int32_t *psum_expert;         /* [E+1] exclusive prefix of the aligned counts */
  const int32_t *cnt_rank;            /* [R] tokens received per rank */
  const int32_t *psum_rank;           /* [R+1] exclusive prefix of cnt_rank */
  const int32_t *psum_rank_src;       /* [R, R+1] per receiving rank, prefix over source ranks */
  const int32_t *dst_buffer_slot_idx; /* [T, K] destination row or -1 */
  const int32_t *recv_src_metadata;   /* [rows, 2] (token, slot) per row, (-1,-1) padding */
  const uint8_t *is_token_in_rank;    /* [T, R] 0/1 */
  const int32_t *totals;              /* [2] device num_recv_tokens, num_expanded_tokens */
  const uint32_t *error_word;         /* [1] EP_ERRBIT_* bits */
  int64_t meta_rows;                  /* rows of recv_src_metadata */
  int64_t expert_capacity;            /* fixed_capacity: rows per expert, else 0 */
  int64_t sf_expert_stride;           /* fixed_capacity: the scales of row e * capacity + i
                                         are recv_sf[e * sf_expert_stride + i *
                                         sf_token_stride + j * sf_hidden_stride]; else 0 */
  int32_t layout_kernels;             /* kernels this layout launched: 1 (rank layouts of at
                                         most 15 chunks of up to 256 tokens whose counts fit
                                         96 KB of shared memory, if the device can place the
                                         cluster: one thread-block cluster of a CTA per chunk
                                         plus one) or 2 (count + assign) */
  int32_t reserved1;
} ep_layout_info;

typedef struct ep_handle ep_handle;

/*
 * ep_layout -- routing layout (DeepEP README interface example,
 * get_dispatch_layout; §7.2 layout metadata; §7.4 expanded layout).
 *
 * topk_idx: device [T, K], int64 or int32 per cfg->topk_idx_is_int64; -1 is
 *   an empty slot.  It is read only during this call (the handle keeps an
 *   int32 copy), so the caller may reuse it once the stream passes the call.
 * Rows: expert e's segment starts at psum_expert[e] (expanded) or rank r's at
 *   psum_rank[r] (rank layout); inside a segment rows follow ascending
 *   (token, slot).  In the rank layout all slots of a token on one rank share
 *   one row.
 * do_cpu_sync = 1: blocks the host until the counts are visible (polling
 *   mapped host memory, deadline cfg->cpu_sync_timeout_ms), then reports the
 *   exact totals; not allowed while `stream` is being captured.  Returns
 *   EP_ERR_TIMEOUT at the deadline (no handle), EP_ERR_BAD_TOPK_IDX if a
 *   value was outside [-1, E) -- the handle is still created, with those
 *   slots empty, and must be freed.
 * do_cpu_sync = 0: no host synchronisation (graph-capturable); rows_alloc is
 *   the upper bound and the device totals / error word tell the real sizes.
 * On EP_OK (or EP_ERR_BAD_TOPK_IDX) *out_handle owns device memory allocated
 *   stream-ordered on `stream`; release it with ep_handle_free.
 */
EP_API ep_status ep_layout(const ep_config *cfg, const void *topk_idx, ep_stream_t stream,
                    ep_handle **out_handle, ep_layout_info *info);

/*
 * ep_dispatch -- copy epilogue (§7.3 launch_dispatch_copy_epilogue, §7.4).
 *
 * x: device BF16 [T, H], 16-byte aligned.
 * topk_weights: device fp32 [T, K] or NULL (then recv_topk_weights must be NULL,
 *   unless T = 0).
 * recv_x: [rows_alloc, H] BF16, or e4m3 bytes when cfg->use_fp8; 16-byte aligned.
 * recv_sf: FP8 only, fp32 [sf_numel]; row-major [rows_alloc, H/128] or, with
 *   use_tma_aligned_col_major_sf, column-major with hidden stride
 *   align(rows_alloc, 4).  scale = amax / 448 per 1x128 block (fp32 IEEE
 *   division), payload = e4m3(x / scale) round-to-nearest-even, saturating;
 *   an all-zero block has scale 0 and zero bytes.  Non-finite inputs: a
 *   block holding a NaN gets a NaN scale and 0x7F (the e4m3 NaN code) in
 *   every byte; a block whose amax is infinite gets scale +inf, signed
 *   zeros for its finite elements and 0x7F for its infinite ones.
 * recv_topk_weights: NULL, or fp32 [rows_alloc] (expanded) / [rows_alloc, K]
 *   (rank layout: the token's weights on that rank, 0 elsewhere).
 * recv_topk_idx: NULL, or (rank layout only) int32 [rows_alloc, K]: the local
 *   expert index (expert - r * L) of the token's slots on that rank, -1 elsewhere.
 * Padding rows (expanded) get weight 0; with do_zero_padding also zero
 *   payload and zero scales.  Rows past the real total are not written.
 * Must be ordered after ep_layout of the same handle (same stream, or the
 *   caller's own event).  May be called again with new x (cached dispatch);
 *   dispatches on one handle (this call, ep_dispatch_fp8, ep_combine_backward)
 *   must not overlap on the GPU: they share the handle's scheduling and
 *   scale-gather counters.  A dispatch whose bounded device wait gave up
 *   (EP_ERRBIT_TIMEOUT in the handle's error word) may leave those counters
 *   set: free such a handle and lay out again instead of dispatching on it.
 */
EP_API ep_status ep_dispatch(ep_handle *h, const void *x, const float *topk_weights,
                      void *recv_x, float *recv_sf, float *recv_topk_weights,
                      int32_t *recv_topk_idx, ep_stream_t stream);

/*
 * ep_plan_layout -- the sizes ep_layout would report for a configuration
 * with do_cpu_sync = 0 (they do not depend on the routing): rows_alloc (the
 * upper bound), sf_numel, sf_token_stride, sf_hidden_stride, meta_rows,
 * expert_capacity and sf_expert_stride.  Every pointer of *info is set to
 * NULL and the counts to -1.  No GPU work.  EP_ERR_INVALID_ARG for
 * do_cpu_sync = 1 or a NULL info.
 */
EP_API ep_status ep_plan_layout(const ep_config *cfg, ep_layout_info *info);

/*
 * ep_layout_dispatch -- ep_layout followed by ep_dispatch, in one call that
 * takes the routing and the activations together, as the DeepEP README's
 * low_latency_dispatch does ("Interfaces and examples").  Results are those
 * of ep_layout and then ep_dispatch with the same arguments: the handle,
 * *info (num_recv_tokens and num_expanded_tokens are -1) and the receive
 * buffers.
 *
 * Requires do_cpu_sync = 0: the caller sizes the receive buffers from
 * ep_plan_layout before the call.  topk_idx and x are read only during the
 * call.  x, an input of the call, is complete before the layout starts, so
 * the dispatch (launched right behind the layout kernels) loads and
 * quantises the first source rows of every CTA while the layout runs; a
 * separate ep_dispatch cannot, since the caller may write x in between.
 * Errors as for ep_layout and ep_dispatch; on any error nothing is allocated
 * and *out_handle is NULL.
 */
EP_API ep_status ep_layout_dispatch(const ep_config *cfg, const void *topk_idx, const void *x,
                                    const float *topk_weights, void *recv_x, float *recv_sf,
                                    float *recv_topk_weights, int32_t *recv_topk_idx,
                                    ep_stream_t stream, ep_handle **out_handle,
                                    ep_layout_info *info);

/*
 * ep_dispatch_fp8 -- copy epilogue for an input that is already FP8 (§7.1:
 * x may be an FP8 data + scale-factor tuple; §7.3 scale-factor layouts).
 *
 * Requires cfg->use_fp8 = 1 (the receive buffers are FP8); nothing is
 * quantised.  x_fp8: device e4m3 bytes [T, H], 16-byte aligned.  x_sf: device
 * fp32, the scale of token t and 128-element block j at
 *   x_sf[t * x_sf_token_stride + j * x_sf_hidden_stride]   (strides >= 0),
 * e.g. row-major [T, H/128] (H/128, 1) or column-major TMA-aligned
 * (1, align(T, 4)).  Every destination row gets its token's bytes unchanged
 * and its token's scales in the handle's layout (row-major, or column-major
 * with use_tma_aligned_col_major_sf); padding rows, weights and local expert
 * ids exactly as ep_dispatch.  The other arguments are those of ep_dispatch,
 * and like it, it must not overlap another dispatch of the same handle.
 */
EP_API ep_status ep_dispatch_fp8(ep_handle *h, const void *x_fp8, const float *x_sf,
                                 int64_t x_sf_token_stride, int64_t x_sf_hidden_stride,
                                 const float *topk_weights, void *recv_x, float *recv_sf,
                                 float *recv_topk_weights, int32_t *recv_topk_idx,
                                 ep_stream_t stream);

/*
 * ep_combine -- reduce expert outputs back to token order (§8.1 combine
 * along the handle; vLLM PR #52781 review: combine requires BF16 input and
 * may be called with topk_weights = None).
 *
 * y: device BF16 [rows_alloc, H] in the dispatch layout, 16-byte aligned.
 * out: device BF16 [T, H], 16-byte aligned; must not overlap y.
 * For each token: acc = 0 (fp32); for k = 0..K-1 over valid slots:
 *   v = y[dst[t,k]] (+ expert_bias[topk_idx[t,k]] if given);
 *   acc += topk_weights[t,k] * v (product and sum each rounded to fp32).
 *   With topk_weights == NULL the weight is 1 and a row already used by an
 *   earlier slot of the same token is skipped (rank layout shares rows).
 *   Then acc += bias_0[t], acc += bias_1[t]; out[t] = bf16_rne(acc).
 * bias_0, bias_1: NULL or device BF16 [T, H]; expert_bias: NULL or BF16 [E, H].
 */
EP_API ep_status ep_combine(const ep_handle *h, const void *y, const float *topk_weights,
                     const void *bias_0, const void *bias_1, const void *expert_bias,
                     void *out, ep_stream_t stream);

/* ---- backward pair (DeepEP README, "Interfaces and examples":
 *      dispatch_backward, combine_backward) ------------------------------- */

/*
 * ep_dispatch_backward -- the backward of ep_dispatch is a combine along the
 * same handle that also reduces the received weight gradients.
 *
 * grad_recv_x: device BF16 [rows_alloc, H] in the dispatch layout, 16-byte
 *   aligned.  grad_x (out): device BF16 [T, H], 16-byte aligned, no overlap.
 *   grad_x[t] = bf16_rne(fp32 sum of grad_recv_x over the token's distinct
 *   rows in slot order) -- ep_combine with topk_weights == NULL and no bias.
 * grad_recv_topk_weights: NULL, or device fp32 [rows_alloc] (expanded) /
 *   [rows_alloc, K] (rank layout), shaped like ep_dispatch's recv_topk_weights.
 * grad_topk_weights (out): NULL (then grad_recv_topk_weights must be NULL
 *   too), or device fp32 [T, K]; grad_recv_topk_weights may then be NULL only
 *   if rows_alloc == 0 (every result is 0).  Per token, the fp32 sum of its distinct rows'
 *   entries in slot order: expanded, slot k reads its own row (0 without
 *   one); rank layout, column c sums column c of the token's rows (every
 *   column, 0 for a token without rows).
 * Ordered after ep_layout of the handle; returns EP_ERR_INVALID_ARG for a
 * missing or misaligned pointer before touching the GPU.
 */
EP_API ep_status ep_dispatch_backward(const ep_handle *h, const void *grad_recv_x,
                                      const float *grad_recv_topk_weights, void *grad_x,
                                      float *grad_topk_weights, ep_stream_t stream);

/*
 * ep_combine_backward -- the backward of an unweighted ep_combine is a
 * dispatch of the gradient along the same handle.
 *
 * grad_combined_x: device BF16 [T, H], 16-byte aligned.
 * grad_recv_x (out): device BF16 [rows_alloc, H], 16-byte aligned: each
 *   destination row gets its token's gradient row, bit for bit.  Always a
 *   BF16 copy, also when cfg->use_fp8 quantises the forward dispatch.
 *   Padding rows (expanded) are zeroed when cfg->do_zero_padding, else left
 *   as they are; rows past the real total are not written.  Like ep_dispatch,
 *   it must not overlap another dispatch of the same handle.
 */
EP_API ep_status ep_combine_backward(ep_handle *h, const void *grad_combined_x,
                                     void *grad_recv_x, ep_stream_t stream);

/*
 * ep_handle_free -- releases the handle's device memory, stream-ordered on
 * the stream given to ep_layout (work enqueued there before this call may
 * still use it).  NULL is ignored.  Work on other streams that uses the
 * handle must be ordered before this call by the caller.
 */
EP_API void ep_handle_free(ep_handle *h);

/* ---- layout without any allocation ------------------------------------- */

/*
 * Caller-owned device buffers that ep_layout_noalloc fills.  Shapes as in
 * ep_layout_info; `rows` = ep_upper_bound_rows(cfg).
 */
typedef struct ep_layout_buffers {
  int32_t *topk_idx32;           /* [T, K] int32 copy, invalid values -> -1 */
  int32_t *cnt_expert;           /* [E] */
  int32_t *cnt_expert_aligned;   /* [E] */
  int32_t *psum_expert;          /* [E+1] */
  int32_t *psum_padding;         /* [E+1] exclusive prefix of the padding rows per expert */
  int32_t *cnt_rank;             /* [R] */
  int32_t *psum_rank;            /* [R+1] */
  int32_t *psum_rank_src;        /* [R, R+1] */
  int32_t *dst_buffer_slot_idx;  /* [T, K] */
  int32_t *recv_src_metadata;    /* [rows, 2] */
  uint8_t *is_token_in_rank;     /* [T, R] */
  int32_t *status;               /* [4]: EP_ERRBIT_* bits, unused, num_recv_tokens,
                                    num_expanded_tokens */
} ep_layout_buffers;

/* Largest scratch ep_layout_noalloc can use: 2 MiB of int32 words. */
#define EP_NOALLOC_SCRATCH_WORDS (512 * 1024)

/*
 * ep_layout_noalloc -- the routing layout of ep_layout, for callers that may
 * not allocate memory while they run: code inside a CUDA-graph capture that
 * must not add allocation nodes, allocator-free inference runtimes that own
 * every byte of device memory up front, or hosts whose allocator is not
 * thread-safe at that point.  The pages have no counterpart of this entry
 * point: it is an allocation-free variant of the layout kernels only.
 *
 * It computes exactly what ep_layout computes with do_cpu_sync = 0 and
 * writes it to the caller's buffers `out` (all device memory, all required);
 * no handle is created and nothing is allocated (no cudaMalloc, cudaFree or
 * pool call).  The per-chunk histograms the layout needs live in one static
 * device array of EP_NOALLOC_SCRATCH_WORDS int32 words that every GPU loading
 * this library holds until the process exits.  A problem needing more,
 * chunks * (E + R + 1) words with chunks = ceil(T / M) * ceil(min(M, T) /
 * 256), is rejected with EP_ERR_UNSUPPORTED before any GPU work;
 * cfg->do_cpu_sync = 1 is rejected with EP_ERR_INVALID_ARG.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  Calls
 * made outside a capture look the address up again (so a context re-created
 * after cudaDeviceReset is served); calls inside a capture reuse the address
 * of the last call outside one.  Every call uses the same array and leaves its last contents
 * there; every word a call reads is written by the same call first, so
 * nothing has to be cleared between calls.  Calls that overlap on the GPU
 * (concurrent streams, or several host threads) race on the array: order
 * them on one stream or with events.
 */
EP_API ep_status ep_layout_noalloc(const ep_config *cfg, const void *topk_idx,
                                   const ep_layout_buffers *out, ep_stream_t stream);

/* ---- diagnostics -------------------------------------------------------- */

/*
 * ep_selftest_bounded_wait -- exercises the bounded device-side wait that
 * every dispatch / combine pipeline stage uses (mbarrier try_wait with a
 * suspend-time hint, a fixed number of attempts).  One CTA waits on an
 * mbarrier for at most about `wait_us` microseconds; with `signal` = 0 nothing
 * ever arrives, so the wait runs out and the kernel reports EP_ERRBIT_TIMEOUT
 * instead of hanging; with `signal` = 1 the barrier is completed first and
 * no bit is set.  The bits are written to *error_bits (host pointer) after
 * the stream has been synchronised.  The CUDA context stays usable either
 * way.  Not part of the method; used by the failure-detection tests.
 */
EP_API ep_status ep_selftest_bounded_wait(int32_t wait_us, int32_t signal,
                                          uint32_t *error_bits, ep_stream_t stream);

/* ---- host-only helpers (no GPU needed) ---------------------------------- */

/* Human-readable name of a status code (static string). */
EP_API const char *ep_status_string(ep_status s);

/* ABI version of this header (bumped on any layout change of the structs). */
EP_API int32_t ep_abi_version(void);

/* Checks cfg against the rules above without touching the GPU. */
EP_API ep_status ep_validate_config(const ep_config *cfg);

/*
 * Upper-bound rows for cfg (§7.2 worst case, ranks packed back to back):
 * min(R * per_rank, global) with per_rank = M * R (rank layout) or
 * align(R * M * min(K, L) + (A - 1) * L, A) (expanded) and global =
 * T * min(K, R) or align(T * K + E * (A - 1), A).  Host only.
 */
EP_API ep_status ep_upper_bound_rows(const ep_config *cfg, int64_t *rows);

/*
 * The host wait of do_cpu_sync in its simplest form: polls *flag until it
 * equals `expected` or `timeout_ms` passes (EP_ERR_TIMEOUT).  (ep_layout polls
 * three tagged words with the same loop and deadline.)  Exposed so the
 * deadline logic can be tested on the host with a flag that nothing sets.
 */
EP_API ep_status ep_host_wait_flag(const volatile int32_t *flag, int32_t expected,
                            int32_t timeout_ms);

#define EP_ABI_VERSION 3

#ifdef __cplusplus
}
#endif

#endif /* EP_H_ */
