/*
 * ep.h -- C ABI of the GB300 MoE expert-parallel dispatch / combine library.
 *
 * What it computes (the pages describe DeepEP's operations in prose only):
 *  - "DeepEP 要約" (stakiran.github.io), section 3 "使うときの流れ":
 *    training / prefill forward is get_dispatch_layout -> dispatch(x,
 *    topk_idx, topk_weights, ...) -> expert computation -> combine(y, handle);
 *    the backward of dispatch is combine and the backward of combine is
 *    dispatch, both reusing the handle; decode uses low_latency_dispatch and
 *    low_latency_combine, which are CUDA-graph compatible.
 *  - "DeepSeek công bố thư viện mã nguồn mở DeepEP cho huấn luyện và suy luận
 *    MoE" (vi.news.hada.io), section "Mẫu sử dụng cho huấn luyện, prefill và
 *    decoding": dispatch routes tokens to the experts of every rank (BF16 or
 *    FP8), the handle carries the routing metadata that combine needs and the
 *    per-expert receive counts for the grouped GEMM; combine reduces the
 *    expert outputs back to the originating rank; a cached handle avoids
 *    recomputing the layout and the CPU synchronisation.
 *  - "Как DeepSeek разогнали обмен данными в своих нейросетях" (devtrends.ru),
 *    section "Как это выглядит в коде": the dispatch and low_latency_dispatch
 *    call shapes; section "Что умеет DeepEP": the number of SMs the kernels
 *    occupy is under the caller's control.
 *  - "DeepSeek выпустила DeepEP V2.5" (aikraft.ru), section "Технические
 *    детали и требования": FP8 dispatch, BF16 combine.
 *
 * One GPU.  The R expert-parallel ranks are logical partitions of one HBM:
 * source rank s owns tokens [s*T/R, (s+1)*T/R); rank r owns experts
 * [r*E_l, (r+1)*E_l) with E_l = E/R.  The all-to-all is a device-wide
 * permutation; there is no communication library underneath.
 *
 * Conventions for every call
 *  - Pointers marked "dev" are device pointers on the device that was
 *    current when the handle was created; "host" pointers are ordinary host
 *    memory.  The caller owns every pointer it passes; the library keeps none
 *    of them after the call returns.
 *  - Tensors are row-major and contiguous.  bf16 is IEEE bfloat16 (2 bytes),
 *    e4m3 is OCP FP8 E4M3 ("FN", max 448, no infinities), weights and scales
 *    are IEEE binary32.  hidden (H) is a positive multiple of 128; FP8 scales
 *    are one fp32 per 128 consecutive channels of a token (G = H/128 per row,
 *    scale = amax/448, dequantised value = e4m3 * scale).
 *  - Every device buffer must be 16-byte aligned.
 *  - All work is enqueued on the caller's stream and is asynchronous unless a
 *    call says it synchronises.  Calls on one handle must not overlap in
 *    time (one stream per handle, or caller-side ordering).
 *  - Argument errors return a status before anything is enqueued.
 *    Conditions found on the device (an expert id outside [-1, E), a receive
 *    buffer that is too small, a bounded wait that gave up) are latched in the
 *    handle: the offending rows are skipped -- never written out of bounds --
 *    and the first such status is returned (and cleared) by
 *    ep_get_device_status() and also reported by ep_get_num_recv().
 *  - No call allocates device memory after ep_handle_create().
 */
#ifndef GB300_EP_H_
#define GB300_EP_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* ep_stream_t;

typedef struct ep_handle* ep_handle_t;

typedef enum {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1, /* a bad size, pointer, alignment or dtype         */
  EP_ERR_CUDA = 2,        /* a CUDA runtime call failed                       */
  EP_ERR_CAPACITY = 3,    /* a receive buffer had fewer rows than needed     */
  EP_ERR_BAD_EXPERT = 4,  /* topk_idx held an id outside [-1, E)             */
  EP_ERR_TIMEOUT = 5,     /* a bounded cross-block wait gave up              */
  EP_ERR_STATE = 6        /* e.g. dispatch before any layout on this handle */
} ep_status_t;

typedef enum { EP_BF16 = 0, EP_FP8_E4M3 = 1 } ep_dtype_t;

/* Receive layouts: rank-major (ep_dispatch: one row per (token,
 * destination rank), ranks' regions packed), low latency ([E][M][H] per
 * expert), expert-major (ep_em_*: one row per (token, expert) entry, expert
 * groups packed and aligned). */
typedef enum { EP_LAYOUT_RANK_MAJOR = 0, EP_LAYOUT_LOW_LATENCY = 1, EP_LAYOUT_EXPERT_MAJOR = 2 } ep_layout_t;

/* Create a handle for R ranks, E experts (E % R == 0), top-k = num_topk
 * (1..32), hidden size H (multiple of 128) and at most max_tokens_per_rank
 * tokens per source rank (so T <= R * max_tokens_per_rank).  Allocates, once,
 * the device metadata arena: routing maps, counts, the cross-block scan
 * state and the error latch.  Limits: R <= 1024, E <= 4096, and the
 * per-block routing tables must fit in shared memory (EP_ERR_INVALID_ARG).
 * Cite: Buffer(group, ...) / ElasticBuffer creation ("DeepEP 要約" section 3;
 * vi.news.hada.io "Giao diện xoay quanh ElasticBuffer"). */
ep_status_t ep_handle_create(int num_ranks, int num_experts, int num_topk, int hidden,
                             int max_tokens_per_rank, ep_handle_t* out);

/* Width of the top-k expert ids that the calls taking `topk_idx` read
 * through this handle: 64 (int64, the default) or 32 (int32).  The default
 * comes from the environment variable EP_NUM_TOPK_IDX_BITS ("64" or "32";
 * any other value makes ep_handle_create fail with EP_ERR_INVALID_ARG) at
 * creation; ep_handle_set_topk_idx_bits changes it for later calls.  The
 * pages list EP_NUM_TOPK_IDX_BITS as the variable that overrides the number
 * of bits of the top-k index encoding (vi.news.hada.io, "Biến môi trường và
 * giá trị cố định khi build").  int32 ids halve the bytes the routing reads.
 * A `topk_idx` pointer must be 8-byte aligned for int64 ids, 4-byte for
 * int32.  ep_get_dispatch_layout_noalloc always reads int64. */
ep_status_t ep_handle_set_topk_idx_bits(ep_handle_t h, int bits);
int ep_handle_topk_idx_bits(ep_handle_t h); /* 64 or 32; 0 for NULL */

/* Free the handle's device and host memory.  The caller must make sure no
 * enqueued work that uses the handle is still pending.  NULL is a no-op. */
ep_status_t ep_handle_destroy(ep_handle_t h);

/* get_dispatch_layout ("DeepEP 要約" section 3, training forward;
 * devtrends.ru "Как это выглядит в коде", num_tokens_per_rank).
 * In:  topk_idx   dev [T][k] ids, int64 or int32 (ep_handle_set_topk_idx_bits);
 *                 -1 marks a masked entry.
 *      T          number of tokens, a multiple of R, <= R*max_tokens_per_rank.
 * Out (each may be NULL):
 *      num_tokens_per_rank    dev int32 [R src][R dst]: tokens source rank s
 *                             sends to rank r (a token counts once per rank);
 *      num_tokens_per_expert  dev int32 [R src][E]: (token, k) entries of
 *                             source rank s routed to expert e;
 *      is_token_in_rank       dev uint8 (bool) [T][R].
 * Also stores in the handle, for ep_dispatch / ep_combine: each token's
 * destination ranks and its row inside every destination rank's region
 * (rows ordered by source rank, then token), the regions' offsets inside the
 * packed receive buffer and the per-rank / per-expert receive counts. */
ep_status_t ep_get_dispatch_layout(ep_handle_t h, const void* topk_idx, int num_tokens,
                                   int* num_tokens_per_rank, int* num_tokens_per_expert,
                                   uint8_t* is_token_in_rank, ep_stream_t stream);

/* Copy the receive counts of the last layout to host memory; synchronises
 * `stream`.  Out (each may be NULL): num_recv_tokens_per_rank host int32 [R],
 * num_recv_tokens_per_expert host int32 [E] (handle.num_recv_tokens_per_expert_list
 * for the grouped GEMM; vi.news.hada.io "Mẫu sử dụng ..."), rank_offset host
 * int32 [R+1] (row where rank r's region starts in the packed receive buffer;
 * rank_offset[R] = total rows P).  Returns the latched device status, if any
 * (without clearing it). */
ep_status_t ep_get_num_recv(ep_handle_t h, int* num_recv_tokens_per_rank,
                            int* num_recv_tokens_per_expert, int* rank_offset,
                            ep_stream_t stream);

/* dispatch, normal mode ("DeepEP 要約" section 3; devtrends.ru "Как это
 * выглядит в коде").  Uses the handle's last layout (so it also serves the
 * backward of combine and a cached handle).
 * In:  x            dev bf16 [T][H].
 *      topk_weights dev fp32 [T][k] or NULL.
 *      dtype        EP_BF16: rows are copied; EP_FP8_E4M3: each row is
 *                   quantised once (per 128 channels: a = max(amax, 1e-4),
 *                   scale = a/448, q = e4m3_rn_satfinite(x * (448/a))).
 * Out: recv_x       dev [cap][H], bf16 or e4m3 bytes; rank r's rows start at
 *                   rank_offset[r]; only the first P rows are written.
 *      recv_scales  dev fp32 [cap][H/128] (FP8 only, else ignored).
 *      recv_capacity_rows  cap; rows beyond it are skipped and latch
 *                   EP_ERR_CAPACITY.
 *      recv_src_idx       dev int32 [cap] or NULL: source token of each row.
 *      recv_topk_idx      dev int32 [cap][k] or NULL: the token's expert id
 *                         made local to the receiving rank, -1 if the expert
 *                         lives elsewhere or is masked.
 *      recv_topk_weights  dev fp32 [cap][k] or NULL (needs topk_weights):
 *                         the weight where recv_topk_idx >= 0, else 0.
 *      num_sms      SMs to occupy (0 = all). */
ep_status_t ep_dispatch(ep_handle_t h, const void* x, const float* topk_weights, ep_dtype_t dtype,
                        void* recv_x, float* recv_scales, int64_t recv_capacity_rows,
                        int* recv_src_idx, int* recv_topk_idx, float* recv_topk_weights,
                        int num_sms, ep_stream_t stream);

/* get_dispatch_layout and dispatch in one call ("DeepEP 要約" section 3,
 * training / prefill forward).  Same inputs and outputs as
 * ep_get_dispatch_layout(topk_idx, T, NULL, NULL, NULL) followed by
 * ep_dispatch(...), and the same handle state afterwards (so ep_combine,
 * ep_get_num_recv and a cached-handle ep_dispatch work as usual); the
 * per-source-rank counts and is_token_in_rank are not produced -- call
 * ep_get_dispatch_layout when they are needed.
 * Because the receive counts are only known on the device, recv_x must have
 * room for the rows this routing produces (at most T * min(k, R)); rows past
 * recv_capacity_rows latch EP_ERR_CAPACITY as in ep_dispatch.
 * For R <= 64 and up to 4096 (token, k) entries per SM this is one
 * cooperative launch: one block per SM ranks its own run of tokens while its
 * rows are already streaming into shared memory, the blocks exchange counts
 * through one grid barrier, then the rows are written.  Otherwise it runs the
 * layout kernel and the dispatch kernel. */
ep_status_t ep_layout_and_dispatch(ep_handle_t h, const void* topk_idx, int num_tokens, const void* x,
                                   const float* topk_weights, ep_dtype_t dtype, void* recv_x,
                                   float* recv_scales, int64_t recv_capacity_rows, int* recv_src_idx,
                                   int* recv_topk_idx, float* recv_topk_weights, int num_sms,
                                   ep_stream_t stream);

/* combine, normal mode ("DeepEP 要約" section 3; vi.news.hada.io: combine
 * reduces the expert outputs back to the originating rank).
 * In:  y      dev bf16 [y_rows][H], laid out like dispatch's recv_x.
 * Out: out    dev bf16 [T][H]: for each token, the fp32 sum of its rows over
 *             its destination ranks in ascending rank order (from +0.0),
 *             rounded to bf16 (nearest-even); 0 for a token sent nowhere.
 * A source row at or past y_rows is skipped (counted as absent) and latches
 * EP_ERR_CAPACITY; nothing is read out of bounds. */
ep_status_t ep_combine(ep_handle_t h, const void* y, int64_t y_rows, void* out, int num_sms,
                       ep_stream_t stream);

/* combine, normal mode, general form.  ep_combine(h, y, rows, out, ...) is
 * ep_combine_ex(h, EP_BF16, y, NULL, rows, NULL, out, NULL, ...).
 * In:  y_dtype  EP_BF16: y is dev bf16 [y_rows][H];
 *               EP_FP8_E4M3: y is dev e4m3 bytes [y_rows][H] with y_scales
 *               dev fp32 [y_rows][H/128]; each value enters the sum as
 *               e4m3 * scale (one fp32 multiply, nearest-even) -- a
 *               low-precision combine input, as the pages' FP8 support
 *               ("DeepSeek công bố thư viện mã nguồn mở DeepEP ...",
 *               vi.news.hada.io: FP8 and other low precisions) extended to
 *               the reduction side.
 *      recv_topk_weights  dev fp32 [y_rows][k] or NULL, laid out like
 *               dispatch's recv_topk_weights.
 * Out: out      dev bf16 [T][H], the sum in ascending rank order as
 *               ep_combine.
 *      combined_topk_weights  dev fp32 [T][k], required exactly when
 *               recv_topk_weights is given: column j of token t = the fp32
 *               sum over t's rows, ascending rank, from +0.0, of
 *               recv_topk_weights[row][j].  On dispatch's own output this
 *               gives back topk_weights (0 where masked); on gradients it is
 *               the backward of the weights ("DeepEP 要約" section 3: the
 *               backward of dispatch is combine). */
ep_status_t ep_combine_ex(ep_handle_t h, ep_dtype_t y_dtype, const void* y, const float* y_scales,
                          int64_t y_rows, const float* recv_topk_weights, void* out,
                          float* combined_topk_weights, int num_sms, ep_stream_t stream);

/* low_latency_dispatch (devtrends.ru "Как это выглядит в коде";
 * "DeepEP 要約" section 3, decode).  Computes its own routing (no separate
 * layout call, no host synchronisation, capturable in a CUDA graph) and
 * stores it in the handle for ep_low_latency_combine.
 * In:  x         dev bf16 [T][H];  topk_idx dev [T][k] (int64 or int32, as the
 *                handle's setting);  T as above.
 * Out: recv_x       dev [E][M][H] (bf16 or e4m3), M = R * max_tokens_per_rank;
 *                   expert e = (rank e / E_l, local expert e % E_l); the
 *                   entries routed to e fill rows 0..count-1 in (source rank,
 *                   token, k-index) order.
 *      recv_scales  dev fp32 [E][M][H/128] (FP8 only).
 *      recv_src_info dev int32 [E][M] or NULL: source token of each row.
 *      recv_count   dev int32 [E] or NULL: rows filled per expert.
 * Rows past M (only possible with duplicated ids in one token) are skipped
 * and latch EP_ERR_CAPACITY.
 * Usually one cooperative launch on at most num_sms SMs (0 = all): each
 * block ranks its own run of tokens, the blocks exchange counts through one
 * grid barrier, then the rows move.  With more than 4096 (token, k) entries
 * per SM it is a routing kernel followed by the row scatter. */
ep_status_t ep_low_latency_dispatch(ep_handle_t h, const void* x, const void* topk_idx,
                                    int num_tokens, ep_dtype_t dtype, void* recv_x,
                                    float* recv_scales, int* recv_src_info, int* recv_count,
                                    int num_sms, ep_stream_t stream);

/* low_latency_combine ("DeepEP 要約" section 3, decode).  Uses the routing of
 * the handle's last ep_low_latency_dispatch.
 * In:  y            dev bf16 [E][M][H], laid out like that dispatch's recv_x.
 *      topk_weights dev fp32 [T][k].
 * Out: out          dev bf16 [T][H]: acc = fmaf(w, y, acc) over the token's
 *                   unmasked entries in ascending expert id (k-index breaks
 *                   ties), from +0.0, rounded to bf16 (nearest-even). */
ep_status_t ep_low_latency_combine(ep_handle_t h, const void* y, const float* topk_weights,
                                   void* out, int num_sms, ep_stream_t stream);

/* ---------------------------------------------------------------------
 * Expert-major ("GEMM") receive layout -- the "new GEMM layout" of the V2
 * release ("DeepSeek công bố thư viện mã nguồn mở DeepEP ..." (vi.news.hada.io),
 * "Những thay đổi chính của bản phát hành V2"), read as: the rows a grouped
 * GEMM consumes directly, one row per unmasked (token, k) entry, grouped by
 * expert in ascending expert id (so rank r's experts form one contiguous
 * region), the entries of one expert in (source rank, token, k-index) order,
 * and each expert's group starting at a multiple of `expert_alignment` rows
 * (the GEMM's M tile).  Padding rows carry source -1 and weight 0; their
 * payload and scales are not written.  FP8 scales are stored group-major,
 * scales[g * scales_ld + row], so the scales of one 128-channel group of
 * consecutive rows are contiguous (scales_ld >= capacity rows, a multiple of
 * 4 so every group's column starts 16-byte aligned).
 * --------------------------------------------------------------------- */

/* Expert-major layout and dispatch in one call.
 * In:  topk_idx [T][k] (width per ep_handle_set_topk_idx_bits), x bf16 [T][H],
 *      topk_weights fp32 [T][k] or NULL, dtype, expert_alignment (1..65536;
 *      T*k + E*(alignment-1) must fit in int32).
 * Out: recv_x [cap][H] (e4m3 bytes or bf16); recv_scales fp32
 *      [H/128][scales_ld] (FP8 only); recv_src_idx int32 [cap] or NULL (the
 *      row's source token, -1 on padding); recv_weights fp32 [cap] or NULL
 *      (needs topk_weights; the entry's weight, 0 on padding).
 *      Rows at or past recv_capacity_rows are skipped and latch
 *      EP_ERR_CAPACITY; at most T*k + E*(alignment-1) rows are needed.
 * The handle keeps the layout for ep_em_get_layout, ep_em_dispatch and
 * ep_em_combine.  Usually one cooperative launch (as ep_layout_and_dispatch);
 * with more than 4096 (token, k) entries per SM a routing kernel, a one-block
 * offsets kernel and the row scatter.  H must leave room for two staged rows
 * in shared memory (H <= ~50k), else EP_ERR_INVALID_ARG. */
ep_status_t ep_em_layout_and_dispatch(ep_handle_t h, const void* topk_idx, int num_tokens, const void* x,
                                      const float* topk_weights, ep_dtype_t dtype, int expert_alignment,
                                      void* recv_x, float* recv_scales, int64_t scales_ld,
                                      int64_t recv_capacity_rows, int* recv_src_idx, float* recv_weights,
                                      int num_sms, ep_stream_t stream);

/* Dispatch another tensor (e.g. gradients, "DeepEP 要約" section 3: the
 * backward of combine is dispatch) through the handle's last expert-major
 * layout; arguments as ep_em_layout_and_dispatch. */
ep_status_t ep_em_dispatch(ep_handle_t h, const void* x, const float* topk_weights, ep_dtype_t dtype,
                           void* recv_x, float* recv_scales, int64_t scales_ld, int64_t recv_capacity_rows,
                           int* recv_src_idx, float* recv_weights, int num_sms, ep_stream_t stream);

/* Copy the last expert-major layout to host memory; synchronises `stream`.
 * Out (each may be NULL): num_recv_tokens_per_expert host int32 [E] (rows
 * per expert, without padding: the grouped GEMM's per-expert M),
 * expert_offset host int32 [E+1] (first row of each group; [E] = rows
 * used).  Returns the latched device status, if any (without clearing it). */
ep_status_t ep_em_get_layout(ep_handle_t h, int* num_recv_tokens_per_expert, int* expert_offset,
                             ep_stream_t stream);

/* Expert-major combine: out bf16 [T][H] = for each token, the fp32 sum of
 * its rows of y (bf16 [y_rows][H], laid out like ep_em_* recv_x) over its
 * unmasked entries in ascending expert id (k-index breaks ties), from +0.0,
 * rounded to bf16 (nearest-even); unweighted, as ep_combine (the entry's
 * weight is the expert side's to apply, e.g. in the GEMM epilogue, from
 * recv_weights).  Rows at or past y_rows are skipped and latch
 * EP_ERR_CAPACITY. */
ep_status_t ep_em_combine(ep_handle_t h, const void* y, int64_t y_rows, void* out, int num_sms,
                          ep_stream_t stream);

/* Receive-buffer sizes for a configuration, before any routing is known
 * (the pages' get_buffer_size_hint: the size needed, to allocate once or to
 * check that an existing buffer can be reused; vi.news.hada.io, "Giao diện
 * xoay quanh ElasticBuffer").  Needs no GPU and no handle.
 * Out: *rows   the most receive rows any routing can need: T*min(k,R)
 *              (rank-major), E*M (low latency, M = R*max_tokens_per_rank),
 *              T*k + E*(alignment-1) (expert-major), T = R*max_tokens_per_rank;
 *      *bytes  the bytes of all receive-side buffers at that row count:
 *              payload (+ fp32 scales for FP8), plus per row the source
 *              index and (rank-major) k local ids and k weights, (low
 *              latency) plus E counts, (expert-major) one weight, with
 *              scales_ld = rows rounded up to 4. */
ep_status_t ep_get_buffer_size_hint(int num_ranks, int num_experts, int num_topk, int hidden,
                                    int max_tokens_per_rank, ep_dtype_t dtype, ep_layout_t layout,
                                    int expert_alignment, int64_t* rows, int64_t* bytes);

/* ep_get_dispatch_layout_noalloc -- the same layout computation as
 * ep_get_dispatch_layout, for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists for this library's
 * users.  Some callers cannot call cudaMalloc at all: serving runtimes that
 * hand all device memory to their own allocator up front and forbid further
 * allocations, and plugin hosts that call in per request with no place to
 * keep a handle (whose creation allocates).  This entry point needs no handle and allocates
 * nothing: every result goes to caller buffers, and the cross-block scan state
 * lives in a fixed 1 MiB array in the library's device memory, which every GPU
 * that loads the library holds until the process exits.
 * Limits: R <= 1024, E <= 4096, E % R == 0, 1 <= k <= 32, T % R == 0, and
 * R * ceil((T/R) / (1024 / k')) * (R + E) <= 131040, where k' is k rounded up
 * to a power of two (V3 shape: 64 * 264; 64 ranks x 512 tokens: 256 * 320);
 * larger sizes return EP_ERR_INVALID_ARG before anything is enqueued.
 * The first call on a device looks up the array's device address (a one-time
 * set-up per device); make that first call before any stream capture.
 * Every call clears the part of the array it uses on `stream`, so calls on
 * one device must not overlap on the GPU: two calls in flight at the same time
 * (on different streams) race on the shared array.
 * In:  topk_idx   dev int64 [T][k] (-1 = masked).
 * Out (may be NULL): num_tokens_per_rank dev int32 [R][R],
 *      num_tokens_per_expert dev int32 [R][E], is_token_in_rank dev uint8 [T][R]
 *      -- as ep_get_dispatch_layout.
 * Out (required): num_recv_tokens_per_rank dev int32 [R],
 *      num_recv_tokens_per_expert dev int32 [E], rank_offset dev int32 [R+1],
 *      token_dest dev int32 [T][min(k,R)][2] (8-byte aligned): each token's
 *      destination ranks in ascending order as (rank, row inside the rank's
 *      region), padded with (-1, -1); topk_idx32 dev int32 [T][k]: the ids as
 *      int32 (bad ids as -1).  The global receive row of (t, r) is
 *      rank_offset[r] + row.
 *      device_status dev int32 [1] or NULL: if given (zeroed by the caller),
 *      receives the first device-side status (EP_ERR_BAD_EXPERT,
 *      EP_ERR_TIMEOUT); if NULL such statuses are dropped.  Bad ids are
 *      treated as masked either way.  Always pass it: after a look-back
 *      timeout the offsets may be partial, and without device_status nothing
 *      tells the caller so. */
ep_status_t ep_get_dispatch_layout_noalloc(int num_ranks, int num_experts, int num_topk,
                                           const int64_t* topk_idx, int num_tokens,
                                           int* num_tokens_per_rank, int* num_tokens_per_expert,
                                           uint8_t* is_token_in_rank, int* num_recv_tokens_per_rank,
                                           int* num_recv_tokens_per_expert, int* rank_offset,
                                           int* token_dest, int* topk_idx32, int* device_status,
                                           ep_stream_t stream);

/* Synchronise `stream`, then return and clear the first device-side status
 * latched since the last call (EP_OK if none). */
ep_status_t ep_get_device_status(ep_handle_t h, ep_stream_t stream);

/* Self-check of the bounded waits (failure detection without a fault).
 * Enqueues one small kernel whose waits cannot complete: a flag wait on a
 * device word that nothing sets and an mbarrier wait with no arrivals, each
 * through the same bounded wait as the routing and dispatch kernels.  Each
 * gives up after its poll limit (about half a second apiece), latches
 * EP_ERR_TIMEOUT in the handle and returns, so the kernel ends by itself
 * and the context stays usable; ep_get_device_status() then returns
 * EP_ERR_TIMEOUT (and, as after any timeout, resets the fused kernel's
 * control words).  Writes nothing but the handle's status latch.
 * Returns EP_ERR_INVALID_ARG for a NULL handle, EP_ERR_CUDA if the launch
 * fails. */
ep_status_t ep_check_wait_timeout(ep_handle_t h, ep_stream_t stream);

/* Static, NUL-terminated name of a status. */
const char* ep_status_str(ep_status_t s);

#ifdef __cplusplus
}
#endif

#endif /* GB300_EP_H_ */
