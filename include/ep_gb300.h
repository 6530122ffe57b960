/*
 * ep_gb300.h -- C ABI of the single-GPU MoE expert-parallel hot path:
 * layout, dispatch (bf16 or fused fp8) and combine, for NVIDIA GB300 (sm_103a).
 *
 * The method is the one of TileScale PR #68 "[Example] EP v2 intranode
 * dispatch/combine" (PR summary and README section "Design"): dispatch is a
 * count phase that deduplicates each (token, destination rank) pair, a count
 * exchange that gives every destination a base, and a scatter that writes
 * every row straight to its final compact index; combine reduces, per source
 * token, the rows that token was sent as.  Here the expert-parallel ranks are
 * logical partitions of the expert set inside one GPU's memory, so the count
 * exchange becomes a device-wide prefix scan and the scatter/gather are
 * ordinary HBM traffic.
 *
 * Conventions shared by every call
 *   - All array arguments are DEVICE pointers, allocated and owned by the
 *     caller, row-major, and must stay alive until the stream has passed the
 *     call.  The library allocates nothing, frees nothing, never synchronises
 *     the device or the stream, and keeps no state between calls beyond
 *     per-device launch parameters (SM count, occupancy, kernel attributes)
 *     set up on first use and kept for the life of the process; a
 *     cudaDeviceReset discards the kernel attributes, so the library must
 *     not be called on a device after it has been reset.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Kernels launch on the calling thread's
 *     current CUDA device (cudaSetDevice): every pointer must be that
 *     device's memory and `stream` must belong to it.
 *   - Sizes: T tokens, K top-k slots, E experts, R logical ranks, H hidden,
 *     N = number of dispatched rows = sum of per-rank token counts.
 *     Expert e belongs to rank floor(e / (E/R)); E % R must be 0.
 *   - topk_idx is int64 [T, K]; -1 means "no selection" (TileScale PR #68,
 *     commit message on the masked-topk case).  Any other value outside
 *     [0, E) is treated as -1 and sets EP_ERRBIT_BAD_INDEX in the layout's
 *     error word.
 *   - Host-detectable problems (null or misaligned pointers, sizes out of
 *     range) are reported synchronously by the return value, before anything
 *     is enqueued.  Data-dependent problems never trap and never hang the GPU:
 *     they set bits in the layout's device error word.
 *   - Pointers to arrays that kernels move with 16-byte vectors or bulk copies
 *     (x, recv_x, y, out, token_slot) must be 16-byte aligned.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *ep_stream_t;

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,  /* a pointer, size or alignment is invalid   */
    EP_ERR_UNSUPPORTED = 2,  /* valid, but beyond this library's limits   */
    EP_ERR_CUDA = 3          /* a CUDA runtime call or launch failed      */
} ep_status_t;

typedef enum {
    EP_DTYPE_BF16 = 0,          /* received rows are bit copies of x          */
    EP_DTYPE_FP8_E4M3 = 1,      /* e4m3 rows + a separate fp32 scale array    */
    EP_DTYPE_FP8_E4M3_PACKED = 2 /* e4m3 codes, fp32 scales and zero padding
                                    in one row of ep_fp8_packed_row_bytes(H) */
} ep_dtype_t;

/* Bits of the device error word (ep_layout_t.error_word). */
#define EP_ERRBIT_BAD_INDEX 0x1u  /* a topk_idx entry outside [-1, E)        */
#define EP_ERRBIT_CAPACITY 0x2u   /* a row's slot >= recv_capacity: skipped  */
#define EP_ERRBIT_TIMEOUT 0x4u    /* a bounded device wait gave up (or a hand-
                                     over between a kernel's roles failed)   */
#define EP_ERRBIT_STALE_LAYOUT 0x8u /* routing and layout disagree on a token's
                                       set of ranks (a layout of another routing) */
#define EP_ERRBIT_DUP_EXPERT 0x10u  /* expanded layout: a token names an expert
                                       twice; the repeat gets no row           */

/* Limits of this implementation (EP_ERR_UNSUPPORTED beyond them). */
#define EP_MAX_RANKS 64
#define EP_MAX_TOPK 32
#define EP_MAX_EXPERTS 4096
#define EP_MAX_HIDDEN 16384
#define EP_FP8_GROUP 128          /* elements per fp8 scale */

/*
 * The layout of one routing (the output of ep_get_layout, the input of
 * ep_dispatch and ep_combine).  All members are caller-allocated device
 * pointers:
 *   num_tokens_per_expert [E]   int32: valid selections of each expert.
 *   num_tokens_per_rank   [R]   int32: tokens sent to each rank (a token
 *                               counts once per rank however many of its
 *                               experts live there).
 *   rank_prefix           [R+1] int32: exclusive prefix sum of the above;
 *                               rank r's received rows are
 *                               [rank_prefix[r], rank_prefix[r+1]) and
 *                               rank_prefix[R] = N.
 *   is_token_in_rank      [T*R] uint8: 1 if token t is sent to rank r.
 *   token_slot            [T*R] int32: the received row of (t, r), or -1.
 *                               Rows of one rank are in ascending token
 *                               order (a stable scatter).
 *   error_word            [1]   uint32: EP_ERRBIT_* flags.  ep_get_layout
 *                               clears it; ep_dispatch and ep_combine given
 *                               this layout OR their bits into it.
 *   work_counters  [EP_WORK_COUNTER_WORDS] uint32, 16-byte aligned, or
 *                               NULL.  Given, ep_dispatch and ep_combine hand
 *                               tokens to their thread blocks from a
 *                               grid-wide counter in these words (a block
 *                               that starts late, or draws tokens with many
 *                               destinations, takes fewer), instead of a
 *                               fixed stripe of tokens per block.  The words
 *                               must be zero when a call starts: ep_get_layout
 *                               zeroes them and every call leaves them zero.
 *                               Calls sharing them must be ordered (the same
 *                               stream, or events).  No effect on any result.
 * The layout is the single-GPU counterpart of the count matrix and
 * send_base[d] + slot of TileScale PR #68 (README section "Design").
 */
#define EP_WORK_COUNTER_WORDS 4
typedef struct {
    int32_t *num_tokens_per_expert;
    int32_t *num_tokens_per_rank;
    int32_t *rank_prefix;
    uint8_t *is_token_in_rank;
    int32_t *token_slot;
    uint32_t *error_word;
    uint32_t *work_counters;
} ep_layout_t;

/*
 * Bytes of device workspace ep_get_layout (and ep_get_layout_and_dispatch)
 * needs for these sizes: the per-block, per-rank token totals the layout
 * kernels exchange, after a 256-byte header.  Zero-fill it once when it is
 * allocated; every call leaves the header zeroed again, so the workspace can
 * be reused by later calls with any sizes up to the ones it was sized for.
 * Calls sharing one workspace must be ordered (the same stream, or events).
 */
size_t ep_layout_workspace_bytes(int num_tokens, int num_experts, int num_ranks);

/*
 * Layout: the count phase and the count exchange of TileScale PR #68
 * (README section "Design"; commit message on do_expand, which splits the
 * work into per-destination counting, a base per destination derived from
 * the counts, and a slot claimed locally and added to that base), on one
 * GPU.  Two kernels, the boundary between
 * them standing in for the count exchange: the first counts each block's
 * tokens per rank (warp ballots, one bit per (token, rank) however many
 * experts map there) and publishes per-rank block totals; the second
 * re-reads the ids, counts the experts (shared-memory atomics), derives
 * each rank's base and the block's first slot in it by an exclusive scan of
 * the totals, and writes token_slot.
 *
 *   topk_idx  [T*K] int64, device.
 *   T >= 0 (T == 0 writes zero counts), 1 <= K <= EP_MAX_TOPK,
 *   1 <= R <= EP_MAX_RANKS, R <= E <= EP_MAX_EXPERTS, E % R == 0.
 *   layout    every member non-null (token_slot 16-byte aligned).
 *   workspace >= ep_layout_workspace_bytes(T, E, R) bytes, 16-byte
 *             aligned, zero-filled at allocation (see above).
 */
ep_status_t ep_get_layout(const int64_t *topk_idx, int num_tokens, int num_topk,
                          int num_experts, int num_ranks,
                          const ep_layout_t *layout, void *workspace,
                          size_t workspace_bytes, ep_stream_t stream);

/*
 * ep_get_layout_noalloc: ep_get_layout for callers that cannot allocate
 * device memory.  The pages have no counterpart to it; it is an interface
 * addition of this library.
 *
 * Some callers have no way to obtain a workspace at call time: a plugin
 * running inside another runtime's enqueue callback (an inference engine
 * that owns all device memory and forbids new allocations once it is built),
 * or a latency-critical serving loop where a cudaMalloc or cudaFree could
 * synchronise the device and stall every other stream.  This entry point
 * takes no workspace: its scratch (the per-block rank totals the layout
 * kernels exchange) is a file-scope static device array of
 * EP_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits.  It calls no allocating
 * routine.  The caller still passes topk_idx and the layout outputs.
 *
 *   Limit: the layout kernels run at most 2048 thread blocks and keep
 *   R four-byte totals per block after a 256-byte header, so a call uses
 *   256 + 4 * R * min(ceil(T / 256), 2048) bytes (rounded up to 256) of
 *   the scratch.  That must not exceed EP_NOALLOC_SCRATCH_BYTES, else
 *   EP_ERR_UNSUPPORTED: any T fits for R <= 31; for R = 32 the limit is
 *   T <= 523,776 tokens, for R = 64, T <= 261,888.
 *   Set-up: the first call on a device looks up the device address of the
 *   scratch array once (with that device current) and keeps it for the
 *   life of the process; make that first call before any stream capture.
 *   Like the library's other per-device set-up (kernel attributes,
 *   device properties), it does not survive a cudaDeviceReset of that
 *   device: do not call the library on a device after resetting it.
 *   Every call clears the scratch it uses, on `stream`, before its kernel.
 *   One scratch per device is shared by every call: calls that overlap on
 *   the GPU (unordered streams) race on it and produce wrong layouts, so
 *   order them (one stream, or events).
 *   Arguments, outputs and errors are otherwise those of ep_get_layout.
 */
#define EP_NOALLOC_SCRATCH_BYTES (256u * 1024u)
ep_status_t ep_get_layout_noalloc(const int64_t *topk_idx, int num_tokens, int num_topk,
                                  int num_experts, int num_ranks,
                                  const ep_layout_t *layout, ep_stream_t stream);

/*
 * Dispatch: the scatter phase of TileScale PR #68 (PR summary: rows go
 * straight to their final compact index, no copy epilogue), with the fp8
 * cast of DeepEP's per_token_cast_to_fp8 layout fused into the same pass
 * (same page, commit message on packing the fp8 row: per-token,
 * per-128-element fp32 scales; no separate scale transfer).  Each token's
 * row is read once and written to every rank it is sent to.
 *
 *   x            [T*H] bf16 (uint16 bit patterns), device, 16-byte aligned.
 *   topk_idx     [T*K] int64 and topk_weights [T*K] fp32, device: the same
 *                routing ep_get_layout saw (topk_weights may be NULL only if
 *                recv_topk_weights is NULL).
 *   layout       from ep_get_layout on this routing.
 *   dtype        EP_DTYPE_BF16: recv_x is bf16 [recv_capacity*H];
 *                  H % 8 == 0.
 *                EP_DTYPE_FP8_E4M3: recv_x is e4m3 [recv_capacity*H] and
 *                  recv_x_scales fp32 [recv_capacity*(H/128)]; H % 128 == 0.
 *                  Per 128-element group: amax = max|x|,
 *                  scale = amax / 448 (fp32, round to nearest even),
 *                  code = e4m3(x / scale) rounded to nearest even and
 *                  saturated to +-448; an all-zero group has scale 0.
 *   recv_src_idx      [recv_capacity] int32: source token of each row.
 *   recv_topk_idx     [recv_capacity*K] int32: local expert (e - r*E/R) of
 *                     each top-k slot whose expert is on the row's rank r,
 *                     else -1 (same page, commit message adding cumulative
 *                     recv stats: recv_topk_idx holds the local expert).
 *   recv_topk_weights [recv_capacity*K] fp32: the gate weight where
 *                     recv_topk_idx != -1, else 0.
 *   The three metadata outputs may each be NULL (not written).
 *   recv_capacity >= 0: rows whose slot >= recv_capacity are skipped and set
 *                EP_ERRBIT_CAPACITY; T*min(K,R) always suffices.
 *   Rows [N, recv_capacity) are not written.
 *   1 <= H <= EP_MAX_HIDDEN.
 *
 * Cached layouts: a layout depends only on each token's set of ranks, so it
 * may be reused for any routing with the same rank sets (TileScale PR #68,
 * commit messages on the cached-layout dispatch: the notify phase is skipped
 * when the routing is unchanged).  A stale layout would misroute silently;
 * here every call compares each token's rank set under `topk_idx` with the
 * ranks that have a slot and sets EP_ERRBIT_STALE_LAYOUT on a mismatch (the
 * rows are still written where the layout says).
 */
ep_status_t ep_dispatch(const void *x, int num_tokens, int hidden,
                        const int64_t *topk_idx, const float *topk_weights,
                        int num_topk, int num_experts, int num_ranks,
                        const ep_layout_t *layout, ep_dtype_t dtype,
                        void *recv_x, float *recv_x_scales,
                        int32_t *recv_src_idx, int32_t *recv_topk_idx,
                        float *recv_topk_weights, int recv_capacity,
                        ep_stream_t stream);

/*
 * Bytes of one packed fp8 row (EP_DTYPE_FP8_E4M3_PACKED): the H e4m3 codes,
 * then the H/128 fp32 scales, then zero padding to a multiple of 16 bytes,
 * or of 512 bytes when that padding adds under 5% to the unpadded row
 * (TileScale PR #68, commit message on packing the fp8 row: 132 raw bytes at
 * hidden 128; 7392 raw, 7680 padded at 7168).  0 if hidden is not a
 * positive multiple of 128.
 */
size_t ep_fp8_packed_row_bytes(int hidden);

/*
 * Dispatch with every option.  Members as for ep_dispatch, plus:
 *   dtype == EP_DTYPE_FP8_E4M3_PACKED: recv_x is uint8
 *     [recv_capacity * ep_fp8_packed_row_bytes(H)]; each row holds the codes,
 *     then the scales, then zeros (TileScale PR #68, commit message on packing
 *     the fp8 row); recv_x_scales is ignored.  H % 128 == 0.
 *   cumulative_recv_stats  uint32 [E] or NULL: for every received
 *     (row, top-k slot) of expert e, stats[e] += 1 -- rank r's count for its
 *     local expert e - r*E/R, accumulated, never cleared, so the caller picks
 *     the window by zeroing it (same page, commit message adding cumulative
 *     recv stats).
 */
typedef struct {
    const void *x;
    int num_tokens;
    int hidden;
    const int64_t *topk_idx;
    const float *topk_weights;
    int num_topk;
    int num_experts;
    int num_ranks;
    const ep_layout_t *layout;
    ep_dtype_t dtype;
    void *recv_x;
    float *recv_x_scales;
    int32_t *recv_src_idx;
    int32_t *recv_topk_idx;
    float *recv_topk_weights;
    int recv_capacity;
    uint32_t *cumulative_recv_stats;
} ep_dispatch_args_t;
ep_status_t ep_dispatch_ex(const ep_dispatch_args_t *args, ep_stream_t stream);

/*
 * ep_get_layout of args->topk_idx into *args->layout, then ep_dispatch_ex
 * with the same arguments, as one call: the notify (count and exchange) and
 * the scatter of TileScale PR #68 issued together (same page, commit
 * messages fusing the layout back into the dispatch).  The work is the same
 * two launches, overlapped: the kernel ahead of the dispatch is known to be
 * the layout, which writes nothing the dispatch reads first, so each
 * dispatch block loads (and for fp8 casts) the rows of its first tokens
 * while the layout still runs, and waits for it only to store them.  With
 * 0 < T <= 524,288 the layout is one launch: it writes is_token_in_rank,
 * each slot relative to its block of 256 tokens and each block's per-rank
 * totals.  When the blocks times the ranks number at most 1024, the
 * dispatch itself scans those totals into each block's base and writes
 * rank_prefix and num_tokens_per_rank; beyond that, the layout's last block
 * to finish does the scan.  The dispatch adds each block's base as it moves
 * the token, writes the final slot back and counts num_tokens_per_expert
 * (and bad ids).  Every output of both calls is written, identical to the
 * two calls (on that path, if the dispatch gives up with
 * EP_ERRBIT_TIMEOUT, the tokens it did not reach keep their block-relative
 * slots and are not counted).
 *   args       as for ep_dispatch_ex; every array of *args->layout is
 *              written (as ep_get_layout), so its token_slot and
 *              is_token_in_rank must be 16-byte aligned.
 *   workspace  ep_layout_workspace_bytes(T, E, R) bytes, as for
 *              ep_get_layout (the same buffer serves both calls).
 * Errors: those of ep_get_layout and ep_dispatch_ex, checked before any
 * launch.
 */
ep_status_t ep_get_layout_and_dispatch(const ep_dispatch_args_t *args, void *workspace, size_t workspace_bytes,
                                       ep_stream_t stream);

/*
 * Combine: the local reduce of TileScale PR #68 (PR summary: one block per
 * source token reduces the rows stored back for it).  On one GPU the
 * store-back slot comm_x[rank][src_token] is the received row
 * token_slot[t][r] itself, so combine gathers straight from the expert
 * stage's output:
 *
 *   out[t] = bf16( sum over r = 0..R-1 ascending with token_slot[t][r] >= 0
 *                  of c[t][r] * y[token_slot[t][r]] )
 *
 * accumulated in fp32 with separate multiply and add, rounded to nearest
 * even at the end.  c = 1 when topk_weights is NULL (the pages' combine);
 * otherwise c[t][r] is the fp32 sum, in k order, of the weights of t's
 * experts on rank r.  A token sent nowhere combines to +0 (same page,
 * commit message on the masked-topk case).
 *
 *   y        [recv_capacity*H] bf16, device, 16-byte aligned: row s is the
 *            expert output for received row s.  Rows with
 *            token_slot >= recv_capacity are skipped (EP_ERRBIT_CAPACITY).
 *   layout   the layout the rows were dispatched with.
 *   topk_idx, topk_weights: [T*K] device, or both NULL for the plain sum.
 *   out      [T*H] bf16, device, 16-byte aligned.  H % 8 == 0.
 *   With weights, a token whose rank set under topk_idx differs from the
 *   layout's sets EP_ERRBIT_STALE_LAYOUT (see ep_dispatch).
 */
ep_status_t ep_combine(const void *y, int recv_capacity, int hidden,
                       const ep_layout_t *layout, int num_tokens, int num_ranks,
                       const int64_t *topk_idx, const float *topk_weights,
                       int num_topk, int num_experts, void *out,
                       ep_stream_t stream);

/*
 * Combine with every option.  Members as for ep_combine, plus:
 *   bias0, bias1  bf16 [T*H] or NULL, 16-byte aligned: they seed the fp32
 *     accumulator, acc = bias0 (or 0), then acc = acc + bias1, before the
 *     rank rows are added, so a token sent nowhere comes back as its bias
 *     (TileScale PR #68, commit message adding combine bias: bias_0/bias_1
 *     seed the reduce accumulator).
 */
typedef struct {
    const void *y;
    int recv_capacity;
    int hidden;
    const ep_layout_t *layout;
    int num_tokens;
    int num_ranks;
    const int64_t *topk_idx;
    const float *topk_weights;
    int num_topk;
    int num_experts;
    const void *bias0;
    const void *bias1;
    void *out;
} ep_combine_args_t;
ep_status_t ep_combine_ex(const ep_combine_args_t *args, ep_stream_t stream);

/* ------------------------------------------------------------------ */
/* Expanded (per-expert) layout                                        */
/* ------------------------------------------------------------------ */

/*
 * The expanded layout of one routing: one received row per (token, expert)
 * selection instead of per (token, rank), rows grouped by expert so that
 * each expert's rows form the contiguous block a grouped GEMM consumes, each
 * block rounded up to expert_alignment rows (TileScale PR #68, commit
 * message on do_expand).  Experts are contiguous per rank, so the rows are
 * rank-major too: rank r's rows are
 * [expert_offset[r*E/R], expert_offset[(r+1)*E/R]).  Caller-allocated:
 *   num_rows_per_expert [E]   int32: rows of each expert.
 *   expert_offset       [E+1] int32: first row of each expert's block (the
 *                             exclusive prefix sum of rows rounded up to the
 *                             alignment); expert_offset[E] is the number of
 *                             rows including padding.
 *   token_slot          [T*K] int32: the row of (t, k), or -1 (no
 *                             selection, an invalid id, or a repeat of an
 *                             expert already named by t).  Inside a block
 *                             rows are in ascending (token, k) order.
 *   error_word          [1]   uint32: EP_ERRBIT_* (cleared by the layout).
 *   work_counters       [EP_WORK_COUNTER_WORDS] uint32 or NULL: as in
 *                             ep_layout_t (zeroed by ep_get_layout_expanded).
 */
typedef struct {
    int32_t *num_rows_per_expert;
    int32_t *expert_offset;
    int32_t *token_slot;
    uint32_t *error_word;
    uint32_t *work_counters;
} ep_expanded_layout_t;

/* Workspace bytes of ep_get_layout_expanded (zero-filled once at
 * allocation, left zeroed by every call, reusable for smaller sizes). */
size_t ep_expanded_layout_workspace_bytes(int num_tokens, int num_experts);

/*
 * The expanded layout: phase 1 tallies rows per expert, phase 2 turns the
 * tallies into aligned segment starts, phase 3 adds each row's rank in its
 * segment -- the do_expand generalisation of the count / exchange / scatter
 * phases with the destination redefined from rank to expert (TileScale PR
 * #68, commit message on do_expand).  One cooperative kernel with a bounded
 * grid barrier.  1 <= expert_alignment <= 4096; limits as ep_get_layout;
 * token_slot 16-byte aligned.
 */
ep_status_t ep_get_layout_expanded(const int64_t *topk_idx, int num_tokens, int num_topk,
                                   int num_experts, int expert_alignment,
                                   const ep_expanded_layout_t *layout, void *workspace,
                                   size_t workspace_bytes, ep_stream_t stream);

/*
 * Expanded dispatch: row token_slot[t][k] receives x[t] (bf16, fp8 + scales,
 * or packed fp8), recv_src_idx = t, and recv_topk_idx / recv_topk_weights
 * mark only slot k -- the row's own expert as a local id, and its weight --
 * with -1 / 0 elsewhere (same page: an expanded row marks only the expert it
 * belongs to).  zero_padding != 0: the padding rows of every block are
 * written as zeros (payload and scales), source -1, all top-k slots -1 and
 * weights 0 (zero_padding clears the gap).  Rows at or past recv_capacity
 * are skipped with EP_ERRBIT_CAPACITY; expert_offset[E] rows always suffice.
 * cumulative_recv_stats counts each written row for its expert.  Members
 * otherwise as ep_dispatch_args_t; num_ranks gives the local ids.
 */
typedef struct {
    const void *x;
    int num_tokens;
    int hidden;
    const int64_t *topk_idx;
    const float *topk_weights;
    int num_topk;
    int num_experts;
    int num_ranks;
    const ep_expanded_layout_t *layout;
    ep_dtype_t dtype;
    void *recv_x;
    float *recv_x_scales;
    int32_t *recv_src_idx;
    int32_t *recv_topk_idx;
    float *recv_topk_weights;
    int recv_capacity;
    int zero_padding;
    uint32_t *cumulative_recv_stats;
} ep_dispatch_expanded_args_t;
ep_status_t ep_dispatch_expanded(const ep_dispatch_expanded_args_t *args, ep_stream_t stream);

/*
 * Expanded combine: out[t] = bf16(bias0 + bias1 + the sum, in ascending row
 * order, of c * y[row] over t's rows), fp32 with separate multiply and add;
 * c is the row's own gate weight (topk_weights given) or 1.  This is
 * DeepEP's kDoExpandedSend -- a token's rows summed before the rank reduce
 * (same page, commit message on the expanded combine) -- on one GPU.
 * y has recv_capacity rows indexed like the dispatched rows.
 */
typedef struct {
    const void *y;
    int recv_capacity;
    int hidden;
    const ep_expanded_layout_t *layout;
    int num_tokens;
    int num_topk;
    const int64_t *topk_idx;
    const float *topk_weights;
    int num_experts;
    const void *bias0;
    const void *bias1;
    void *out;
} ep_combine_expanded_args_t;
ep_status_t ep_combine_expanded(const ep_combine_expanded_args_t *args, ep_stream_t stream);

/*
 * Self-test of the bounded device waits (the pages have no counterpart: the
 * library's own guarantee that a data or hand-over problem never hangs the
 * GPU).  Launches two blocks of 32 threads on `stream`: block 0 waits on an
 * mbarrier that nothing arrives on, the form of the dispatch and combine
 * stage waits; block 1 enters a grid barrier that block 0 never reaches, the
 * form of the expanded layout's barrier.  Each wait gives up after the
 * library's wait limit (1 s of the GPU's global timer), and the kernel
 * returns.
 *   error_word  [1] uint32: EP_ERRBIT_TIMEOUT is OR-ed in by a wait that gave up
 *   gave_up     [2] int32 : 1 where wait i (0: mbarrier, 1: grid barrier)
 *                           gave up, 0 where it completed
 *   elapsed_ns  [2] uint64: the time each wait took, from the global timer
 * Device pointers, caller-owned, 4-, 4- and 8-byte aligned; NULL or
 * misaligned gives EP_ERR_INVALID_ARG.  Takes about one second of GPU time;
 * calls must not overlap on the GPU (the grid barrier's words are a static
 * device variable).
 */
ep_status_t ep_selftest_bounded_waits(uint32_t *error_word, int32_t *gave_up, uint64_t *elapsed_ns,
                                      ep_stream_t stream);

/* A static, human-readable name of a status. */
const char *ep_status_str(ep_status_t status);

/* The detail message of the last failing call on this host thread ("" if
 * none).  Valid until the next call on the same thread. */
const char *ep_last_error(void);

/* ABI version of this header: bumped on any incompatible change. */
#define EP_ABI_VERSION 2
int ep_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
