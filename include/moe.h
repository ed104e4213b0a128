/*
 * moe.h - C ABI of the GB300 MoE dispatch + combine library (libmoe.so).
 *
 * One MoE layer on one GPU: tokens are routed to experts (dispatch), expert
 * outputs are gathered back and reduced with the router weights (combine).
 * "Ranks" are logical partitions of one GPU's memory: logical rank s owns
 * tokens [s*T/N, (s+1)*T/N) and experts [r*E/N, (r+1)*E/N) live on rank r.
 * Nothing crosses a GPU boundary.
 *
 * The four calls follow the split send/receive kernel pairs of
 * "Efficient and portable mixture-of-experts communication" (Portable
 * kernels; Dispatch; Combine) and "Enabling trillion-parameter models on AWS
 * EFA" (Dispatch and combine: send halves pack, receive halves hand the
 * grouped tensor to the grouped GEMM or compute the weighted average).
 *
 * Conventions for every call:
 *  - Device pointers are plain CUDA device addresses owned by the caller; the
 *    library allocates no device memory and keeps no global device state.
 *    The only host allocation is the small moe_ctx handle.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on that stream and returns
 *    without waiting, except moe_get_error, which synchronises the stream.
 *  - bf16 tensors are row-major, rows of H elements; x, expert_x, expert_y and
 *    out must be 16-byte aligned (H must be a multiple of 8, so every row is).
 *  - Return value: MOE_OK or one of the MOE_E* codes below.  Argument errors
 *    are detected on the host before anything is enqueued.  Routing errors
 *    (an expert index out of range or repeated within one token) are detected
 *    on the device; they are reported by moe_get_error and by the error word
 *    that moe_dispatch_recv exposes.  After a routing error no row of
 *    expert_x and no row of out is written.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_EINVAL 1    /* bad argument: null/misaligned pointer, bad sizes */
#define MOE_ESTATE 2    /* calls out of order for this context */
#define MOE_EROUTE 3    /* device: expert index out of range or repeated in a token */
#define MOE_ECUDA 4     /* a CUDA runtime call or a launch failed */
#define MOE_EBOUND 5    /* device: a rank would receive more than N*T/N*max(K,E/N) rows */
#define MOE_ETIMEDOUT 6 /* device: a bounded wait inside a kernel gave up */
#define MOE_ECORRUPT 7  /* device, checked builds only: a routing-table entry points outside its buffer */

/* Limits of this implementation. */
#define MOE_MAX_TOP_K 16
#define MOE_MAX_EXPERTS 1024

/* Sizes of one layer.  T % N == 0, E % N == 0, 1 <= K <= min(E, 16),
 * E <= 1024, H % 8 == 0, T*K < 2^31.  T == 0 is allowed (an empty layer). */
typedef struct moe_config {
  int32_t num_tokens;  /* T: tokens over all logical ranks */
  int32_t hidden;      /* H: bf16 elements per token row */
  int32_t top_k;       /* K: experts per token */
  int32_t num_experts; /* E */
  int32_t num_ranks;   /* N: logical ranks */
} moe_config;

/* Opaque per-layer context: the configuration, the caller's workspace and
 * the phase of the send/recv sequence. */
typedef struct moe_ctx moe_ctx;

/* Where dispatch put things.  All pointers are device pointers into the
 * workspace, valid until the next moe_dispatch_send on the same context;
 * their contents are ready in stream order after moe_dispatch_send.
 *
 * Row layout of expert_x (and of expert_y for combine): rows are grouped by
 * expert, experts in index order, so the rows of logical rank r's experts are
 * the contiguous range [rank_offsets[r], rank_offsets[r+1]).  Inside one
 * expert, rows are ordered by source rank, then by token within the rank
 * (equivalently, by global token index).  This placement is unique. */
typedef struct moe_dispatch_layout {
  const int32_t* expert_counts;  /* [E]   rows received by each expert */
  const int32_t* expert_offsets; /* [E+1] first row of each expert; [E] = T*K */
  const int32_t* src_offsets;    /* [E*N] first row of (expert e, source rank s) at e*N+s */
  const int32_t* rank_offsets;   /* [N+1] first row of rank r's experts; [N] = T*K */
  const int32_t* slot_row;       /* [T*K] row that token t's k-th choice went to, at t*K+k */
  const int32_t* row_src;        /* [T*K] for each row, t*K+k of the (token, slot) it holds */
  const int32_t* error_word;     /* [1]   MOE_OK or the device-detected status */
  int64_t rows;                  /* T*K: rows written at the front of expert_x */
  int64_t recv_bound_rows;       /* N*(T/N)*max(K, E/N): most rows one rank can receive */
} moe_dispatch_layout;

/* Checks a configuration against the limits above.  MOE_OK or MOE_EINVAL. */
int moe_validate_config(const moe_config* cfg);

/* Device workspace (bytes, a multiple of 256) that one context needs: counts,
 * offsets, slot_row, row_src, the error word, the send tables of
 * moe_dispatch_send_staged and moe_dispatch_send_dense, the plan of
 * moe_combine_recv_two_level and the
 * pack's and the combine's work-queue counters.  Allocate it 256-byte
 * aligned; its contents need no initialisation (every dispatch writes what it
 * later reads). */
int moe_workspace_bytes(const moe_config* cfg, size_t* bytes);

/* The receive bound of "Enabling trillion-parameter models on AWS EFA"
 * (Send and receive buffers): with N ranks of T/N tokens each routed to K of
 * E experts, one rank receives at most N*(T/N)*max(K, E/N) rows. */
int moe_recv_bound_rows(const moe_config* cfg, int64_t* rows);

/* Creates a context over a caller-owned device workspace of at least
 * moe_workspace_bytes() bytes.  Must be called with the device that owns the
 * workspace current; all later calls must use a stream of that device.
 * The context is not thread-safe: one host thread drives one context.
 * MOE_EINVAL for a bad configuration, a null, short or misaligned workspace,
 * a configuration whose routing tables do not fit in shared memory, or when
 * the host handle cannot be allocated; MOE_ECUDA if a device query fails. */
int moe_ctx_create(const moe_config* cfg, void* workspace, size_t workspace_bytes, moe_ctx** out);

/* Frees the host handle (not the workspace). NULL is a no-op. */
int moe_ctx_destroy(moe_ctx* ctx);

/* Dispatch, send half ("Enabling trillion-parameter models on AWS EFA",
 * Dispatch and combine: count tokens per expert with shared-memory atomics,
 * take the cumulative sum of the counts, pack the tokens at those offsets).
 * Enqueues the routing kernels (counts, exclusive scan, stable slot ranks,
 * routing error check: by default route_cluster, one thread-block cluster of
 * up to 16 CTAs that exchange per-chunk counts through distributed shared
 * memory; see MOE_OPT_ROUTE_VARIANT) and dispatch_pack (copies each token row
 * x[t] to expert_x[slot_row[t,k]] for every k).  For small layers (T*K <=
 * 16384, E*ceil(T/32) <= 4096) both run as one kernel, route_pack, whose CTAs
 * each compute the routing tables before copying: one kernel boundary less
 * on the layer's critical path.  The results are the same either way.
 *   x         device bf16 [T, H], read only
 *   topk_idx  device int32 [T, K], read only, 4-byte aligned
 *   expert_x  device bf16 [expert_x_rows, H]; rows [0, T*K) are written,
 *             later rows are left untouched.  expert_x_rows >= T*K.
 * Valid in the idle phase (after create or after moe_combine_recv). */
int moe_dispatch_send(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* expert_x,
                      int64_t expert_x_rows, void* stream);

/* Dispatch, send half, with a block-scaled fp8 payload ("Efficient and
 * portable mixture-of-experts communication", Dispatch: tokens are sent with
 * their block scaling factors; "Enabling trillion-parameter models on AWS
 * EFA", evaluation: block-scale fp8 dispatch, bf16 combine).  Same routing
 * and row placement as moe_dispatch_send; each token row is quantised once:
 * for every block of MOE_FP8_BLOCK consecutive elements,
 *   scale = amax(|x|) / 448 in float32 (1 for an all-zero block),
 *   inv = 1 / scale (float32 division, once per block),
 *   q = E4M3(x * inv), float32 product, round to nearest even, saturating;
 * and expert_xq[slot_row[t,k]] = q[t], expert_scales[slot_row[t,k]] = scale[t].
 *   x              device bf16 [T, H], H % MOE_FP8_BLOCK == 0
 *   expert_xq      device E4M3 bytes [expert_rows, H], 16-byte aligned
 *   expert_scales  device float32 [expert_rows, H / MOE_FP8_BLOCK]
 *   expert_rows    >= T*K; rows [0, T*K) of both are written
 * The combine that follows still takes bf16 expert outputs.  For the small
 * layers of moe_dispatch_send's route_pack, routing and quantisation run as
 * one kernel, route_pack_fp8 (MOE_OPT_ROUTE_VARIANT_FP8 reports the path);
 * the results are the same either way.  Valid in the idle phase; MOE_EINVAL
 * if H is not a multiple of the block or a bf16 row is too large for two
 * shared-memory stages. */
#define MOE_FP8_BLOCK 128
int moe_dispatch_send_fp8(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* expert_xq,
                          float* expert_scales, int64_t expert_rows, void* stream);

/* Dispatch, send half, for tokens the caller has already quantised to fp8
 * (the other reading of "Efficient and portable mixture-of-experts
 * communication", Dispatch: tokens travel together with their block scaling
 * factors).  Same routing and row placement as moe_dispatch_send; the E4M3
 * code rows and their float32 block-scale rows are copied as they are:
 *   expert_xq[slot_row[t,k]] = xq[t], expert_scales[slot_row[t,k]] = x_scales[t].
 *   xq             device E4M3 bytes [T, H], 16-byte aligned
 *   x_scales       device float32 [T, H / MOE_FP8_BLOCK], 16-byte aligned
 *   expert_xq      device E4M3 bytes [expert_rows, H], 16-byte aligned
 *   expert_scales  device float32 [expert_rows, H / MOE_FP8_BLOCK], 16-byte aligned
 *   expert_rows    >= T*K; rows [0, T*K) of both are written
 * H must be a multiple of 512 (scale rows a multiple of 16 bytes); MOE_EINVAL
 * otherwise.  Errors and call order as for moe_dispatch_send. */
int moe_dispatch_send_quantized(moe_ctx* ctx, const void* xq, const float* x_scales, const int32_t* topk_idx,
                                void* expert_xq, float* expert_scales, int64_t expert_rows, void* stream);

/* Dispatch, send half, two-stage form ("Enabling trillion-parameter models on
 * AWS EFA", dispatch and combine timing: the sender copies tokens into
 * contiguous per-peer send buffers at offsets from the cumulative sum of its
 * per-expert counts; the receiver then shuffles them from its receive buffer
 * into the grouped-GEMM input).  Same routing and same results as
 * moe_dispatch_send, which writes every row straight to its grouped position
 * (send and receive memory are one on a single GPU); this form keeps the
 * pages' extra copy so that its cost can be measured.  Enqueues routing, a
 * send-layout kernel and two pack kernels:
 *   stage 1: source rank s's (token, slot) pairs, in (expert, token) order,
 *            go to send rows [s*T/N*K, (s+1)*T/N*K) of send_buf (x rows);
 *   stage 2: every send row is copied to its row of expert_x.
 *   send_buf   device bf16 [send_rows, H], send_rows >= T*K, 16-byte aligned,
 *              caller-owned scratch (only rows [0, T*K) are written)
 *   x, topk_idx, expert_x, expert_x_rows  as for moe_dispatch_send
 * Errors as for moe_dispatch_send; after a routing error nothing is written to
 * send_buf or expert_x.  Valid in the idle phase; moe_dispatch_recv follows. */
int moe_dispatch_send_staged(moe_ctx* ctx, const void* x, const int32_t* topk_idx, void* send_buf, int64_t send_rows,
                             void* expert_x, int64_t expert_x_rows, void* stream);

/* ---- Dense padded all-to-all (the pages' comparison system) -----------------
 * "Efficient and portable mixture-of-experts communication" (Sharding and
 * parallelism): torch's all_to_all needs padding (or a GPU-CPU
 * synchronisation) because ranks send different numbers of tokens to each
 * peer; (Benchmarks) the dense all-to-all is bandwidth-bound and moves an
 * order of magnitude more data than the sparse kernels.  These two calls run
 * a layer that way on one GPU, for measuring that difference: every (source
 * rank s, destination rank r) chunk is a block of `capacity` rows fixed before
 * the layer, so no count is exchanged.
 *
 * Smallest valid capacity: the most rows one source rank can send to one
 * rank, T/N * min(K, E/N) (at least 1).  MOE_EINVAL for an invalid config. */
int moe_dense_capacity(const moe_config* cfg, int64_t* rows);

/* Dispatch, send half, through the dense padded all-to-all.  Same routing and
 * same grouped rows in expert_x as moe_dispatch_send; on the way:
 *   send_buf block s*N+r (rows [(s*N+r)*capacity, +capacity)): source rank s's
 *     rows for the experts of rank r, in (expert, token) order, then padding
 *     (rows left as they were);
 *   recv_buf block r*N+s = send_buf block s*N+r, all `capacity` rows
 *     (padding included: the exchange moves N*N*capacity rows);
 *   expert_x: the receivers' rows, grouped by expert.
 *   capacity        >= moe_dense_capacity; N*N*capacity < 2^31
 *   send_buf, recv_buf  device bf16 [buf_rows, H] each, caller-owned scratch,
 *                   16-byte aligned, buf_rows >= N*N*capacity
 *   x, topk_idx, expert_x, expert_x_rows  as for moe_dispatch_send
 * Enqueues routing, a block-layout kernel (each pair's block rows), the bulk
 * pack into send_buf, the exchange (dense_a2a) and a row copy into expert_x.
 * After a routing error nothing is written to send_buf, recv_buf or expert_x.
 * Errors and call order as for moe_dispatch_send; moe_combine_recv (grouped
 * rows) or moe_combine_recv_dense may follow. */
int moe_dispatch_send_dense(moe_ctx* ctx, const void* x, const int32_t* topk_idx, int64_t capacity, void* send_buf,
                            void* recv_buf, int64_t buf_rows, void* expert_x, int64_t expert_x_rows, void* stream);

/* Combine, receive half, through the dense padded all-to-all back: every
 * expert rank returns its outputs (expert_y of moe_combine_send) in the
 * blocks they came in by, the exchange moves block r*N+s of send_buf to block
 * s*N+r of recv_buf whole, then the receiver-only combine of moe_combine_recv
 * runs on the returned rows (same float32 chain, same bits).  Valid after
 * moe_combine_send when the dispatch was moe_dispatch_send_dense with the same
 * capacity (MOE_ESTATE otherwise; MOE_EINVAL for another capacity).
 * send_buf and recv_buf as for moe_dispatch_send_dense (the dispatch's may be
 * reused); out and topk_w as for moe_combine_recv. */
int moe_combine_recv_dense(moe_ctx* ctx, const float* topk_w, int64_t capacity, void* send_buf, void* recv_buf,
                           int64_t buf_rows, void* out, void* stream);

/* Dispatch, receive half.  On one GPU the send half already placed every row
 * in the grouped layout (the shared-buffer case of "Efficient and portable
 * mixture-of-experts communication", Further improvements), so this enqueues
 * nothing: it fills `layout` with device pointers to the counts, offsets and
 * routing tables.  Valid after moe_dispatch_send, moe_dispatch_send_fp8,
 * moe_dispatch_send_quantized, moe_dispatch_send_staged or
 * moe_dispatch_send_dense. */
int moe_dispatch_recv(moe_ctx* ctx, moe_dispatch_layout* layout, void* stream);

/* Combine, send half: registers the expert outputs, one row per dispatched
 * (token, slot) pair in the same row layout as expert_x.  Nothing is copied
 * (the senders' per-expert regions are this GPU's own memory).
 *   expert_y  device bf16 [expert_y_rows, H], expert_y_rows >= T*K
 * Valid after moe_dispatch_recv. */
int moe_combine_send(moe_ctx* ctx, const void* expert_y, int64_t expert_y_rows, void* stream);

/* Combine, receive half ("Efficient and portable mixture-of-experts
 * communication", Combine: the weighted average of all expert contributions,
 * computed where the token lives, into a caller-allocated tensor).  Enqueues
 * the combine kernel:
 *   out[t, h] = bf16_rne( fma chain over k = 0..K-1 of
 *                         topk_w[t, k] * expert_y[slot_row[t, k], h], from +0.0f )
 * accumulated in float32 in top-k order, rounded once to bf16 (nearest even).
 *   topk_w  device float32 [T, K], 4-byte aligned
 *   out     device bf16 [T, H]
 * Valid after moe_combine_send; returns the context to the idle phase. */
int moe_combine_recv(moe_ctx* ctx, const float* topk_w, void* out, void* stream);

/* Combine, receive half, two-level form: partial sums on the sending side
 * ("Enabling trillion-parameter models on AWS EFA", evaluation, prefill:
 * DeepEP adds a token's expert outputs on the sender to move less data, which
 * can cost precision; moe_combine_recv adds only at the receiver).  An
 * alternative to moe_combine_recv, for measuring that trade.  Enqueues a
 * plan kernel (each token's slots sorted by rank) and two reduction kernels:
 *   level 1: for each token t and each rank r holding some of its experts,
 *     partial = bf16_rne( fma chain over those experts in top-k order of
 *                         topk_w[t, k] * expert_y[slot_row[t, k], h], from +0.0f )
 *     written to partial row t*min(K,N) + d, d = the position of r among the
 *     token's ranks in ascending order;
 *   level 2: out[t, h] = bf16_rne( float32 sum of the token's partials in
 *                                  ascending rank order, from +0.0f ).
 *   topk_w        device float32 [T, K], 4-byte aligned
 *   partial       device bf16 [partial_rows, H], 16-byte aligned, caller-owned
 *                 scratch; partial_rows >= T*min(K,N) (moe_partial_rows);
 *                 rows a token does not use are left untouched
 *   out           device bf16 [T, H]
 * A token whose routing failed (MOE_EROUTE) gets nothing written.  Returns
 * MOE_EINVAL for a short or misaligned buffer.  Valid after moe_combine_send;
 * returns the context to the idle phase. */
int moe_combine_recv_two_level(moe_ctx* ctx, const float* topk_w, void* partial, int64_t partial_rows, void* out,
                               void* stream);

/* Rows of the partial buffer moe_combine_recv_two_level needs: T*min(K,N).
 * Returns MOE_EINVAL for an invalid configuration. */
int moe_partial_rows(const moe_config* cfg, int64_t* rows);

/* Launch options of one context (tuning knobs; the defaults are the tuned
 * configuration).  Returns MOE_EINVAL for an unknown option or value.
 *   MOE_OPT_PACK_VARIANT      0 = bulk copies through shared memory (TMA
 *                             engine, default), 1 = 16-byte vector loads/stores
 *                             (the receive shuffle of moe_dispatch_send_staged
 *                             always uses the vector copy)
 *   MOE_OPT_PACK_STAGES       shared-memory stages per bulk CTA, 2..16, 0 =
 *                             automatic (about 200 KiB of stages per SM, default;
 *                             fp8 pack: about 72 KiB per CTA for K >= 4, else 3;
 *                             route_pack_fp8: whole-row stages per group of 128
 *                             threads, as many as fit)
 *   MOE_OPT_PACK_PIECE_BYTES  bytes of a row moved per work unit, a multiple of
 *                             16, 0 = automatic (whole row up to 8 KiB, else
 *                             equal pieces of at most 8 KiB)
 *   MOE_OPT_PACK_CTAS_PER_SM  0 = automatic (bulk variant: 2 for K >= 4, else 3;
 *                             fp8 pack: 3 for K >= 4, else up to 8;
 *                             route_pack: copy warps per CTA; route_pack_fp8:
 *                             groups of 128 threads per CTA, at most 8), else
 *                             1..32
 *   MOE_OPT_PDL               1 = launch pack/combine with programmatic
 *                             dependent launch (default), 0 = plain launches
 *   MOE_OPT_ROUTE_VARIANT     routing kernels: 0 = automatic (for
 *                             moe_dispatch_send of a small layer, 4 when the
 *                             bulk pack and its automatic or static split are
 *                             selected; otherwise route_cluster when the
 *                             device can schedule its cluster, else
 *                             route_local + route_finalize), 1 = the
 *                             single-block route_count, 2 = route_local +
 *                             route_finalize, 3 = route_cluster (MOE_EINVAL
 *                             if the device cannot schedule it), 4 =
 *                             route_pack: moe_dispatch_send routes and packs
 *                             in one kernel, every CTA of the pack grid
 *                             computing the routing tables itself (bulk
 *                             copies, static split; MOE_EINVAL unless
 *                             T*K <= 16384 and E*ceil(T/32) <= 4096), and
 *                             moe_dispatch_send_fp8 routes and quantises in
 *                             one kernel, route_pack_fp8 (automatic too for
 *                             those layers with MOE_OPT_FP8_ORDER 1 and no
 *                             forced pack queue); the other dispatch calls
 *                             route as with 0 */
#define MOE_OPT_PACK_VARIANT 1
#define MOE_OPT_PACK_STAGES 2
#define MOE_OPT_PACK_PIECE_BYTES 3
#define MOE_OPT_PACK_CTAS_PER_SM 4
#define MOE_OPT_PDL 5
#define MOE_OPT_ROUTE_VARIANT 6
int moe_ctx_set_option(moe_ctx* ctx, int option, int64_t value);

/* Reads back a launch option.  For MOE_OPT_ROUTE_VARIANT set to 0
 * (automatic) it reports the path moe_dispatch_send will take (2, 3 or 4);
 * MOE_OPT_ROUTE_CLUSTER_CTAS reports the route_cluster cluster size chosen
 * for this configuration (0 if the device cannot schedule it);
 * MOE_OPT_ROUTE_VARIANT_FP8 (read only) the routing of
 * moe_dispatch_send_fp8 in the same numbering (4: route_pack_fp8). */
#define MOE_OPT_ROUTE_CLUSTER_CTAS 7
#define MOE_OPT_ROUTE_VARIANT_FP8 22
/*   MOE_OPT_COMBINE_VARIANT     0 = a producer warp gathers the K expert-row
 *                               pieces with bulk copies into shared-memory
 *                               stages, consumer warps reduce; 1 = one thread
 *                               per 16-byte chunk, direct loads; -1 = automatic
 *                               (default: 0 for K >= 4, else 1)
 *   MOE_OPT_COMBINE_STAGES      bulk: stages per CTA, 2..8, 0 = automatic
 *   MOE_OPT_COMBINE_PIECE_BYTES bulk: bytes of a row per unit, 0 = automatic
 *                               (equal pieces of at most 4 KiB, or 2 KiB with
 *                               MOE_OPT_COMBINE_ORDER 0)
 *   MOE_OPT_COMBINE_CTAS_PER_SM bulk: 0 = as many as fit, else 1..32 */
#define MOE_OPT_COMBINE_VARIANT 8
#define MOE_OPT_COMBINE_STAGES 9
#define MOE_OPT_COMBINE_PIECE_BYTES 10
#define MOE_OPT_COMBINE_CTAS_PER_SM 11
/*   MOE_OPT_PACK_PREFETCH       bulk pack: while routing runs, each CTA
 *                               prefetches its later token rows into L2:
 *                               2 = with an evict-last policy when all of them
 *                               fit in a third of L2, else as 1 (default); each
 *                               row goes back to normal priority once loaded;
 *                               1 = all of them with normal priority; 0 = off */
#define MOE_OPT_PACK_PREFETCH 12
/*   MOE_OPT_CACHE_HINTS         bit flags, L2 evict-first policy on: 1 = pack
 *                               loads, 2 = pack stores, 4 = combine loads
 *                               (default 7: all streamed data) */
#define MOE_OPT_CACHE_HINTS 13
/*   MOE_OPT_PACK_STORE_DEPTH    bulk pack: store groups left in flight before a
 *                               stage is refilled, 1..8 (0 = automatic:
 *                               2, or 1 when a pack writes more than 1 GiB) */
#define MOE_OPT_PACK_STORE_DEPTH 14
/*   MOE_OPT_MAX_SMS             sizes the persistent pack and combine grids
 *                               (bulk and fp8 pack, bulk combine) for this
 *                               many SMs instead of all of them (CTAs = SMs
 *                               x CTAs per SM), so that they hold only that
 *                               share of the GPU's shared memory and warps
 *                               and work the caller runs on another stream
 *                               can be resident at the same time; 0 = all
 *                               (default), else 1..SM count.  The flat
 *                               vector kernels and the two-level combine are
 *                               not bounded by it. */
#define MOE_OPT_MAX_SMS 15
/*   MOE_OPT_TEST_DROP_COMBINE_UNIT  failure-injection hook for tests, -1 = off
 *                               (default).  With a unit index u >= 0 (token
 *                               u / pieces, piece u % pieces), the bulk
 *                               combine's producer never posts unit u, so the
 *                               consumers' bounded wait (2 s) runs out: the
 *                               combine writes nothing for the rest of that
 *                               CTA's units, reports MOE_ETIMEDOUT in the error
 *                               word and returns; the context stays usable
 *                               (the next dispatch resets the error word).
 *                               Only the bulk combine variant honours it. */
#define MOE_OPT_TEST_DROP_COMBINE_UNIT 16
/*   MOE_OPT_COMBINE_ORDER       bulk combine: which tokens a CTA takes; 0 = one
 *                               contiguous range of (token, piece) units (and
 *                               automatic pieces of up to 2 KiB); 1 or -1
 *                               (default) = tokens b, b+G, b+2G, ... of G CTAs
 *                               for the T/G full rounds, the leftover tokens'
 *                               units split evenly, so that the gathered rows
 *                               being read at any moment lie close together in
 *                               each expert's region (automatic pieces of up
 *                               to 4 KiB) */
#define MOE_OPT_COMBINE_ORDER 17
/*   MOE_OPT_FP8_ORDER           fp8 pack: which tokens a CTA takes; 0 = one
 *                               contiguous range, 1 = tokens b, b+G, b+2G, ...
 *                               of G CTAs (default: their destination rows lie
 *                               close together in each expert's region) */
#define MOE_OPT_FP8_ORDER 18
/*   MOE_OPT_KERNEL_EVENTS       1 = record CUDA events on the caller's stream
 *                               right before and after the pack kernel of
 *                               moe_dispatch_send / moe_dispatch_send_fp8 and
 *                               the combine kernel of moe_combine_recv, for
 *                               moe_kernel_times (diagnostics: the events keep
 *                               those kernels from overlapping the kernel
 *                               before them); 0 = off (default) */
#define MOE_OPT_KERNEL_EVENTS 19
/*   MOE_OPT_PACK_SCHEDULE       bulk pack of moe_dispatch_send and of the
 *                               first stage of the staged and quantised
 *                               dispatches, and (with MOE_OPT_FP8_ORDER 1,
 *                               tokens as units) the pack of
 *                               moe_dispatch_send_fp8: 0 = static (CTA b copies units b,
 *                               b+G, b+2G, ... of the G CTAs); 1 = unit queue
 *                               (each CTA takes its first `stages` units
 *                               statically, then claims units in increasing
 *                               order from a counter in the workspace that the
 *                               routing kernel resets, so faster CTAs take
 *                               more); -1 = automatic (default: the queue when
 *                               a CTA has more than 1.5x its first `stages`
 *                               units, 3x for the fp8 pack).  Results are
 *                               identical. */
#define MOE_OPT_PACK_SCHEDULE 20
/*   MOE_OPT_COMBINE_SCHEDULE    bulk combine of moe_combine_recv: 0 = the
 *                               static order of MOE_OPT_COMBINE_ORDER; 1 =
 *                               token queue (CTA b combines token b, then
 *                               claims tokens in increasing order from a
 *                               counter in the workspace that the routing
 *                               kernel resets, all pieces of a claimed token
 *                               in turn); -1 = automatic (default: the queue).
 *                               Results are identical. */
#define MOE_OPT_COMBINE_SCHEDULE 21
int moe_ctx_get_option(const moe_ctx* ctx, int option, int64_t* value);

/* Durations, in milliseconds, of the pack kernel of the context's last
 * dispatch and of the combine kernel of its last combine.  Each is -1 unless
 * that call was moe_dispatch_send / moe_dispatch_send_fp8 (pack) or
 * moe_combine_recv (combine) made with MOE_OPT_KERNEL_EVENTS on; the
 * staged, quantised and two-level variants are not timed.  Waits for the
 * events to complete.  MOE_EINVAL for null pointers, MOE_ECUDA if an event
 * query fails. */
int moe_kernel_times(moe_ctx* ctx, float* pack_ms, float* combine_ms);

/* ---- Dispatch without any device allocation ------------------------------
 * The pages have no counterpart to this call; it exists for callers that
 * cannot call cudaMalloc (code running inside another framework's memory
 * pool without an allocator handle, allocation-free runtime sections,
 * processes that may not grow their device footprint after start-up), so
 * they cannot provide the workspace that moe_ctx_create needs.
 *
 * Gives the same results as moe_dispatch_send (the same grouped rows, counts
 * and offsets) but routes with the single-block route_count kernel (slower
 * than moe_dispatch_send's default routing on large layers) and packs with
 * the bulk pack's static split; it keeps the routing tables in one fixed
 * static device array inside the library (MOE_NOALLOC_SCRATCH_BYTES, held by
 * every GPU that loads libmoe.so until the process exits) and allocates
 * nothing.
 *   x, topk_idx, expert_x, expert_x_rows  as for moe_dispatch_send
 *   expert_counts   device int32 [E], written
 *   expert_offsets  device int32 [E+1], written
 *   status          device int32 [1], written: MOE_OK or the device-detected
 *                   status (MOE_EROUTE, MOE_EBOUND, MOE_ETIMEDOUT)
 * Returns MOE_EINVAL, before enqueuing anything, when T*K exceeds
 * MOE_NOALLOC_MAX_PAIRS or E*N exceeds MOE_NOALLOC_MAX_EXPERT_RANKS, or for
 * the argument errors of moe_dispatch_send; MOE_ECUDA on a CUDA failure.
 * The first call on a device (with that device current) looks up the static
 * array's device address and sets kernel attributes; make that first call
 * before any stream capture.  All calls share the array: calls whose kernels
 * may overlap on the GPU (unordered streams, several host threads) race.
 * No context is involved; there is no combine counterpart. */
#define MOE_NOALLOC_MAX_PAIRS 262144
#define MOE_NOALLOC_MAX_EXPERT_RANKS 65536
#define MOE_NOALLOC_SCRATCH_BYTES 2363648
int moe_dispatch_send_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx, void* expert_x,
                              int64_t expert_x_rows, int32_t* expert_counts, int32_t* expert_offsets,
                              int32_t* status, void* stream);

/* Synchronises `stream` and returns the device status of the last dispatch
 * (MOE_OK, MOE_EROUTE, MOE_EBOUND or MOE_ETIMEDOUT), or MOE_ECUDA. */
int moe_get_error(moe_ctx* ctx, void* stream);

/* Static description of a status code. */
const char* moe_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
