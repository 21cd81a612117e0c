/*
 * attn_decode.h -- C ABI of the GB300 split-K flash-decoding library
 * (libattn.so).
 *
 * Scope: single- and few-token attention of query rows against a KV cache
 * on one GPU.  The key dimension is split into partitions (with more than
 * one partition every block takes one contiguous key range and leaves its
 * exponential sum and running maximum for a separate reduce pass,
 * mha_decoding_single_batch_pipelined, summary); the partials are merged by
 * a log-sum-exp reduce.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers marked "device" are CUDA device (or managed) memory of the
 *   current device.  The caller owns every buffer.  The library never
 *   allocates device memory, never synchronises, and enqueues all work on
 *   the given stream (NULL = legacy default stream).  Calls are
 *   asynchronous: device-side results are ready once the stream reaches
 *   them.
 * - Arguments are validated on the host before anything is launched.  A
 *   failed check returns a status and launches nothing.  A failed launch
 *   returns ATTN_ERR_CUDA (the CUDA error is left for cudaGetLastError).
 * - bf16 for q, K, V and out; fp32 for scale, sink logits, lse and the
 *   split-K workspace.  All element strides are in elements.
 * - lse is the natural-log log-sum-exp of the scaled scores, sink
 *   included; it is -inf for a row with no visible key and no sink (its
 *   output row is then 0).
 * - Query head h reads KV head h / group (groups of consecutive query
 *   heads share one KV head; group is the GQA group size, the count of
 *   query heads per KV head, mha_sm100_dispatch, Parameters).
 * - The number of partitions comes only from host integers, never from
 *   device data, so a call can be captured in a CUDA graph and replayed
 *   while the per-sequence lengths change (capture-invariant partition
 *   ceiling, mha_sm100_dispatch, Args: num_partitions_override).
 */
#ifndef ATTN_DECODE_H
#define ATTN_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *attn_stream_t; /* identical to cudaStream_t */

enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* null pointer, bad size, inconsistent shape */
    ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head dim, page size, ...) */
    ATTN_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small */
    ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call failed */
    ATTN_ERR_DEVICE = 5        /* a kernel reported a device-side error flag */
};

/* Largest split-K partition count accepted by every entry point. */
#define ATTN_MAX_PARTITIONS 1024
/* attn_plan_partitions request: the balanced split (MLA: num_partitions 0;
 * attn_decode on the tensor cores: num_partitions ATTN_PARTITIONS_BALANCED) */
#define ATTN_PARTITIONS_BALANCED (-1)
/* attn_plan_partitions request and attn_decode num_partitions on the tile
 * path: two Q tiles per CTA pair sharing each K/V tile */
#define ATTN_PARTITIONS_TILE_PAIR (-2)

/*
 * One K or V cache operand (the KV operand type carries the element type and
 * the page size, mha_sm100_dispatch, Parameters: KVType; paged KVCache operand
 * or contiguous tensor operand, flare_mla_decoding_dispatch, Parameters: k_t).
 *
 * Token t of sequence b, KV head kh, channel c is the bf16 element
 *   base[page * page_stride + (t % page_size) * token_stride
 *        + kh * head_stride + c]
 * with page = page_table[b * max_pages + t / page_size] when page_table is
 * non-NULL (paged cache) and page = b when it is NULL (contiguous cache,
 * one "page" of page_size >= every kv_len per sequence).
 *
 * Requirements: base 16-byte aligned; channels contiguous; page_stride,
 * token_stride and head_stride multiples of 8 elements (16 bytes);
 * num_pages = number of pages in the pool (= batch for a contiguous
 * cache).  For a paged cache page_size must be a power of two >= 8.  Page
 * table entries must lie in [0, num_pages); entries are read only for
 * pages that hold tokens < kv_len[b].
 */
typedef struct attn_kv {
    const void *base;          /* device, bf16 */
    int64_t page_stride;
    int64_t token_stride;
    int64_t head_stride;
    int32_t page_size;
    int32_t num_pages;
    const int32_t *page_table; /* device int32 [batch][max_pages], or NULL */
    int32_t max_pages;         /* row length of page_table */
    int32_t reserved;          /* must be 0 */
} attn_kv_t;

/*
 * attn_plan_partitions -- choose the split-K partition count.
 *
 * Follows the automatic partition ladder with an exact override
 * (a non-zero num_partitions_override is used as given and zero selects the
 * automatic ladder, mha_sm100_dispatch, Args; an absent num_partitions lets
 * a heuristic choose, flare_mla_decoding_dispatch, Args).
 *
 *   num_sms       SMs to plan for; <= 0 queries the current device.
 *   batch         sequences; num_q_rows total query rows (= batch for
 *                 single-token decode).
 *   max_q_len     host upper bound of the query rows of any sequence (1 for
 *                 single-token decode), as attn_decode takes it.  It picks
 *                 the GQA kernel exactly as attn_decode does: a few rows
 *                 (head_dim_v 128, max_q_len * group <= 16, batch <= 2048)
 *                 fold onto the split-K decode kernel; longer row runs take
 *                 the tile kernels, which do not split: the plan is P = 1
 *                 (one Q tile per CTA, for requests 0 and 1) or, for the
 *                 request ATTN_PARTITIONS_TILE_PAIR, that value (two Q tiles
 *                 per CTA pair), with workspace 0; a request above 1 returns
 *                 ATTN_ERR_UNSUPPORTED.  MLA ignores it.
 *   num_q_heads, num_kv_heads   heads (num_kv_heads = 1 for MLA).
 *   head_dim_v    output channels (128 for GQA d128, 512 for MLA).
 *   max_kv_len    host upper bound of every kv_len[b].
 *   requested     0 = automatic; > 0 = use exactly this many partitions;
 *                 ATTN_PARTITIONS_BALANCED = the balanced split (MLA shapes:
 *                 num_kv_heads 1, head_dim_v 512, num_partitions out 0; or
 *                 attn_decode with head_dim 128 on its split-K route, single
 *                 rows or the few-row fold, num_partitions out
 *                 ATTN_PARTITIONS_BALANCED);
 *                 ATTN_PARTITIONS_TILE_PAIR = two Q tiles per CTA pair (the
 *                 tile path only); any other shape or negative value:
 *                 ATTN_ERR_INVALID_ARG.
 *   num_partitions  out: partitions P (1 <= P <= ATTN_MAX_PARTITIONS), 0 for
 *                 the balanced MLA split, ATTN_PARTITIONS_BALANCED for the
 *                 balanced GQA split, or ATTN_PARTITIONS_TILE_PAIR.
 *   workspace_bytes out: workspace size attn_decode / attn_mla_decode need
 *                 for this P (0 when P == 1).
 *
 * Key slice p of a sequence is [p*C, min((p+1)*C, kv_len)) with
 * C = ceil(ceil(max_kv_len / P) / T) * T, T = 128 for attn_decode with
 * head_dim 128, 32 for head_dim 64, and 64 for attn_mla_decode; slices past
 * kv_len are empty.  With head_dim 128, P = 2 or 4 needs no workspace
 * (workspace_bytes 0): a cluster of P CTAs splits each (sequence, KV head)
 * into P equal key slices of that sequence and merges them on chip.  The
 * automatic choice treats num_kv_heads == 1 with head_dim_v == 512 as the
 * MLA shape and everything else as GQA.  GQA with head_dim 128 on the
 * split-K route and at most 8 num_sms (sequence, KV head) units (max_kv_len
 * above one 128-key tile) takes the balanced split: the 128-key
 * tiles of every unit (an empty unit counts one), concatenated, are dealt
 * out in contiguous ranges of equal cost (tiles plus 2 tiles' worth for
 * every unit a range opens) to num_sms CTAs; a unit a range end cuts
 * leaves one partial per piece, merged by the reduce.  Its workspace_bytes
 * = (num_sms + units) slots of 16 x 128 fp32 plus 16 m and 16 l each (each
 * array 256-byte aligned) plus 8 bytes per unit (256-byte aligned).  GQA with head_dim 128 and
 * max_q_len > 1 on the few-row fold: P = 1 when there are at
 * least 2 (sequence, KV head) units per SM, else the many-unit rule (at
 * least four items per CTA at full length and slices of at most ~1024
 * keys) whatever the unit count.  MLA: with
 * P' = max(floor(num_sms / 2 / num_q_rows), ceil(max_kv_len / (4096 n))),
 * n = ceil(num_q_rows / batch) query rows per sequence, capped at
 * ceil(max_kv_len / 64), the plan is P = 1 (no split) when P' <= 1 and
 * otherwise P = 0, the balanced split: the 64-key tiles of every query row,
 * concatenated, are dealt out in contiguous ranges of equal cost (tiles
 * plus 8 tiles' worth for every row a range opens) to min(num_sms / 2,
 * tiles) two-CTA clusters (one wave), with workspace_bytes = (num_sms / 2 +
 * num_q_rows) slots of fp32 partials (128 x 512 O, m, l, each array
 * 256-byte aligned) plus 8 num_q_rows bytes (256-byte aligned) for the
 * table of where each row's partials are; it does not depend on max_kv_len.
 * For attn_mla_decode_sparse pass max_kv_len = indices_stride.
 * Returns ATTN_OK, ATTN_ERR_INVALID_ARG, or ATTN_ERR_CUDA if the SM count
 * query fails.  Launches nothing.
 */
int attn_plan_partitions(int num_sms, int batch, int num_q_rows, int max_q_len,
                         int num_q_heads, int num_kv_heads, int head_dim_v, int max_kv_len,
                         int requested, int *num_partitions, size_t *workspace_bytes);

/*
 * attn_decode -- GQA/MHA attention of few query rows per sequence against a
 * paged or contiguous cache, with split-K for single- and few-token decode
 * (mha_decoding_single_batch_pipelined; mha_sm100_dispatch).
 *
 *   q          device bf16 [num_q_rows][num_q_heads][head_dim]
 *              (q_arg, mha_decoding_single_batch_pipelined, Args).
 *   k, v       cache operands (host structs describing device memory); both
 *              head_dim wide and sharing one page table layout.
 *   kv_len     device uint32 [batch]: keys of sequence b, including its own
 *              query tokens (valid_length, the per-row count of valid
 *              keys, mha_sm100_dispatch, Args).  The cache already holds the
 *              current tokens' K/V.
 *   q_row_offsets  device uint32 [batch + 1] (rows of sequence b are
 *              [off[b], off[b+1])), or NULL for one row per sequence.
 *   batch, num_q_rows   sequences and total query rows (num_q_rows = batch
 *              when q_row_offsets is NULL; otherwise = off[batch]).  The
 *              split-K decode kernel accepts batch <= 2048.
 *   num_q_heads, group  num_q_heads % group == 0; group in {1, 2, 4, 8}.
 *   head_dim   64 or 128 (128 when max_q_len > 1).
 *   max_q_len  host upper bound of the rows of any sequence (max_prompt_len,
 *              mha_sm100_dispatch, Args); no sequence may have more rows.
 *              1 selects the split-K decode kernel.  A few rows (head_dim
 *              128, max_q_len * group <= 16, batch <= 2048: e.g. draft
 *              tokens being verified) stay on that kernel: the rows of a
 *              sequence fold onto the tensor-core N side next to the group's
 *              heads and share every K/V tile, split-K included.  More rows
 *              select the tensor-core tile path, which takes every sequence
 *              of the batch, single-token ones included (that page handles
 *              one-token decode as the degenerate case of prefill rather
 *              than a route of its own, mha_sm100_dispatch, summary), and does
 *              not split: one 128-row Q tile per CTA, or two adjacent Q tiles
 *              per CTA pair sharing each K/V tile through the pair's MMA (the
 *              1Q and 2Q configurations that page chooses between).
 *   max_kv_len host upper bound of kv_len ("max_cache_valid_length_arg").
 *   scale      multiplies Q.K' before the softmax.
 *   sink       device fp32 [num_q_heads] attention-sink logits, or NULL.
 *              A sink adds exp(sink[h]) to the softmax normaliser of head h
 *              and carries no value; it is not multiplied by scale.
 *   causal     non-zero: row i of a sequence with n rows and L keys sees
 *              keys j <= L - n + i (bottom-right aligned).  A no-op for
 *              single-row sequences.
 *   num_partitions  P from attn_plan_partitions (or any 1..MAX), or 0 for
 *              the planner's automatic choice on the current device (the
 *              same call as attn_plan_partitions with num_sms 0 and
 *              requested 0: size the workspace with that call), or
 *              ATTN_PARTITIONS_BALANCED (head_dim 128, not the tile path):
 *              the balanced split over one CTA per SM of the current device,
 *              the workspace sized for it; must be 0 or
 *              1 on the tile path (max_q_len > 1 beyond the few-row fold),
 *              both one Q tile per CTA, or ATTN_PARTITIONS_TILE_PAIR there:
 *              two adjacent Q tiles per CTA pair.  The automatic choice (0)
 *              is one tile per CTA, measured faster than the pair on every
 *              shape tried; the pages choose between the two by occupancy
 *              and prompt length and make a non-zero override force the
 *              smaller tile (mha_sm100_dispatch, summary and Args:
 *              num_partitions_override).
 *   workspace  device, 256-byte aligned, >= the planner's workspace_bytes
 *              for this P; may be NULL when P == 1, and with head_dim 128
 *              when P is 2 or 4 (those merge on chip).  Contents on entry
 *              are ignored; it holds fp32 partial O, qk_max and exp_sum
 *              after.
 *   out        device bf16 [num_q_rows][num_q_heads][head_dim].
 *   lse        device fp32 [num_q_rows][num_q_heads], or NULL.
 *
 * Decode launches the partition kernel (a persistent grid over (sequence,
 * KV head, key slice) items) and, for P > 1, the split-K reduce.  Returns
 * ATTN_OK or an error status.
 */
int attn_decode(const void *q, const attn_kv_t *k, const attn_kv_t *v, const uint32_t *kv_len,
                const uint32_t *q_row_offsets, int batch, int num_q_rows, int num_q_heads,
                int group, int head_dim, int max_q_len, int max_kv_len, float scale,
                const float *sink, int causal, int num_partitions, void *workspace,
                size_t workspace_bytes, void *out, float *lse, attn_stream_t stream);

/*
 * attn_mla_decode -- multi-head latent attention decode: one KV head whose
 * rows are dim_qk = 576 wide (512 latent + 64 rope), V = K[:, :dim_v]
 * with dim_v = 512 (MLA has exactly one KV head, and V is the leading
 * depth_v channels of K rather than a second operand that is read,
 * flare_mla_decoding_dispatch, Parameters: kv_num_heads and Args: k).
 *
 *   q          device bf16 [batch][num_q_heads][dim_qk]; num_q_heads = 128.
 *   kv         the single cache operand (num_kv_heads = 1).
 *   kv_len, max_kv_len, scale, sink, workspace_bytes, lse
 *              as for attn_decode.
 *   num_partitions  0 (the balanced split) or 1..MAX (P key slices per row),
 *              from attn_plan_partitions or chosen.
 *   workspace  as for attn_decode, sized by attn_plan_partitions for this P;
 *              needed unless P == 1.
 *   out        device bf16 [batch][num_q_heads][dim_v].
 *
 * P >= 1: one two-CTA cluster per (key slice, row); slice p of a row is
 * [p C, (p+1) C) as attn_plan_partitions states, then the split-K reduce.
 * P == 0: the decode grid (one wave of clusters) finds each cluster's tile
 * range from kv_len and walks it, a cluster writing the final rows of the
 * rows its range holds whole and fp32 partials of the rows a range end
 * cuts, and the entry of the workspace table saying where the partials of
 * each row whose first tile it holds are; the reduce merges them (two
 * launches).  kv_len above max_kv_len is then clamped to it and sets error
 * bit 2, as a length above P C does for P >= 1.
 */
int attn_mla_decode(const void *q, const attn_kv_t *kv, const uint32_t *kv_len, int batch,
                    int num_q_heads, int dim_qk, int dim_v, int max_kv_len, float scale,
                    const float *sink, int num_partitions, void *workspace,
                    size_t workspace_bytes, void *out, float *lse, attn_stream_t stream);

/*
 * attn_mla_decode_rows -- MLA decode of several query rows per sequence, for
 * draft tokens being verified (the multi-token-prediction rows that
 * max_prompt_len bounds, flare_mla_decoding_dispatch, Args).
 *
 *   q          device bf16 [num_q_rows][num_q_heads][dim_qk] (128, 576).
 *   kv, kv_len, max_kv_len, scale, sink, num_partitions, workspace,
 *   workspace_bytes   as for attn_mla_decode; kv_len counts every key of the
 *              sequence, its own query tokens included.
 *   q_row_offsets  device uint32 [batch + 1]: rows of sequence b are
 *              [off[b], off[b+1]); num_q_rows = off[batch].  Required.
 *   causal     nonzero: row i of a sequence with n rows and L keys sees keys
 *              j <= L - n + i (the rows are the last n tokens); zero: every
 *              row sees all L keys.
 *   out, lse   device bf16 [num_q_rows][num_q_heads][dim_v] / fp32
 *              [num_q_rows][num_q_heads] (lse may be NULL).
 *
 * P and the workspace come from attn_plan_partitions with num_q_rows rows.
 * P >= 1: every row of a sequence runs over the same key slices, one
 * two-CTA cluster per (slice, row), and clusters of the rows of a sequence
 * are launched next to each other so the second and later reads of a key
 * tile are served from L2.  P == 0: the balanced split over all rows' tiles
 * (each row with its own causal length) as for attn_mla_decode.
 * num_q_rows <= 65535.  Returns as attn_mla_decode.
 */
int attn_mla_decode_rows(const void *q, const attn_kv_t *kv, const uint32_t *kv_len,
                         const uint32_t *q_row_offsets, int batch, int num_q_rows,
                         int num_q_heads, int dim_qk, int dim_v, int max_kv_len, float scale,
                         const float *sink, int causal, int num_partitions, void *workspace,
                         size_t workspace_bytes, void *out, float *lse, attn_stream_t stream);

/*
 * attn_mla_decode_sparse -- MLA decode in which every sequence attends only
 * to the cache rows that a top-k index list names (flare_mla_decoding_dispatch,
 * Parameters: sparse; Args: d_indices, indices_stride, topk_lengths).
 *
 *   q          device bf16 [batch][num_q_heads][dim_qk]; num_q_heads = 128,
 *              dim_qk = 576, dim_v = 512 as for attn_mla_decode.
 *   kv         the cache read as num_pages * page_size rows at one stride:
 *              row r is slot r % page_size of page r / page_size, and
 *              page_stride must equal page_size * token_stride (a contiguous
 *              pool; otherwise ATTN_ERR_UNSUPPORTED).  page_table must be
 *              NULL (the indices take its place); any page_size >= 1; the
 *              other requirements of attn_kv_t hold.
 *   indices    device int32 [batch][indices_stride]: key t of sequence b is
 *              row indices[b * indices_stride + t].  Entries at t >=
 *              topk_lengths[b] are never read.  A row may appear more than
 *              once (it then counts once per appearance).  May be NULL when
 *              indices_stride is 0.
 *   indices_stride  row length of indices (the largest top-k of the batch);
 *              it plays the part of max_kv_len for partition planning
 *              (attn_plan_partitions with num_kv_heads 1, head_dim_v 512,
 *              max_kv_len = indices_stride gives num_partitions and the
 *              workspace size).
 *   topk_lengths  device int32 [batch]: valid keys of sequence b,
 *              0 <= topk_lengths[b] <= indices_stride.  0 gives out = 0 and
 *              lse = -inf (or the sink alone).
 *   scale, sink, num_partitions, workspace, workspace_bytes, out, lse
 *              as for attn_mla_decode.  extra_k (an always-attended second
 *              cache) is not supported.
 *
 * An index outside [0, num_pages * page_size) sets bit 1 of the device
 * error word and that key is not read.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE or ATTN_ERR_CUDA; launches nothing
 * on an error return.
 */
int attn_mla_decode_sparse(const void *q, const attn_kv_t *kv, const int32_t *indices,
                           int indices_stride, const int32_t *topk_lengths, int batch,
                           int num_q_heads, int dim_qk, int dim_v, float scale,
                           const float *sink, int num_partitions, void *workspace,
                           size_t workspace_bytes, void *out, float *lse,
                           attn_stream_t stream);

/*
 * attn_splitk_reduce -- merge split-K partials by log-sum-exp
 * (mha_splitk_reduce / mla_splitk_reduce, named in
 * mha_decoding_single_batch_pipelined, summary, and
 * flare_mla_decoding_dispatch, summary).
 *
 * For each row r and head h, with m_p = ws_m[p][r][h], l_p = ws_l[p][r][h],
 * O_p = ws_o[p][r][h][:], t = sink[h] (or -inf):
 *   M = max(max_p m_p, t);  w_p = exp(m_p - M)  (0 when m_p = -inf)
 *   Z = sum_p w_p l_p + exp(t - M)
 *   out[r][h][:] = sum_p w_p O_p / Z   (bf16, 0 when Z = 0)
 *   lse[r][h] = M + ln Z               (-inf when Z = 0)
 *
 *   ws_o       device fp32 [num_partitions][rows][num_q_heads][dim_v]
 *              (unnormalised partial outputs).
 *   ws_m, ws_l device fp32 [num_partitions][rows][num_q_heads]: partial
 *              max score (natural-log units, -inf for an empty partition)
 *              and partial exp-sum relative to it.
 *   dim_v      a multiple of 4, <= 1024.
 *   sink       device fp32 [num_q_heads] or NULL.
 *   out        device bf16 [rows][num_q_heads][dim_v]; lse device fp32
 *              [rows][num_q_heads] or NULL.
 */
int attn_splitk_reduce(const float *ws_o, const float *ws_m, const float *ws_l,
                       int num_partitions, int rows, int num_q_heads, int dim_v,
                       const float *sink, void *out, float *lse, attn_stream_t stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device
 * memory: an engine plugin bound to a memory plan fixed at start-up, or a
 * plain C program with no allocator at hand.  The source pages have no
 * counterpart; it exists only because split-K needs scratch space.
 *
 * Arguments are those of attn_decode without workspace / workspace_bytes.
 * The call is routed and planned by attn_plan_partitions, exactly as
 * attn_decode routes it: num_partitions 0 plans automatically, a non-zero
 * count is used as given (single rows and the few-row fold split K with it;
 * the tile kernel for longer row runs does not split and rejects a count
 * above 1 with ATTN_ERR_UNSUPPORTED).  The split-K scratch is a fixed 32 MiB
 * array inside the library (a file-scope device array that every GPU loading
 * the library keeps until the process exits); a partition count whose
 * workspace would exceed it returns ATTN_ERR_WORKSPACE and launches nothing.
 * The call itself allocates nothing (no cudaMalloc/cudaFree, no allocating
 * library routine).
 *
 * Every call looks up the array's device address (cudaGetSymbolAddress,
 * with the call's device current), so the address stays right after a
 * device reset; the first call on a device may load the library's device
 * code, so make it before any stream capture.  Every call shares the one
 * array and leaves its partials there: calls that can overlap on the GPU
 * (other streams, other host threads) race on it and must be serialised by
 * the caller.  Nothing in it needs to start at zero.
 */
int attn_decode_noalloc(const void *q, const attn_kv_t *k, const attn_kv_t *v,
                        const uint32_t *kv_len, const uint32_t *q_row_offsets, int batch,
                        int num_q_rows, int num_q_heads, int group, int head_dim, int max_q_len,
                        int max_kv_len, float scale, const float *sink, int causal,
                        int num_partitions, void *out, float *lse, attn_stream_t stream);

/*
 * attn_device_error_flags -- read (and optionally clear) the device-side
 * error word that kernels set instead of hanging: bit 0 = a pipeline wait
 * ran past its time limit (250 ms), bit 1 = a page-table entry outside
 * [0, num_pages) or a sparse index outside [0, num_pages * page_size) was
 * seen (that page or row was not read; the output is then undefined),
 * bit 2 = a kv_len above num_partitions x slice length, or a top-k count
 * above indices_stride or below 0, was seen (it was clamped).  Synchronises
 * the current device.  Returns ATTN_OK or ATTN_ERR_CUDA.
 */
int attn_device_error_flags(unsigned int *flags, int clear);

/*
 * attn_selftest_wait_timeout -- the pages have no counterpart: a check of
 * the failure path for deployments (and this library's tests).  Launches one
 * kernel that waits, with the kernels' own bounded mbarrier wait, on a
 * barrier nothing arrives on; after the time limit the wait gives up, sets
 * bit 0 of the error word and the kernel returns, leaving the context
 * usable.  Asynchronous on `stream`; read the result with
 * attn_device_error_flags.  Returns ATTN_OK or ATTN_ERR_CUDA.
 */
int attn_selftest_wait_timeout(attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_DECODE_H */
