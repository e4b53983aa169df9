/*
 * sai.h -- C ABI of libsai, the GB300 (sm_103a) sparse-attention indexer
 * decode path: FP8 paged MQA logits, then per-row top-k.
 *
 * Source of the operations.  The logits op and its arguments are those of
 * `deepgemm_fp8_paged_mqa_logits(q_fp8, kv_cache, weights, out_logits,
 * context_lens, block_tables, max_model_len, ...)` as called by the
 * reproducer of aiter PR 4244 ("fix silent tail-row drop in
 * deepgemm_fp8_paged_mqa_logits at large output stride", section "small
 * reproducer"); the top-k is `top_k_per_row_decode`, which the same page's
 * opening paragraph runs right after the logits launch to fill the
 * persistent sparse-KV index buffer.  The scoring rule is the DeepSeek-style
 * indexer definition
 *
 *     logits[r, t] = sum_h w[r, h] * ReLU(q[r, h] . k[t]) * scale[t]   (t < ctx_r)
 *     logits[r, t] = -inf                                              (ctx_r <= t < W)
 *
 * with query row r = b * next_n + j and ctx_r = ctx_b - next_n + j + 1 (MTP
 * row j sees one token more than row j - 1).
 *
 * Conventions for every call:
 *   - Pointers marked "device" must be device memory (or managed memory) of
 *     the current device.  Nothing is read from or written to host memory.
 *   - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *     never synchronise.  They allocate nothing.  State kept across calls,
 *     per process: each device's SM count; up to 32 encoded TMA tensor maps,
 *     keyed by device, buffer address, extent and box (a hit is always valid
 *     for the buffer it names); per kernel and device, a flag that its
 *     shared-memory size attribute has been raised; and the static request
 *     counters of sai_paged_mqa_logits_topk_static (a device array).
 *   - The caller owns every buffer.  The library keeps no pointer after the
 *     call returns (kernels still in flight use them until they finish).
 *   - Return value: SAI_OK (0), or a negative SAI_ERR_* code.  On any error
 *     nothing is launched and no output is touched.
 *   - Problems only the device can see (a page id outside the pool, a
 *     context longer than the output or the block table, a pipeline wait that
 *     ran out of time) never trap: they set bits in the optional device status
 *     word (SAI_STATUS_*), which the library only ORs into and never clears.
 *   - All byte offsets are formed in 64 bits: row bases are
 *     int64(row) * stride, page bases int64(page_id) * page_bytes, so outputs
 *     past 2^31 bytes and KV pages past 2^31 bytes are addressed correctly
 *     (aiter PR 4244, section "Fix"; ATOM PR 2533, "[MLA] Address Triton
 *     decode KV rows with int64 ids").
 */
#ifndef SAI_H_
#define SAI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SAI_API __attribute__((visibility("default")))
#else
#define SAI_API
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
typedef struct CUstream_st* sai_stream_t;

/* Return codes. */
#define SAI_OK                    0
#define SAI_ERR_INVALID_ARGUMENT (-1)  /* null pointer, negative size, stride < width, ... */
#define SAI_ERR_UNSUPPORTED      (-2)  /* valid but not built: head_dim != 128, page size, ... */
#define SAI_ERR_MISALIGNED       (-3)  /* a pointer lacks the alignment stated below */
#define SAI_ERR_WORKSPACE        (-4)  /* workspace missing or too small */
#define SAI_ERR_CUDA             (-5)  /* a CUDA runtime call or kernel launch failed */

/* Bits of the device status word (OR-ed in by kernels, never cleared). */
#define SAI_STATUS_BAD_PAGE     0x1u  /* a block-table entry outside [0, num_pages): its tokens' logits are NaN */
#define SAI_STATUS_CTX_CLAMPED  0x2u  /* a context_len < 0, > max_model_len or > table capacity: clamped */
#define SAI_STATUS_TIMEOUT      0x4u  /* a bounded pipeline wait expired: the outputs of that CTA are incomplete */

/* Paged K-cache byte layouts (kv_layout argument). */
#define SAI_KV_PAGE_SPLIT   0  /* page = P*D value bytes (token-major), then P fp32 scales */
#define SAI_KV_INTERLEAVED  1  /* page = P tokens of (D value bytes, then 4 scale bytes) */

/*
 * sai_paged_mqa_logits -- FP8 paged MQA logits (one launch).
 *
 *   q_fp8         device, uint8 [batch, next_n, heads, head_dim], contiguous,
 *                 OCP e4m3fn bytes.  16-byte aligned.
 *   kv_cache      device, uint8, num_pages pages of page_size * (head_dim + 4)
 *                 bytes each, page p starting at byte p * page_size * (head_dim + 4)
 *                 (the reproducer's [num_blocks, block_size, 1, head_dim + 4]
 *                 byte tensor).  Inside a page, kv_layout decides where a
 *                 token's head_dim e4m3fn values and its little-endian fp32
 *                 scale lie (SAI_KV_PAGE_SPLIT: values of all page_size tokens
 *                 first, token-major, then their page_size scales).
 *                 16-byte aligned.  Only pages the block table names for
 *                 t < ctx_r are read.
 *   num_pages     pages in the pool (>= 1; page ids are checked against it).
 *   page_size     tokens per page: 8, 16, 32, 64, 128 or 256.
 *   weights       device, fp32 [batch * next_n, heads], contiguous.  16-byte aligned.
 *   context_lens  device, int32 [batch]: tokens in each request's K-cache.
 *   block_table   device, int32 [batch, block_table_stride]: page ids of each
 *                 request, in token order (token t is in entry t / page_size).
 *                 Entries past ceil(ctx_b / page_size) are never read.
 *   block_table_stride  int32 entries between table rows (>= 1).
 *   batch         requests (>= 0; 0 launches nothing).
 *   next_n        query rows per request, 1..4 (MTP).
 *   heads         64 or 128.
 *   head_dim      must be 128.
 *   logits        device, fp32 [batch * next_n, logits_stride]: receives
 *                 columns [0, max_model_len) of every row; columns
 *                 [max_model_len, logits_stride) are never written.  4-byte aligned.
 *   logits_stride fp32 elements between rows (>= max_model_len); int64.
 *   max_model_len W, the logical logits width (>= 1).
 *   kv_layout     SAI_KV_PAGE_SPLIT or SAI_KV_INTERLEAVED.
 *   status        nullable device uint32 word; SAI_STATUS_* bits are OR-ed in.
 *   stream        stream to launch on.
 *
 * Every cell of [0, batch * next_n) x [0, W) is written on every call.  Row r
 * sees ctx_r = clamp(ctx_b - next_n + j + 1, 0, min(W, block_table_stride *
 * page_size)) tokens; the clamp raises SAI_STATUS_CTX_CLAMPED.
 */
SAI_API int sai_paged_mqa_logits(const uint8_t* q_fp8, const uint8_t* kv_cache,
                         int64_t num_pages, int32_t page_size,
                         const float* weights, const int32_t* context_lens,
                         const int32_t* block_table, int64_t block_table_stride,
                         int32_t batch, int32_t next_n, int32_t heads, int32_t head_dim,
                         float* logits, int64_t logits_stride, int64_t max_model_len,
                         int32_t kv_layout, uint32_t* status, sai_stream_t stream);

/*
 * sai_top_k_workspace_bytes -- bytes of device workspace that
 * sai_top_k_per_row_decode needs for `rows` rows of up to `max_len` columns and
 * this k.  May be 0, in which case the workspace pointer may be null.
 */
SAI_API size_t sai_top_k_workspace_bytes(int32_t rows, int64_t max_len, int32_t k);

/*
 * sai_top_k_per_row_decode -- per-row top-k of the logits (one launch).
 *
 *   logits        device, fp32 [batch * next_n, logits_stride] as written by
 *                 sai_paged_mqa_logits.  4-byte aligned.
 *   context_lens  device, int32 [batch]; row r = b * next_n + j considers
 *                 columns [0, n_r) with n_r = clamp(ctx_b - next_n + j + 1, 0,
 *                 max_model_len).
 *   k             1 .. 65536.
 *   indices       device, int32 [batch * next_n, indices_stride] (>= k): row r
 *                 receives, in entries [0, k), the column indices of its
 *                 min(k, n_r) largest logits, then -1 in every remaining entry
 *                 up to k.  If n_r <= k the indices are exactly 0 .. n_r - 1.
 *                 Of the columns tied at the k-th largest value, the lowest
 *                 are taken.  Order (deterministic): the select reads the
 *                 k-th largest key in radix digits of 8, 12 and 12 bits and
 *                 stops at the first digit whose bin it takes whole (at the
 *                 last digit the bin holds only ties); entries are the
 *                 columns above that bin, ascending, then the columns taken
 *                 from it, ascending.
 *   workspace     device, workspace_bytes >= sai_top_k_workspace_bytes(...);
 *                 may be null when that is 0.
 *
 * Every entry [0, k) of every row is written on every call (no stale indices
 * survive in a persistent index buffer: aiter PR 4244, opening paragraph).
 */
SAI_API int sai_top_k_per_row_decode(const float* logits, int64_t logits_stride,
                             const int32_t* context_lens, int32_t batch, int32_t next_n,
                             int64_t max_model_len, int32_t k,
                             int32_t* indices, int64_t indices_stride,
                             void* workspace, size_t workspace_bytes, sai_stream_t stream);

/*
 * sai_paged_mqa_logits_topk_workspace_bytes -- bytes of device workspace that
 * sai_paged_mqa_logits_topk needs for `batch` requests: 4 * (5 * batch + 4)
 * (a tile counter per request, a queue of up to four rows per request, its
 * head, tail and done count, and a counter of -inf fill units; 0 for
 * batch <= 0, which launches nothing).
 */
SAI_API size_t sai_paged_mqa_logits_topk_workspace_bytes(int32_t batch);

/*
 * sai_paged_mqa_logits_topk -- logits and their per-row top-k in one launch.
 *
 * The two ops above, fused: the same logits are written to `logits` exactly
 * as sai_paged_mqa_logits writes them, and `indices` receives what
 * sai_top_k_per_row_decode would select from them, in the same order.  The
 * arguments up to max_model_len, `status` and `stream` are those of
 * sai_paged_mqa_logits, and k, indices and indices_stride those of
 * sai_top_k_per_row_decode; only SAI_KV_PAGE_SPLIT caches are accepted.
 * Row r's top-k runs over its ctx_r columns, ctx_r clamped as for the logits
 * (to min(max_model_len, block_table_stride * page_size)).
 *
 *   workspace       device, >= sai_paged_mqa_logits_topk_workspace_bytes(batch)
 *                   bytes, 4-byte aligned, ALL ZERO before the first call.
 *                   Each call leaves it all zero again, so it is zeroed once
 *                   and reused; after a call that raised SAI_STATUS_TIMEOUT
 *                   it must be zeroed again.  Two calls in flight at once
 *                   (on different streams) must not share it.
 *
 * How the launch joins the two steps: each CTA, once its logits are stored,
 * adds the number of tiles it computed for a request to that request's
 * counter; the CTA whose addition completes the request pushes the
 * request's rows onto a queue of ready rows in the workspace.  Every CTA,
 * once its own tiles are done, takes rows from the queue and selects them
 * while its other warps write the -inf fill, whose units all CTAs take from
 * one counter in the workspace (a CTA that selects less fills more).  A CTA waiting for a queue
 * entry whose request is still being computed elsewhere waits at most
 * about one second of SM clock (SAI_STATUS_TIMEOUT, incomplete indices).
 * The launch needs every one of its CTAs resident at once: it launches one
 * CTA per SM of the device, so a context restricted to fewer SMs times out.
 */
SAI_API int sai_paged_mqa_logits_topk(const uint8_t* q_fp8, const uint8_t* kv_cache,
                              int64_t num_pages, int32_t page_size,
                              const float* weights, const int32_t* context_lens,
                              const int32_t* block_table, int64_t block_table_stride,
                              int32_t batch, int32_t next_n, int32_t heads, int32_t head_dim,
                              float* logits, int64_t logits_stride, int64_t max_model_len,
                              int32_t k, int32_t* indices, int64_t indices_stride,
                              void* workspace, size_t workspace_bytes,
                              uint32_t* status, sai_stream_t stream);

/*
 * sai_paged_mqa_logits_topk_static -- sai_paged_mqa_logits_topk without a
 * caller workspace.
 *
 * The source pages have no counterpart of this entry point.  It serves
 * callers that cannot allocate or lend device memory: an engine whose device
 * memory plan is fixed before it runs, a plugin interface that passes only a
 * kernel's inputs and outputs, a C caller with no CUDA allocator at hand.  It
 * allocates nothing either: its workspace (request counters and ready-row
 * queue) is a static device array of 5 * 16384 + 4 int32 (320 KB) inside
 * libsai.
 *
 * Arguments and results are those of sai_paged_mqa_logits_topk minus the
 * workspace.  batch > 16384 returns SAI_ERR_WORKSPACE before any CUDA call.
 *
 *   - Set-up: every call looks up the array's device address on the
 *     current device (cudaGetSymbolAddress; no pointer is kept, so a device
 *     reset between calls leaves nothing stale); a failure there returns
 *     SAI_ERR_CUDA.  The first lookup on a device loads the library's module
 *     there: make the first call, on every device used, before any stream
 *     capture begins.
 *   - Zero state: the array is zero when the library is loaded, and every
 *     call that completes leaves it zero.  After a call that raised
 *     SAI_STATUS_TIMEOUT it may hold partial counts and queue entries, and
 *     later calls of this entry point on that device may select from
 *     incomplete rows until sai_paged_mqa_logits_topk_static_reset has
 *     zeroed it.
 *   - Concurrency: all calls on one device share the array.  Two calls in
 *     flight at once (on different streams, or from different threads
 *     without ordering) race on them and give wrong indices; order such calls
 *     on one stream.
 */
SAI_API int sai_paged_mqa_logits_topk_static(const uint8_t* q_fp8, const uint8_t* kv_cache,
                              int64_t num_pages, int32_t page_size,
                              const float* weights, const int32_t* context_lens,
                              const int32_t* block_table, int64_t block_table_stride,
                              int32_t batch, int32_t next_n, int32_t heads, int32_t head_dim,
                              float* logits, int64_t logits_stride, int64_t max_model_len,
                              int32_t k, int32_t* indices, int64_t indices_stride,
                              uint32_t* status, sai_stream_t stream);

/*
 * sai_paged_mqa_logits_topk_static_reset -- zero the static workspace of
 * sai_paged_mqa_logits_topk_static on the current device (one memset of its
 * 5 * 16384 + 4 int32 on `stream`; nothing is allocated).  After a call that
 * raised SAI_STATUS_TIMEOUT, a reset ordered after that call and before the
 * next one makes the static entry point usable again.  It races with a
 * static call in flight on another stream, like two static calls do.
 * Returns SAI_OK, or SAI_ERR_CUDA when the array's address cannot be looked
 * up on the current device or the memset cannot be enqueued.
 */
SAI_API int sai_paged_mqa_logits_topk_static_reset(sai_stream_t stream);

/*
 * sai_indexer_k_quant_insert -- quantise new K rows to FP8 and write them into
 * the paged K-cache (one launch).  The step before the logits: the cache
 * kernels address slots in int64 (ATOM PR 2533, "[MLA] Address Triton decode
 * KV rows with int64 ids", section "Problem").
 *
 *   k_bf16        device, bf16 bits [num_tokens, head_dim], contiguous.  16-byte aligned.
 *   num_tokens    rows of k (>= 0; 0 launches nothing and accepts null pointers).
 *   head_dim      must be 128.
 *   slot_mapping  device, int64 [num_tokens]: token t goes to slot
 *                 slot_mapping[t] = page * page_size + position.  A negative
 *                 slot writes nothing (padding); a slot at or past
 *                 num_pages * page_size writes nothing and raises
 *                 SAI_STATUS_BAD_PAGE.  Slots must be distinct.  8-byte aligned.
 *   kv_cache      device, the paged cache of sai_paged_mqa_logits (num_pages
 *                 pages of page_size * (head_dim + 4) bytes, layout kv_layout).
 *                 Only the written tokens' bytes change.  16-byte aligned.
 *   page_size     8, 16, 32, 64, 128 or 256.
 *   status        nullable device uint32 word; SAI_STATUS_* bits are OR-ed in.
 *
 * Per token: scale = amax / 448 in fp32 (448 is the largest e4m3fn
 * magnitude; 1 for an all-zero row); each value's byte is the e4m3fn code
 * of the fp32 quotient value / scale, rounded to nearest, ties to even,
 * saturating at +-448.  The scale is stored as the token's fp32 scale.
 */
SAI_API int sai_indexer_k_quant_insert(const uint16_t* k_bf16, int64_t num_tokens, int32_t head_dim,
                               const int64_t* slot_mapping, uint8_t* kv_cache, int64_t num_pages,
                               int32_t page_size, int32_t kv_layout, uint32_t* status,
                               sai_stream_t stream);

/*
 * sai_gather_selected_kv -- the consumer's gather of the selected tokens' KV
 * rows (one launch).  Row ids are formed and multiplied by the row size in
 * 64 bits (ATOM PR 2533, "[MLA] Address Triton decode KV rows with int64
 * ids": an int32 product wraps past row 2^31 / 576).
 *
 *   indices       device, int32 [rows, indices_stride] (>= k): token
 *                 positions, as written by sai_top_k_per_row_decode; -1 = none.
 *   rows, k       query rows (>= 0; 0 launches nothing) and entries per row.
 *   next_n        rows per request: row r belongs to request r / next_n.
 *   block_table   device, int32 [rows / next_n, block_table_stride]: token t of
 *                 a request is at position t % page_size of page
 *                 block_table[b, t / page_size].
 *   page_size     tokens per page of the KV pool, 1 .. 65536.
 *   kv_pool       device, token-major rows: row id j = page * page_size +
 *                 position occupies bytes [j * row_bytes, (j + 1) * row_bytes).
 *                 16-byte aligned; may be null when out is null.
 *   num_pages     pages in the pool (page ids are checked against it).
 *   row_bytes     bytes per KV row: a multiple of 16, at most 4096 (576 for
 *                 an FP8 MLA row).
 *   row_ids       nullable device int64 [rows, k]: the selected row ids, -1
 *                 for a -1 index or a bad table entry.  8-byte aligned.
 *   out           nullable device [rows, k, row_bytes]: the selected rows, all
 *                 zero where the row id is -1.  16-byte aligned.
 *   status        nullable device word: SAI_STATUS_BAD_PAGE for an index whose
 *                 table entry lies past the table row or names a page outside
 *                 the pool.
 * At least one of row_ids and out must be non-null.
 */
SAI_API int sai_gather_selected_kv(const int32_t* indices, int64_t indices_stride, int32_t rows, int32_t k,
                           int32_t next_n, const int32_t* block_table, int64_t block_table_stride,
                           int32_t page_size, const uint8_t* kv_pool, int64_t num_pages, int32_t row_bytes,
                           int64_t* row_ids, uint8_t* out, uint32_t* status, sai_stream_t stream);

/*
 * sai_selftest_bounded_wait -- exercises the bounded wait that every pipeline
 * wait of the library's kernels uses (one launch of one CTA).  The pages have
 * no counterpart: a correct pipeline never lets a wait run out, so this entry
 * point builds the one situation that does, a shared-memory barrier that
 * nothing ever arrives on, to check that the wait ends, reports
 * SAI_STATUS_TIMEOUT and leaves the context usable.
 *
 *   mode     0: the wait's cycle budget is `cycles`;
 *            1: the wait has the kernels' budget (2^31 SM cycles, about 1 s)
 *               and a second warp raises the CTA's abort flag after `cycles`
 *               cycles, as a failing warp does in the kernels.
 *   cycles   1 .. 2^31 SM clock cycles.
 *   status   device uint32 word (required); SAI_STATUS_TIMEOUT is OR-ed in
 *            when the wait gives up, which it always does.
 * Returns SAI_ERR_INVALID_ARGUMENT for another mode, a cycle count out of
 * range or a null status.
 */
SAI_API int sai_selftest_bounded_wait(int32_t mode, int64_t cycles, uint32_t* status, sai_stream_t stream);

/* Static, human-readable name of a return code. */
SAI_API const char* sai_error_string(int code);

/* Version of this ABI: major * 10000 + minor * 100 + patch. */
SAI_API int sai_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SAI_H_ */
