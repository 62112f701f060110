/*
 * idx_fp4 — MXFP4 DSA lightning indexer for GB300 (sm_103a): C ABI.
 *
 * The indexer keeps index keys as MXFP4 in a paged cache and, for each query row q,
 * scores every visible key t as
 *
 *     logit[q, t] = sum_h w[q, h] * relu(q_h . k_t)
 *
 * then returns the top-k keys by logit. Sources, by page and section:
 *   "Score a DSA sparse indexer in FP4" (ROCm/ATOM pull 2216)
 *     - squashed commit message: keys stored as packed E2M1 plus e8m0 scales; one index
 *       region declared in two planes, read in place by prefill and decode; decode and
 *       prefill scorers driven by a persistent-grid CTA schedule built once per step at a
 *       CUDA-graph-stable address; index_head_dim 128; page block size 64;
 *     - review finding 2 and the sub-commit "Use the index scale plane's own row order
 *       when staging FP4 prefill under DCP": the packed plane's in-page rows are flat, the
 *       scale plane stores them as a 16x4 transpose, slot (row % 16) * 4 + row / 16;
 *     - sub-commit "Schedule, refuse and document the FP4 indexer paths the review found":
 *       the fused writer skips slots < 0; a schedule that under-covers rows is an error,
 *       never a silent truncation; the prefill top-k takes per-row key bounds; padding
 *       rows carry zero weights.
 *   "PCP correctness fixes" (ROCm/ATOM pull 2125), Technical Details section 3: padding
 *       rows are folded into the last request's group at position 0 and read no key.
 *
 * Conventions for every call
 *   - Pointers marked "device" are device pointers owned by the caller; the library
 *     allocates no memory. Host sizing functions (which query nothing on the device) say how
 *     large the caller's schedule and workspace buffers must be. The one exception to
 *     "no device state of its own" is idx_fp4_decode_logits_topk_static (end of this file):
 *     a fixed array on every GPU that loads the library, whose first call per device must
 *     come before any stream capture, and whose overlapping calls race. On the host the
 *     library caches, per device and kernel, that the kernel's shared-memory attribute was
 *     set (under a lock), and the static array's device address.
 *   - Every other call is asynchronous on `stream`, launches only kernels, and may be
 *     captured into a CUDA graph. Nothing is sized from device data, so a captured graph may
 *     be replayed after the device-side inputs (context lengths, row ends, tables) change.
 *     The decode scorer is a cooperative launch of one CTA per SM (its CTAs exchange
 *     histograms through the workspace and wait for each other, boundedly).
 *   - Kernels are launched with programmatic stream serialization: each waits for the
 *     preceding grid in the stream to complete before it touches memory, then lets the next
 *     kernel begin launching. Stream order is unchanged for ordinary kernels, copies and
 *     events that follow a call. A caller's own kernel launched with programmatic stream
 *     serialization right after a call must wait for its prerequisite grid
 *     (cudaGridDependencySynchronize / griddepcontrol.wait) before it reads the call's
 *     outputs, as such kernels must after any kernel.
 *   - Return value: IDX_FP4_OK, or an IDX_FP4_ERR_* code from host-side argument checks
 *     (nothing is launched then), or IDX_FP4_ERR_CUDA if a launch failed.
 *   - `status_dev` (device int32, nullable): kernels OR IDX_FP4_DEV_* bits into it when
 *     they meet invalid device data (a slot past the pool, a page id outside the pool, a
 *     context longer than the table, row ends past the context, an inconsistent
 *     schedule). The offending work is skipped or clamped to safe addresses; no kernel
 *     traps. The caller clears the word; the library only sets bits.
 *   - Shape gate (mirrors the structural gate on the pages; there is no fallback):
 *     head_dim 128 and page 64 are fixed by the layout; num_heads in {16, 32, 64, 128};
 *     1 <= topk <= IDX_FP4_MAX_TOPK. A mismatch returns IDX_FP4_ERR_SHAPE.
 *
 * Data layout
 *   kv_packed  uint8 [num_pages][4][64][16]  group g holds dims 32g..32g+31 of the key in
 *              row `row` of page `page`, two E2M1 codes per byte, even dim in the low nibble.
 *   kv_scale   uint8 [num_pages][4][64]      e8m0 scale of (page, group g, row) at index
 *              [page][g][(row % 16) * 4 + row / 16].
 *   q_packed   uint8 [rows][num_heads][64]   plain, dims in order, even dim in the low nibble.
 *   q_scale    uint8 [rows][num_heads][4]    plain e8m0 scale per 32 dims.
 *   weights    float [rows][num_heads]
 *   block_tables int32 [tables][block_table_stride]: logical page i of table b is
 *              block_tables[b * block_table_stride + i]; entries past the last page a row
 *              reads are never read.
 *   topk_idx   int32 [rows][topk]: selected logical token indices in ascending order, then
 *              -1; topk_val float [rows][topk] (nullable): their logits, then -inf.
 *   Selection is exact: the min(topk, n) keys with the largest logits, ties going to the
 *   lower token index.
 */
#ifndef IDX_FP4_H
#define IDX_FP4_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define IDX_FP4_OK 0
#define IDX_FP4_ERR_ARG 1      /* null pointer where one is required, negative size, bad stride */
#define IDX_FP4_ERR_SHAPE 2    /* unsupported num_heads or topk */
#define IDX_FP4_ERR_CAPACITY 3 /* a caller buffer is smaller than the sizing function requires */
#define IDX_FP4_ERR_CUDA 4     /* a CUDA launch or device query failed */

#define IDX_FP4_DEV_BAD_SLOT 0x01     /* writer: slot >= num_pages * 64 (token skipped) */
#define IDX_FP4_DEV_BAD_PAGE 0x02     /* scorer: page id outside [0, num_pages) (page 0 read instead) */
#define IDX_FP4_DEV_BAD_CTX 0x04      /* context < 0, > max_ctx, or past the block-table width */
#define IDX_FP4_DEV_BAD_ROWS 0x08     /* prefill: cu_seqlens not monotone / not ending at num_rows, or a
                                         row end past its request's context (clamped) */
#define IDX_FP4_DEV_BAD_SCHEDULE 0x10 /* decode: schedule built for another batch or grid, or ctx_lens
                                         changed since it was built (call skipped) */
#define IDX_FP4_DEV_TIMEOUT 0x20      /* a bounded on-chip wait gave up (results undefined) */
#define IDX_FP4_DEV_CAPACITY 0x40     /* the schedule or workspace was sized for smaller contexts than
                                         the call met (affected rows come out as -1) */
#define IDX_FP4_DEV_SYNC 0x80         /* decode: the CTAs sharing a sequence saw inconsistent counts (a
                                         workspace not zero-filled, or calls overlapping on it) */

#define IDX_FP4_MAX_TOPK 2048
#define IDX_FP4_MAX_BATCH 4096        /* sequences per decode call, requests per prefill call */
#define IDX_FP4_MAX_PREFILL_ROWS 8192 /* query rows per prefill call */

/* Writer: quantise bf16 keys to MXFP4 and store them in the paged cache; optionally quantise
 * query heads to the plain MXFP4 layout. ("Score a DSA sparse indexer in FP4", squashed commit
 * message: the FP4 output mode of the fused writer; sub-commit "Schedule, refuse and document
 * ...": slots < 0 are skipped.)
 *   k_bf16        device uint16 [num_tokens][128], bf16 bit patterns (may be NULL if num_tokens == 0)
 *   slot_mapping  device int32 [num_tokens]; token i goes to page slot/64, row slot%64; slot < 0
 *                 is skipped; slot >= num_pages*64 sets IDX_FP4_DEV_BAD_SLOT and is skipped
 *   kv_packed, kv_scale  device cache planes (layout above), written in place
 *   q_bf16        device uint16 [num_q_rows][num_heads][128] or NULL (then q is not touched)
 *   q_packed, q_scale    device outputs [num_q_rows][num_heads][64] / [..][4] (required iff q_bf16)
 * Quantiser: per 32 dims, scale 2^e with e the smallest integer such that max|x| <= 6 * 2^e
 * (byte e + 127; an all-zero block gets byte 0); each element rounds to the nearest E2M1 value,
 * ties to the even code; the sign bit is set iff the input is negative. */
int idx_fp4_quant_and_cache(const uint16_t *k_bf16, int64_t num_tokens, const int32_t *slot_mapping,
                            uint8_t *kv_packed, uint8_t *kv_scale, int64_t num_pages, const uint16_t *q_bf16,
                            int64_t num_q_rows, int num_heads, uint8_t *q_packed, uint8_t *q_scale,
                            int32_t *status_dev, cudaStream_t stream);

/* Bytes of the decode schedule buffer for up to `max_batch` sequences of up to `max_ctx` keys,
 * for any next_n and any GPU of up to 1024 SMs (host only; 0 for invalid arguments, or when
 * max_batch * ceil(max_ctx / 128) exceeds 2^31 - 1). */
size_t idx_fp4_decode_schedule_bytes(int max_batch, int64_t max_ctx);

/* Build the decode CTA schedule once per step, before the layers; every decode call of the
 * step reads it. ("Score a DSA sparse indexer in FP4", squashed commit message and PR section
 * "Decode grid floor": a persistent-grid schedule built once a step at a CUDA-graph-stable
 * address; here the grid is sized to the work — each CTA gets an equal share of 128-key tiles
 * — instead of to a fixed floor, and the count lives on the device.)
 *   ctx_lens_dev  device int32 [batch]: keys visible to each sequence (0 allowed)
 *   batch <= max_batch; max_ctx bounds every context (larger sets IDX_FP4_DEV_BAD_CTX and the
 *   sequence is treated as empty)
 *   sched_dev     device buffer of sched_bytes >= idx_fp4_decode_schedule_bytes(max_batch, max_ctx)
 * The schedule targets the current device's SM count; use it on that device. All sequences'
 * 128-key tiles are laid end to end and cut into rounds of one equal range per SM, a range
 * holding at most 16384 keys (one query row per sequence); a sequence spread over several
 * ranges is selected jointly by the CTAs holding it, inside idx_fp4_decode_logits_topk. */
int idx_fp4_build_decode_schedule(const int32_t *ctx_lens_dev, int batch, int max_batch, int64_t max_ctx,
                                  void *sched_dev, size_t sched_bytes, int32_t *status_dev, cudaStream_t stream);

/* Bytes of the decode workspace for schedules built with (max_batch, max_ctx) and the given topk
 * (host only; 0 for invalid arguments). The workspace holds the exchange between the CTAs that
 * share a sequence: each unit's published histogram bins, the sequence's candidate keys (at most
 * 8 bytes per key of the batch) and a few counters. It must be zero-filled before its first use;
 * every call leaves its counters at zero again, except a call that reports IDX_FP4_DEV_TIMEOUT,
 * after which the caller zero-fills the workspace again. Calls that share a workspace must not
 * overlap on the GPU. */
size_t idx_fp4_decode_workspace_bytes(int max_batch, int64_t max_ctx, int topk);

/* Decode: one query row per sequence b scores keys [0, ctx_lens[b]) through block_tables[b]
 * and selects its top-k. ("Score a DSA sparse indexer in FP4": the decode scorer reads q,
 * q_scale, the paged planes, the block table and the CTA schedule; the top-k of a row is
 * bounded by its context.) Logits never leave the chip unless logits_debug is given.
 *   q_packed [batch][H][64], q_scale [batch][H][4], weights [batch][H]   device
 *   kv_packed, kv_scale, num_pages   the cache
 *   block_tables, block_table_stride  device int32 [batch][stride]
 *   ctx_lens_dev   the vector the schedule was built from (checked against it)
 *   sched_dev/sched_bytes   from idx_fp4_build_decode_schedule for this batch
 *   workspace      device, >= idx_fp4_decode_workspace_bytes(max_batch, max_ctx, topk) for the
 *                  schedule's sizes, zero-filled before first use (a smaller one sets
 *                  IDX_FP4_DEV_CAPACITY and every row comes out empty)
 *   topk_idx [batch][topk] (device, required), topk_val [batch][topk] (nullable)
 *   logits_debug   nullable device float [batch][logits_stride]: every scored logit (testing) */
int idx_fp4_decode_logits_topk(const uint8_t *q_packed, const uint8_t *q_scale, const float *weights,
                               const uint8_t *kv_packed, const uint8_t *kv_scale, int64_t num_pages,
                               const int32_t *block_tables, int block_table_stride, const int32_t *ctx_lens_dev,
                               int batch, int num_heads, int topk, const void *sched_dev, size_t sched_bytes,
                               void *workspace, size_t workspace_bytes, int32_t *topk_idx, float *topk_val,
                               float *logits_debug, int64_t logits_stride, int32_t *status_dev,
                               cudaStream_t stream);

/* ---- Decode with next_n query rows per sequence (speculative-decoding verify rows) --------
 * ("Score a DSA sparse indexer in FP4", squashed commit message: the MTP draft folds its
 * batch x next_n verify rows back onto the batch's sequences and rebuilds the decode schedule for
 * them.) Sequence b carries rows b * next_n + j, j < next_n; row j sees keys
 * [0, ctx_lens[b] - next_n + 1 + j), so the last row sees the whole context and every row a key
 * pass shared with the others: the keys are streamed once for all next_n rows.
 * next_n is 1, 2 or 4 with next_n * num_heads <= 128 (else IDX_FP4_ERR_SHAPE; larger shapes go
 * through idx_fp4_prefill_logits_topk, one request per sequence).
 *   Schedule: idx_fp4_build_decode_schedule_mtp with the same next_n (a range holds at most
 *   16384 keys for next_n 2, 8192 for 4), into a buffer of idx_fp4_decode_schedule_bytes.
 *   Workspace: idx_fp4_decode_mtp_workspace_bytes, zero-filled before first use.
 *   q_packed [batch * next_n][H][64], q_scale [batch * next_n][H][4], weights [batch * next_n][H];
 *   topk_idx / topk_val [batch * next_n][topk]; logits_debug [batch * next_n][logits_stride].
 * Everything else as for idx_fp4_decode_logits_topk, which is this call with next_n = 1. */
int idx_fp4_build_decode_schedule_mtp(const int32_t *ctx_lens_dev, int batch, int next_n, int max_batch,
                                      int64_t max_ctx, void *sched_dev, size_t sched_bytes, int32_t *status_dev,
                                      cudaStream_t stream);

size_t idx_fp4_decode_mtp_workspace_bytes(int max_batch, int64_t max_ctx, int topk, int next_n);

int idx_fp4_decode_mtp_logits_topk(const uint8_t *q_packed, const uint8_t *q_scale, const float *weights,
                                   const uint8_t *kv_packed, const uint8_t *kv_scale, int64_t num_pages,
                                   const int32_t *block_tables, int block_table_stride, const int32_t *ctx_lens_dev,
                                   int batch, int next_n, int num_heads, int topk, const void *sched_dev,
                                   size_t sched_bytes, void *workspace, size_t workspace_bytes, int32_t *topk_idx,
                                   float *topk_val, float *logits_debug, int64_t logits_stride, int32_t *status_dev,
                                   cudaStream_t stream);

/* ---- Key-sharded decode (context parallelism) -----------------------------------------------
 * ("Score a DSA sparse indexer in FP4", section "Decode context parallelism": each rank scores its
 * own shard of every sequence's keys and keeps its local top-k; the ranks' candidates are gathered
 * and merged into each row's top-k.) On one GPU the shards are key ranges scored by separate
 * decode calls; across GPUs each rank runs its own range and the caller gathers the candidate
 * lists (an all-gather of [rows][topk] indices and values per rank) before the merge.
 *
 * idx_fp4_build_decode_schedule_range: a decode schedule (next_n = 1) in which sequence b scores
 * only the keys [key_begin[b], key_end[b]) (device int32 [batch] each). key_begin[b] must be a
 * multiple of 128 (the scorer's key tile) with 0 <= key_begin[b] <= key_end[b] <= max_ctx, else
 * IDX_FP4_DEV_BAD_CTX is set and the row scores no key. Run it with idx_fp4_decode_logits_topk,
 * passing key_end_dev as ctx_lens_dev: row b then holds the top-min(topk, key_end - key_begin)
 * keys of its range with absolute token indices (ascending), padded with -1 / -inf. Sizing
 * functions, workspace and the other arguments are those of the plain decode call. */
int idx_fp4_build_decode_schedule_range(const int32_t *key_begin_dev, const int32_t *key_end_dev, int batch,
                                        int max_batch, int64_t max_ctx, void *sched_dev, size_t sched_bytes,
                                        int32_t *status_dev, cudaStream_t stream);

/* idx_fp4_merge_candidates: the exact top-k of the union of num_lists candidate lists per row.
 *   cand_val f32 / cand_idx int32 [num_lists][rows][k_in] (device): list l of row r at
 *     (l * rows + r) * k_in; entries with a negative index are empty. The indices of one row
 *     are distinct (shards hold disjoint keys).
 *   topk_idx [rows][topk] (required), topk_val [rows][topk] (nullable), device, caller-owned.
 * Row r keeps the min(topk, valid entries) best by (value descending, index ascending) and
 * writes them in ascending index order, padded with -1 / -inf: merging the lists of every key
 * range of a sequence gives exactly the sequence's decode top-k. One CTA per row.
 * num_lists * k_in <= IDX_FP4_MERGE_MAX_CANDIDATES (else IDX_FP4_ERR_CAPACITY); 1 <= topk <=
 * IDX_FP4_MAX_TOPK (else IDX_FP4_ERR_SHAPE); rows == 0 launches nothing. status_dev may be NULL:
 * this call detects nothing on the device. */
#define IDX_FP4_MERGE_MAX_CANDIDATES 16384
int idx_fp4_merge_candidates(const float *cand_val, const int32_t *cand_idx, int num_lists, int rows, int k_in,
                             int topk, int32_t *topk_idx, float *topk_val, int32_t *status_dev,
                             cudaStream_t stream);

/* Bytes of the prefill workspace (the call's unit table, and candidate lists for rows longer
 * than one unit's 8192-key (64-head) / 16384-key (128-head) share) for rows of up to max_ctx
 * keys (host; 0 for invalid arguments). */
size_t idx_fp4_prefill_workspace_bytes(int num_requests, int num_rows, int num_heads, int64_t max_ctx, int topk);

/* Causal prefill: row r of request g (cu_seqlens[g] <= r < cu_seqlens[g+1]) scores keys
 * [0, row_ends[r]) through block_tables[g] and selects its top-min(topk, row_ends[r]).
 * ("Score a DSA sparse indexer in FP4": the prefill scorer finds a row's page table through
 * its group and takes per-row key bounds; "PCP correctness fixes", section 3: padding rows sit
 * at position 0 in the last request's group and read no key — here they carry row_end 0 and
 * come out as all -1.)
 *   q_packed [num_rows][H][64], q_scale [num_rows][H][4], weights [num_rows][H]   device
 *   ctx_lens_dev [num_requests]: keys cached per request; row_ends[r] <= ctx_lens[g] is checked
 *   cu_seqlens_dev [num_requests + 1], non-decreasing, cu_seqlens[0] = 0, cu_seqlens[G] = num_rows
 *   row_ends_dev [num_rows]: a real row at 0-based position p carries p + 1
 *   max_ctx    bound on every row end, the value the workspace was sized with
 *   workspace  device, >= idx_fp4_prefill_workspace_bytes(num_requests, num_rows, num_heads, max_ctx, topk)
 * Rows longer than one unit's share are scored in key chunks and merged inside the call.
 * Decode with next_n query rows per sequence can also be run as this call, with one request per
 * sequence b of next_n rows, row j carrying row_end ctx_b - next_n + 1 + j (num_heads stays the
 * index head count of one row); idx_fp4_decode_mtp_logits_topk is the decode-shaped form.
 *   topk_idx [num_rows][topk] (required), topk_val (nullable), logits_debug as for decode */
int idx_fp4_prefill_logits_topk(const uint8_t *q_packed, const uint8_t *q_scale, const float *weights,
                                const uint8_t *kv_packed, const uint8_t *kv_scale, int64_t num_pages,
                                const int32_t *block_tables, int block_table_stride, const int32_t *ctx_lens_dev,
                                const int32_t *cu_seqlens_dev, const int32_t *row_ends_dev, int num_requests,
                                int num_rows, int num_heads, int topk, int64_t max_ctx, void *workspace,
                                size_t workspace_bytes, int32_t *topk_idx, float *topk_val, float *logits_debug,
                                int64_t logits_stride, int32_t *status_dev, cudaStream_t stream);

/* ---- Decode without a caller workspace -------------------------------------------------
 * The pages have no counterpart of this call; it is here for callers that cannot allocate
 * device memory (code running inside an allocator or memory-pool hook, an embedding runtime
 * that owns every device allocation, or a path that must never wait on the allocator). It does
 * what idx_fp4_decode_logits_topk does, with the workspace taken from a fixed array of
 * IDX_FP4_STATIC_SCRATCH_BYTES (16 MiB) that the library holds on every GPU it is loaded on
 * until the process exits. It allocates nothing.
 *   Arguments as for idx_fp4_decode_logits_topk, minus workspace/workspace_bytes, plus
 *   max_ctx: the bound the schedule was built with (every ctx_lens[b] <= max_ctx). The schedule
 *   must be built with max_batch = batch and this max_ctx (else IDX_FP4_DEV_CAPACITY is set and
 *   every row comes out empty).
 *   Returns IDX_FP4_ERR_CAPACITY, launching nothing, when the workspace such a schedule needs
 *   (idx_fp4_decode_static_bytes) exceeds the array: split the batch or use the workspace call.
 * The first call on a device looks up the array's device address (and may load the library's
 * device code); make that first call before any stream capture. All calls on a device share
 * the one array, so calls that overlap on the GPU (other streams, other host threads) race and
 * must be serialised by the caller. Each call first clears the array's synchronisation words
 * on `stream` (cudaMemsetAsync); everything else it reads is written earlier in the same call.
 * The cached device address does not survive cudaDeviceReset: do not use this call afterwards
 * in the same process. */
#define IDX_FP4_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* Scratch bytes idx_fp4_decode_logits_topk_static needs for this batch (host only; the same as
 * idx_fp4_decode_workspace_bytes(batch, max_ctx, topk); 0 for invalid arguments). */
size_t idx_fp4_decode_static_bytes(int batch, int64_t max_ctx, int topk);

int idx_fp4_decode_logits_topk_static(const uint8_t *q_packed, const uint8_t *q_scale, const float *weights,
                                      const uint8_t *kv_packed, const uint8_t *kv_scale, int64_t num_pages,
                                      const int32_t *block_tables, int block_table_stride,
                                      const int32_t *ctx_lens_dev, int batch, int num_heads, int topk,
                                      int64_t max_ctx, const void *sched_dev, size_t sched_bytes,
                                      int32_t *topk_idx, float *topk_val, float *logits_debug,
                                      int64_t logits_stride, int32_t *status_dev, cudaStream_t stream);

/* ---- Measurement ------------------------------------------------------------------------
 * The MXFP4 tensor-core rate the prefill scorer is measured against (the pages give no FP4
 * peak): idx_fp4_mxf4_probe launches, on `stream`, one CTA per SM whose warps issue `iters`
 * pairs of block-scaled MXFP4 MMAs each (tcgen05.mma kind::mxf4, M = 128, N = 128, K = 64, the
 * scorers' instruction) from shared-memory operands; time it with events and divide
 * idx_fp4_mxf4_probe_flops(iters) (host: the launch's FLOPs on the current device, 0 for
 * iters < 1) by the time. 1 <= iters <= 2^20 (else IDX_FP4_ERR_ARG). Reads and writes no
 * caller memory except status_dev (nullable; IDX_FP4_DEV_TIMEOUT if a bounded wait gave up). */
int64_t idx_fp4_mxf4_probe_flops(int iters);
int idx_fp4_mxf4_probe(int iters, int32_t *status_dev, cudaStream_t stream);

/* Human-readable name of a return code. */
const char *idx_fp4_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* IDX_FP4_H */
