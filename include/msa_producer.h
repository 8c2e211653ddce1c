/*
 * msa_producer.h -- C ABI of the MiniMax-M3 MSA per-layer fused producer and
 * paged-cache write, for NVIDIA GB300 (sm_103a).
 *
 * The operation ("[None][perf] Fuse MiniMax-M3 QKV and index projection",
 * TensorRT-LLM PR 18205, Description, "AFTER" diagram and the list under "This
 * change adds"): one fused producer takes the packed projection row
 * [Q | K | V | index-Q | index-K] of every new token, applies per-head Q/K
 * RMSNorm and RoPE, emits compact Q and index-Q, and writes the current K, V and
 * index-K directly into paged head-major (HND) caches, with strided cache
 * layouts, 64-bit element offsets, CUDA Graph replay and safe containment of
 * padded or out-of-range cache slots.  The page and in-page offset of a token are
 * derived once per token ("[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache
 * writes into one kernel", PR 18614, "The fix"), from a slot that is either a
 * physical slot or a logical slot looked up through a page table ("Wire in
 * custom decode kernels for MinimaxM3", PR 18611, merge commit message: write
 * slots re-derived from the staged block table).
 *
 * Per token t, with D = head_dim, P = page_size:
 *   placement   ls = slot_mapping[t]; nothing is written to a cache when ls < 0.
 *               block = ls / P, off = ls % P; page = page_table[block] when a
 *               table is given (nothing written when block >= page_table_len),
 *               else page = block; a cache takes the token only when
 *               0 <= page < that cache's num_pages.
 *   RMSNorm     y = (x * r) * w, r = 1 / sqrt(sum(x^2) / D + rms_eps), per head,
 *               one weight vector [D] per tensor shared by its heads; applied to
 *               Q, K, index-Q and index-K, not to V.
 *   RoPE        after the norm, on dims [0, rotary_dim) at angle
 *               positions[t] * rope_theta^(-2k / rotary_dim) for pair k;
 *               NeoX pairs (k, k + rotary_dim/2), GPT-J pairs (2k, 2k + 1):
 *               u' = u cos - v sin, v' = v cos + u sin.  Other dims pass through.
 *   outputs     q_out[t, h, :] and idx_q_out[t, h, :] in bf16 (round to nearest
 *               even), written for every token, padded ones included.
 *   caches      cache[page*stride_page + h*stride_head + off*stride_token + d]:
 *               FP8 E4M3 caches store e4m3(x * (1/scale)), round to nearest even,
 *               saturating to +-448; BF16 caches store bf16(x) (no scale).
 *               K and index-K take the normed, rotated values, V the raw ones.
 *
 * Arithmetic is fp32 inside the kernel.
 *
 * Ownership and threading: the caller owns every buffer.  The library
 * allocates no memory, never synchronises, never reads device memory on the
 * host, and enqueues at most one kernel on `stream`; a call is therefore
 * stream-ordered and can be captured into a CUDA graph.  Calls on different
 * streams that write the same cache cells race, as any two kernels would.
 *
 * Errors: every argument check runs on the host before any launch; a call that
 * returns an error has enqueued nothing and written nothing.
 */
#ifndef MSA_PRODUCER_H
#define MSA_PRODUCER_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MSA_OK = 0,
    MSA_ERR_INVALID_ARGUMENT = 1,  /* null pointer, negative size, inconsistent count,
                                      overlapping cache rows, unknown flag */
    MSA_ERR_UNSUPPORTED = 2,       /* valid but not built: head_dim other than 64 or 128,
                                      rotary_dim not a multiple of 16 (NeoX) or 8 (GPT-J),
                                      unknown dtype, rope style or scale mode */
    MSA_ERR_MISALIGNED = 3,        /* a base pointer or stride breaks the alignment below */
    MSA_ERR_OFFSET_OVERFLOW = 4,   /* the furthest reachable cache byte does not fit in
                                      a signed 64-bit offset or wraps the address space */
    MSA_ERR_CUDA = 5               /* the CUDA runtime refused a query or the launch */
} msa_status;

typedef enum { MSA_DTYPE_BF16 = 0, MSA_DTYPE_FP8_E4M3 = 1 } msa_dtype;
typedef enum { MSA_ROPE_NEOX = 0, MSA_ROPE_GPTJ = 1 } msa_rope_style;
typedef enum { MSA_SCALE_PER_TENSOR = 0, MSA_SCALE_PER_HEAD = 1 } msa_scale_mode;

/* Launch flags (bit set). */
#define MSA_LAUNCH_PERSISTENT 1   /* grid of at most (SMs x resident CTAs) CTAs that
                                     stride over the tokens; otherwise one CTA per token */
#define MSA_LAUNCH_PDL 2          /* programmatic dependent launch: the kernel may start
                                     before the kernels enqueued ahead of it on the stream
                                     have completed.  It reads qkv and writes anything only
                                     after waiting for them; it reads the norm weights,
                                     positions, slot mapping and page table before that
                                     wait.  The producer lets the next kernel start as soon
                                     as it begins, so a run of launches with this flag may
                                     be in flight together: those four arrays must not be
                                     written by any kernel enqueued after the last kernel
                                     of the stream launched without programmatic dependent
                                     launch.  Stage them with plain launches (a copy) before
                                     the run, e.g. once at the start of a decode step. */
#define MSA_LAUNCH_QUERY_RUNS 4   /* msa_indexer_forward only: the queries come in runs of
                                     one sequence (consecutive queries with the same
                                     table_offset, as in a prefill chunk), so tiles of 8
                                     or 16 consecutive queries are scored together on the
                                     tcgen05 tensor cores against each 128-token block they
                                     share (block_tokens 128; other block sizes take the
                                     per-query kernel).  The results are those of the
                                     per-query kernel; a tile spanning several sequences
                                     is scored one sequence at a time. */

/* One paged cache.  Element (page, head, off, d) lives at
 *   data + (page*stride_page + head*stride_head + off*stride_token + d) * elem_size
 * with elem_size 1 for FP8 E4M3 and 2 for BF16.  HND pages [num_heads, P, D] are
 * stride_head = P*D, stride_token = D; any other non-overlapping strides work
 * (padded pages, K and V interleaved in one pool, NHD).  Requirements: data
 * 16-byte aligned; the three strides non-negative multiples of 8 elements; the
 * rows (head, off) of different pages and heads must not overlap. */
typedef struct {
    void *data;              /* device memory; caller-owned */
    int32_t dtype;           /* msa_dtype */
    int32_t reserved;        /* must be 0 */
    int64_t num_pages;       /* pages in this cache; pages >= num_pages are dropped */
    int64_t num_heads;       /* must equal the number of heads written to it */
    int64_t stride_page;     /* elements */
    int64_t stride_head;     /* elements */
    int64_t stride_token;    /* elements; the dim stride is 1 */
} msa_cache_desc;

typedef struct {
    int32_t num_q_heads;      /* Hq  >= 0 */
    int32_t num_kv_heads;     /* Hkv >= 0 (K and V each) */
    int32_t num_idx_q_heads;  /* Hiq >= 0 */
    int32_t num_idx_k_heads;  /* Hik >= 0 */
    int32_t head_dim;         /* D: 64 or 128 */
    int32_t rotary_dim;       /* 0 <= rotary_dim <= D */
    int32_t rope_style;       /* msa_rope_style */
    int32_t page_size;        /* P > 0 tokens per page */
    float rope_theta;         /* > 0 */
    float rms_eps;            /* >= 0 */
    int32_t scale_mode;       /* msa_scale_mode */
    int32_t reserved;         /* must be 0 */
} msa_producer_cfg;

/*
 * Runs the fused producer over num_tokens tokens on `stream`.
 *
 * qkv            device bf16 [num_tokens, qkv_row_stride]; row t holds
 *                [Q (Hq*D) | K (Hkv*D) | V (Hkv*D) | idx-Q (Hiq*D) | idx-K (Hik*D)],
 *                each section head-major; qkv_row_stride >= that width, in
 *                elements, a multiple of 8; qkv 16-byte aligned.
 * positions      device int32 [num_tokens]: RoPE position of each token.
 * slot_mapping   device int64 [num_tokens]: slot of each token (-1 = padding).
 * page_table     device int32 [page_table_len] or NULL: logical block -> page
 *                (a [seqs, max_blocks] table flattened row-major).  NULL: slots
 *                are physical (page = slot / P).
 * *_norm_w       device bf16 [D] RMSNorm weights for Q, K, idx-Q, idx-K; a weight
 *                may be NULL only when its tensor has no heads or is not written.
 * q_out          device bf16 [num_tokens, Hq, D], 16-byte aligned (NULL iff Hq = 0).
 * idx_q_out      device bf16 [num_tokens, Hiq, D], 16-byte aligned (NULL iff Hiq = 0).
 * k_cache, v_cache  required when Hkv > 0.  idx_k_cache: NULL skips index-K.
 * scales         device fp32: per tensor [3] = {k, v, idx_k}; per head
 *                [2*Hkv + Hik] = K heads, then V heads, then index-K heads.
 *                Read only by FP8 caches; may be NULL when no cache is FP8.
 * launch_flags   MSA_LAUNCH_* bits.
 * stream         CUDA stream (0 = legacy default stream).
 *
 * num_tokens == 0 returns MSA_OK and launches nothing.  Device-side values
 * (slots, table entries, positions) need no checking by the caller: any slot or
 * table entry outside a cache is dropped, so no write leaves the cache extent
 * the descriptor implies.  Two tokens of one call with the same valid slot
 * leave that cell's contents unspecified (each 8-element piece comes from one
 * of them); callers give every token its own slot.
 */
msa_status msa_producer_forward(const msa_producer_cfg *cfg, int64_t num_tokens,
                                const void *qkv, int64_t qkv_row_stride,
                                const int32_t *positions, const int64_t *slot_mapping,
                                const int32_t *page_table, int64_t page_table_len,
                                const void *q_norm_w, const void *k_norm_w,
                                const void *idx_q_norm_w, const void *idx_k_norm_w,
                                void *q_out, void *idx_q_out,
                                const msa_cache_desc *k_cache, const msa_cache_desc *v_cache,
                                const msa_cache_desc *idx_k_cache,
                                const float *scales, int32_t launch_flags, cudaStream_t stream);

/*
 * The host-side checks of msa_producer_forward alone, with the same arguments
 * minus the stream; touches no GPU state.  Lets a caller check a layer once
 * before capturing it into a graph.
 */
msa_status msa_producer_validate(const msa_producer_cfg *cfg, int64_t num_tokens,
                                 const void *qkv, int64_t qkv_row_stride,
                                 const int32_t *positions, const int64_t *slot_mapping,
                                 const int32_t *page_table, int64_t page_table_len,
                                 const void *q_norm_w, const void *k_norm_w,
                                 const void *idx_q_norm_w, const void *idx_k_norm_w,
                                 void *q_out, void *idx_q_out,
                                 const msa_cache_desc *k_cache, const msa_cache_desc *v_cache,
                                 const msa_cache_desc *idx_k_cache,
                                 const float *scales, int32_t launch_flags);

/*
 * Launch shape the forward call would use on the current device: CTAs, threads
 * per CTA and dynamic shared memory bytes.  Returns MSA_ERR_CUDA when the device
 * cannot be queried.  Host-side; enqueues nothing.
 */
msa_status msa_producer_launch_shape(const msa_producer_cfg *cfg, int64_t num_tokens,
                                     int32_t launch_flags, int32_t *grid, int32_t *block,
                                     int32_t *smem_bytes);

/* ------------------------------------------------------------------------ */
/* Indexer: the consumer of the index-K cache (decode)                      */
/* ------------------------------------------------------------------------ */
/*
 * For each query token, scores the visible index-K history and selects the
 * top-k blocks ("[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into
 * one kernel", the layer walk-through: proxy attention over index-K, max-reduce,
 * select the top 16 of 128-token blocks; "[None][perf] Fuse MiniMax-M3 QKV and
 * index projection", AFTER diagram: score visible index-K, max-pool scores by
 * block, select top-k block ids).
 *
 *   token score   s_j = max over index heads h of idx_q[t,h,:] . k_j, where k_j is
 *                 the index-K row of token j (FP8 codes times *k_scale, or bf16),
 *                 for the visible tokens j < kv_len[t]; the page of token j is
 *                 page_table[table_offset[t] + j / page_size]; a token whose table
 *                 index or page falls outside the table or the cache is skipped.
 *   block score   block_scores[t, b] = max of s_j over the tokens of block b
 *                 (block_tokens tokens each), -inf when it has none; blocks at or
 *                 beyond max_blocks are not scored.
 *   top-k         topk_ids[t, :] = the ids of the topk highest finite block scores,
 *                 highest first, ties to the lower id, padded with -1.
 *
 * A positive softmax scale would change neither a max nor the order, so none is
 * applied.  Accumulation is fp32.  Two kernels are enqueued on `stream`; the
 * library allocates nothing (block_scores is an output).
 */
typedef struct {
    int32_t num_heads;     /* index-Q heads: 1..16 */
    int32_t head_dim;      /* 64 or 128 */
    int32_t page_size;     /* tokens per page of the index-K cache, > 0 */
    int32_t block_tokens;  /* tokens per scored block: a multiple of 32, 32..1024 */
    int32_t topk;          /* ids selected per query: 1..64 */
    int32_t max_blocks;    /* columns of block_scores: 1..65536 */
    int32_t reserved[2];   /* must be 0 */
} msa_indexer_cfg;

/*
 * idx_q          device bf16 [num_queries, num_heads, head_dim], 16-byte aligned
 *                (the compact index-Q the producer writes).
 * kv_len         device int32 [num_queries]: visible tokens per query (< 0 as 0).
 * table_offset   device int64 [num_queries]: start of the query's row in page_table.
 * page_table     device int32 [page_table_len].
 * idx_k_cache    one-head cache descriptor (the producer's index-K cache).
 * k_scale        device fp32 [1]: dequantisation scale of an FP8 cache (NULL for bf16).
 * block_scores   device fp32 [num_queries, max_blocks], written in full.
 * topk_ids       device int32 [num_queries, topk].
 * launch_flags   MSA_LAUNCH_PDL: the indexer's first kernel is launched with
 *                programmatic dependent launch; the per-query path reads kv_len,
 *                table_offset and page-table entries before waiting for the kernels
 *                ahead of it on the stream (the rule of MSA_LAUNCH_PDL applies to
 *                them); idx_q, the cache, k_scale and the outputs are touched only
 *                after the wait (the query-run kernel waits before reading anything).
 *                The indexer's kernels let the next kernel on the stream start only
 *                after their own wait.
 *                MSA_LAUNCH_QUERY_RUNS: see its definition.
 * Arithmetic: an FP8 cache's codes are exact in every kernel, and scores accumulate
 * in fp32.  The query is rounded to f16 by the per-query kernel; where the keys are
 * multiplied as stored on the tensor cores (E4M3 keys of 128 dims on the query-run
 * kernels, and decode batches of up to 1,024 queries of up to 16 heads whose index-K
 * pages are whole TMA boxes), each query is split into two E4M3 halves hi + lo under
 * a power-of-two scale, which reproduces its bf16 values exactly except elements
 * below 2^-9 of the query's largest magnitude.  Which kernel runs depends only on
 * the arguments, so a call is deterministic.
 * Errors as for msa_producer_forward; num_queries == 0 launches nothing.
 */
msa_status msa_indexer_forward(const msa_indexer_cfg *cfg, int64_t num_queries, const void *idx_q,
                               const int32_t *kv_len, const int64_t *table_offset,
                               const int32_t *page_table, int64_t page_table_len,
                               const msa_cache_desc *idx_k_cache, const float *k_scale,
                               float *block_scores, int32_t *topk_ids, int32_t launch_flags,
                               cudaStream_t stream);

/*
 * msa_indexer_forward in a single launch, with the top-k taken inside the per-query
 * score kernel instead of a second kernel.  The block scores and ids equal
 * msa_indexer_forward's bit for bit, except where that entry takes the tensor-core
 * decode kernel (see its arithmetic note): there the scores agree within the query
 * split's rounding, and the ids wherever the scores separate them.  Each of the query's CTAs that scores blocks counts itself in
 * counters[t] once its block scores are stored; the CTA that arrives last resets
 * counters[t] to zero and ranks the query's row.
 *
 * counters       device int32 [num_queries], caller-owned scratch: every entry must
 *                be 0 on entry, and a launch that runs to completion leaves every
 *                entry 0 again, so one buffer zeroed once serves any number of
 *                launches issued one after another on a stream (or replayed in a
 *                graph).  Launches that may run at the same time need separate
 *                buffers.  4-byte aligned.
 * launch_flags   as for msa_indexer_forward; with MSA_LAUNCH_QUERY_RUNS the
 *                query-run kernel and the top-k kernel run as there, and counters is
 *                not touched.
 * Other arguments and errors as for msa_indexer_forward; counters NULL is
 * MSA_ERR_INVALID_ARGUMENT, misaligned MSA_ERR_MISALIGNED.  One kernel is enqueued
 * on `stream`; the library allocates nothing.
 */
msa_status msa_indexer_forward_fused(const msa_indexer_cfg *cfg, int64_t num_queries,
                                     const void *idx_q, const int32_t *kv_len,
                                     const int64_t *table_offset, const int32_t *page_table,
                                     int64_t page_table_len, const msa_cache_desc *idx_k_cache,
                                     const float *k_scale, float *block_scores, int32_t *topk_ids,
                                     int32_t *counters, int32_t launch_flags, cudaStream_t stream);

/*
 * msa_indexer_forward_fused_noalloc -- msa_indexer_forward_fused on per-query
 * counters that the library owns instead of the caller: a file-scope device array
 * of 65,536 int32 per device.  No counterpart in the source pages; it exists for
 * callers that cannot allocate device memory on the call path -- a runtime whose
 * allocator does not reach this library (a plain C host, a plugin handed only
 * pointers to its inputs and outputs), or a step being assembled where an
 * allocation would be a synchronising call.  Neither this function nor its kernel
 * allocates anything.
 *
 * The first call on a device looks the array's address up (cudaGetSymbolAddress,
 * its status checked) and zeroes it with cudaMemsetAsync on `stream`, ordered
 * before that call's launch; make that first call outside stream capture.  Later
 * calls only launch.  The array is shared by every call on the device: calls that
 * may run at the same time (on different streams without an ordering between them)
 * race on the counters and give wrong ids -- order them, or give each its own
 * counters through msa_indexer_forward_fused.  A launch that does not run to
 * completion can leave counters nonzero for the calls after it.
 *
 * Arguments, results and errors as for msa_indexer_forward_fused without
 * `counters`; num_queries above 65,536 is MSA_ERR_UNSUPPORTED (checked on the host,
 * before any device call).
 */
msa_status msa_indexer_forward_fused_noalloc(const msa_indexer_cfg *cfg, int64_t num_queries,
                                             const void *idx_q, const int32_t *kv_len,
                                             const int64_t *table_offset, const int32_t *page_table,
                                             int64_t page_table_len,
                                             const msa_cache_desc *idx_k_cache, const float *k_scale,
                                             float *block_scores, int32_t *topk_ids,
                                             int32_t launch_flags, cudaStream_t stream);

/*
 * Device address at which the GPU of the current device reaches host memory
 * `host_ptr` (pinned, mapped host memory; on Grace-Blackwell the GPU reads and
 * writes it over NVLink-C2C).  Sets *device_ptr and returns MSA_OK when the
 * buffer is device-accessible; MSA_ERR_INVALID_ARGUMENT when it is not (pageable
 * or unregistered memory) or an argument is NULL.  Lets a caller pass host
 * buffers straight to msa_producer_forward (rows, positions, slots, compact
 * outputs) with the copies done by the kernel itself.  Host-side; enqueues nothing.
 */
msa_status msa_host_buffer_device_address(const void *host_ptr, void **device_ptr);

/* Static, human-readable name of a status; never NULL. */
/*
 * msa_checked_violations -- diagnostics of a checked build (compiled with
 * -DMSA_CHECKED, the stand-in for a memory sanitizer): every global store of the
 * producer and projection kernels is checked against the byte range its
 * destination's descriptor implies (compact outputs: num_tokens rows; caches: up
 * to the furthest element their page count and strides reach), and a store
 * outside it is skipped and counted.  Synchronises the device, writes the count
 * of skipped stores since the last reset to *count and, if reset != 0, zeroes it.
 * A normal build returns MSA_ERR_UNSUPPORTED with *count = 0.
 */
msa_status msa_checked_violations(uint64_t *count, int32_t reset);

const char *msa_status_string(msa_status status);

/* Last detailed message of a failed check on this thread (static storage). */
const char *msa_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* MSA_PRODUCER_H */
