// Internal helpers shared by the library's translation units (not exported).
#pragma once

#include "msa_producer.h"

#include <cuda.h>  // CUtensorMap

// Time limit of every bounded wait in the kernels (mbarrier waits), in
// nanoseconds of %globaltimer.  A build-time knob: the starved test build (below)
// sets a short one.
#ifndef MSA_WAIT_LIMIT_NS
#define MSA_WAIT_LIMIT_NS 2000000000ull
#endif

// MSA_STARVE (the starved test build only, never the product): the projection's
// TMA warps and the query-run indexer's MMA thread issue nothing, so that every
// wait on their barriers runs out; the tests check that each kernel then stops
// (the projection without writing, the indexer scoring what it could not finish
// NaN), reports the timeout and frees its tensor memory.  No copy or MMA is in
// flight when the waits give up.

// Records a detail message for msa_last_error_detail() on this thread.
void msa_internal_set_detail(const char *msg);

// The cache-descriptor checks of msa_producer_forward (null data, dtype, head count,
// alignment, int64 extent, non-overlapping rows).
msa_status msa_internal_check_cache(const char *name, const msa_cache_desc *c, int64_t heads,
                                    int32_t head_dim, int32_t page_size);

// Every check of msa_producer_forward except those of the token rows (qkv, its
// stride and the row-size limit of the producer's shared-memory ring), for entry
// points that compute the rows themselves.  Sets the detail message.
msa_status msa_internal_validate_producer(const msa_producer_cfg *cfg, int64_t num_tokens,
                                          const int32_t *positions, const int64_t *slot_mapping,
                                          const int32_t *page_table, int64_t page_table_len,
                                          const void *q_norm_w, const void *k_norm_w,
                                          const void *idx_q_norm_w, const void *idx_k_norm_w,
                                          void *q_out, void *idx_q_out,
                                          const msa_cache_desc *k_cache,
                                          const msa_cache_desc *v_cache,
                                          const msa_cache_desc *idx_k_cache, const float *scales);

// First byte past the reachable extent of a cache (the checked build's bound).
const uint8_t *msa_internal_cache_end(uint8_t *const *data, int64_t heads, int64_t num_pages,
                                      int64_t stride_page, int64_t stride_head,
                                      int64_t stride_token, int64_t elem_size, int32_t head_dim,
                                      int32_t page_size);

// Checked build: the projection kernel's violation counter (read, and optionally
// reset); synchronises the device.
msa_status msa_internal_projection_violations(uint64_t *count, int32_t reset);

// A TMA tensor map over `rows` rows of 128 bytes (8-bit elements) that start
// `stride_bytes` apart from `base`, copied `box_rows` rows per box with the 128-byte
// swizzle.  False when the driver's encoder is unavailable or rejects the layout.
bool msa_internal_encode_byte_rows(CUtensorMap *m, const void *base, int64_t rows, int64_t stride_bytes,
                                   int box_rows);
