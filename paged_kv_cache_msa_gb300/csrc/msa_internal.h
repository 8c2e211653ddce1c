// Internal helpers shared by the library's translation units (not exported).
#pragma once

#include "msa_producer.h"

// Records a detail message for msa_last_error_detail() on this thread.
void msa_internal_set_detail(const char *msg);

// The cache-descriptor checks of msa_producer_forward (null data, dtype, head count,
// alignment, int64 extent, non-overlapping rows).
msa_status msa_internal_check_cache(const char *name, const msa_cache_desc *c, int64_t heads,
                                    int32_t head_dim, int32_t page_size);
