/*
 * msa_projection.h -- the wide [Q | K | V | index-Q | index-K] projection with the
 * MSA producer fused into its epilogue, as a C ABI.
 *
 * Source: "[None][perf] Fuse MiniMax-M3 QKV and index projection" (TensorRT-LLM
 * PR 18205), Description, BEFORE/AFTER diagrams: the separate main-QKV and
 * index-QK GEMMs become one wider GEMM whose output row is [Q | K | V | index-Q |
 * index-K], followed by one fused producer (Q/K norm + RoPE, compact Q and
 * index-Q, current K/V and index-K written to their paged caches).  Here the
 * producer runs inside the GEMM's epilogue, so the projection row never leaves
 * the chip.
 *
 * What is computed, per token t and projection output j < W, W = (Hq + 2*Hkv +
 * Hiq + Hik) * head_dim:
 *
 *     row[t, j] = bf16_rne( (sum_k hidden[t, k] * weight[j, k]) * sx[t] * sw[j] )
 *
 * with the operands bf16, or FP8 E4M3 with dequantisation scales sx (per token)
 * and sw (per output) -- the pages' projection is a quantised one; the sum is
 * accumulated in fp32 on the tensor cores and scaled as (sum * sx[t]) * sw[j] in
 * fp32 -- then exactly what msa_producer_forward
 * does to a row it reads (see msa_producer.h): the same configuration, placement,
 * norm, RoPE, compact outputs, cache encodings, scales, padded-slot containment
 * and error checks.  The result equals msa_producer_forward applied to the bf16
 * rows of the GEMM, up to the fp32 accumulation order of the GEMM.
 *
 * Ownership and threading: as for msa_producer_forward.  The library allocates
 * nothing, never synchronises, reads no device memory on the host, and the call
 * is stream-ordered and graph-capturable.
 */
#ifndef MSA_PROJECTION_H
#define MSA_PROJECTION_H

#include <stdint.h>

#include "msa_producer.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bits the kernel ORs into *status (when status is not NULL). */
#define MSA_STATUS_WAIT_TIMEOUT 1u /* a pipeline wait exceeded its time limit: outputs incomplete */

/*
 * msa_projection_forward -- one launch: projection GEMM + producer epilogue.
 *
 * cfg, num_tokens, positions, slot_mapping, page_table, page_table_len, the four
 * norm weights, q_out, idx_q_out, k_cache, v_cache, idx_k_cache, scales: exactly
 * as for msa_producer_forward (same meaning, layout, nullability and checks).
 *
 * hidden             device [num_tokens, hidden_row_stride] of operand_dtype; the
 *                    first hidden_size elements of each row are the token's hidden
 *                    state.  16-byte aligned; the row stride a multiple of 16 bytes.
 * hidden_size        K >= 1 (any value; no multiple is required).
 * weight             device [W, weight_row_stride] of operand_dtype, output-major:
 *                    row j holds the K weights of projection output j, in the
 *                    section order [Q | K | V | index-Q | index-K], each section
 *                    head-major.  16-byte aligned; the row stride a multiple of 16
 *                    bytes, >= K.
 * operand_dtype      MSA_DTYPE_BF16 or MSA_DTYPE_FP8_E4M3 (both operands).
 * hidden_scales      optional device fp32 [num_tokens]: sx (NULL: 1).
 * weight_scales      optional device fp32 [W]: sw (NULL: 1).
 * rows_out           optional (NULL: not written) device bf16 [num_tokens,
 *                    rows_out_stride]: the bf16 projection rows themselves.
 *                    16-byte aligned; rows_out_stride a multiple of 8, >= W.
 * status             optional device word; the kernel ORs MSA_STATUS_* bits into
 *                    it and never clears it (the caller zeroes it beforehand).
 * stream             the CUDA stream the launch is enqueued on.
 *
 * Limits: num_tokens < 2^31 - 128; head_dim 64 or 128.  The kernel needs a GPU
 * with tcgen05 tensor cores (sm_100 family); it is built for sm_103a.
 *
 * Errors: every argument check runs before the launch and returns a status with
 * nothing enqueued; num_tokens == 0 returns MSA_OK with no launch.  A device-side
 * wait that runs out of time (a hardware or scheduling failure, never expected)
 * makes the kernel stop, release its tensor memory and set
 * MSA_STATUS_WAIT_TIMEOUT in *status.
 */
msa_status msa_projection_forward(const msa_producer_cfg *cfg, int64_t num_tokens,
                                  const void *hidden, int64_t hidden_size,
                                  int64_t hidden_row_stride, const void *weight,
                                  int64_t weight_row_stride, msa_dtype operand_dtype,
                                  const float *hidden_scales, const float *weight_scales,
                                  const int32_t *positions,
                                  const int64_t *slot_mapping, const int32_t *page_table,
                                  int64_t page_table_len, const void *q_norm_w,
                                  const void *k_norm_w, const void *idx_q_norm_w,
                                  const void *idx_k_norm_w, void *q_out, void *idx_q_out,
                                  const msa_cache_desc *k_cache, const msa_cache_desc *v_cache,
                                  const msa_cache_desc *idx_k_cache, const float *scales,
                                  void *rows_out, int64_t rows_out_stride, uint32_t *status,
                                  cudaStream_t stream);

/*
 * msa_projection_validate -- every check msa_projection_forward makes before it
 * launches, with the same arguments minus the stream; launches nothing and never
 * touches device memory.  Returns the status msa_projection_forward would return
 * before launching.
 */
msa_status msa_projection_validate(const msa_producer_cfg *cfg, int64_t num_tokens,
                                   const void *hidden, int64_t hidden_size,
                                   int64_t hidden_row_stride, const void *weight,
                                   int64_t weight_row_stride, msa_dtype operand_dtype,
                                   const float *hidden_scales, const float *weight_scales,
                                   const int32_t *positions,
                                   const int64_t *slot_mapping, const int32_t *page_table,
                                   int64_t page_table_len, const void *q_norm_w,
                                   const void *k_norm_w, const void *idx_q_norm_w,
                                   const void *idx_k_norm_w, void *q_out, void *idx_q_out,
                                   const msa_cache_desc *k_cache, const msa_cache_desc *v_cache,
                                   const msa_cache_desc *idx_k_cache, const float *scales,
                                   void *rows_out, int64_t rows_out_stride, uint32_t *status);

#ifdef __cplusplus
}
#endif

#endif /* MSA_PROJECTION_H */
