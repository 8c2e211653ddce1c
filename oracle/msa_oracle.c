/*
 * Oracle for the MiniMax-M3 MSA per-layer fused producer and paged-cache write.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct CPU
 * definition that the CUDA path is checked against.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load it; the product
 * path never calls it and shares no code, header or table with it.
 *
 * What is computed, and where the pages say so:
 *   - "[None][perf] Fuse MiniMax-M3 QKV and index projection" (TensorRT-LLM PR
 *     18205), Description: one fused producer takes the packed projection row
 *     [Q | K | V | index-Q | index-K], applies Q/K normalisation and RoPE, emits
 *     compact Q and index-Q, and writes the current K/V and index-K into paged
 *     HND FP8 caches; it supports strided caches, 64-bit element offsets and
 *     safe containment of padded or out-of-range cache slots.
 *   - "[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into one
 *     kernel" (TensorRT-LLM PR 18614), "The problem" / "The fix": the legacy
 *     write path derives the page by division and the in-page offset by
 *     remainder from the slot, then scatters with index_put; the fused kernel
 *     computes page/offset once per token and writes K, V and index-K together.
 *   - "Wire in custom decode kernels for MinimaxM3" (TensorRT-LLM PR 18611),
 *     merge commit message: write slots are re-derived from the staged block
 *     table, so a slot can be a logical slot looked up through a page table.
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes): RMSNorm is y = x * (1/sqrt(mean(x^2) + eps)) * w with one weight
 * vector of length head_dim per tensor shared by its heads; norm comes before
 * RoPE; V gets neither; index-Q and index-K get both, with the main RoPE
 * parameters; RoPE is NeoX rotate-half (style 0) or GPT-J interleaved (style 1)
 * on the first rotary_dim dims; the cache value is enc(x * (1/scale)) with
 * round-to-nearest-even, E4M3 saturating to +-448; compact Q rows are written
 * for every token, padded ones included; only cache writes are skipped.
 *
 * Arithmetic is single precision (the precision the producer is specified in),
 * accumulated in index order, compiled without fast-math and without
 * floating-point contraction, so that x86-64 and AArch64 builds agree.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DTYPE_BF16 0
#define ORACLE_DTYPE_E4M3 1

#define ORACLE_ROPE_NEOX 0
#define ORACLE_ROPE_GPTJ 1

#define ORACLE_SCALE_PER_TENSOR 0
#define ORACLE_SCALE_PER_HEAD 1

typedef struct {
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t num_idx_q_heads;
    int32_t num_idx_k_heads;
    int32_t head_dim;
    int32_t rotary_dim;
    int32_t rope_style;
    int32_t page_size;
    float rope_theta;
    float rms_eps;
    int32_t scale_mode;
    int32_t reserved;
} oracle_shape;

typedef struct {
    uint8_t *data;      /* NULL: this cache is not written */
    int32_t dtype;      /* ORACLE_DTYPE_* */
    int32_t reserved;
    int64_t num_pages;
    int64_t num_heads;
    int64_t stride_page;   /* in elements */
    int64_t stride_head;   /* in elements */
    int64_t stride_token;  /* in elements; the dim stride is 1 */
} oracle_cache;

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bfloat16: the upper half of an IEEE binary32. */
float oracle_bf16_decode(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even.  The 16 dropped bits are
 * compared against one half of the last kept bit; overflow carries into the
 * exponent and reaches infinity, which is the correctly rounded result. */
uint16_t oracle_bf16_encode(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f))
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* FP8 E4M3 (the "fn" variant: no infinities, one NaN pattern per sign).
 * Layout s.eeee.mmm, exponent bias 7.  Exponent field 0 holds subnormals
 * m * 2^-9; fields 1..15 hold (1 + m/8) * 2^(e-7), except s.1111.111 = NaN.
 * Largest finite magnitude: s.1111.110 = 448. */
float oracle_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    float mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = ldexpf((float)m, -9);
    else
        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return s ? -mag : mag;
}

/* binary32 -> E4M3, round to nearest, ties to even, saturating: every finite or
 * infinite magnitude that rounds above 448 becomes +-448; NaN becomes 0x7F. */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    float a = fabsf(x);
    if (a >= 448.0f)
        return sign | 0x7E;
    if (a == 0.0f)
        return sign;
    int e2;
    frexpf(a, &e2);            /* a = f * 2^e2, f in [0.5, 1) */
    int E = e2 - 1;            /* a = (2f) * 2^E, 2f in [1, 2) */
    if (E < -6) {
        /* subnormal range: multiples of 2^-9; 8 * 2^-9 is the smallest normal */
        float n = rintf(ldexpf(a, 9));   /* exact scaling, then RNE to integer */
        return sign | (uint8_t)n;        /* n in [0, 8] */
    }
    float n = rintf(ldexpf(a, 3 - E));   /* in [8, 16] */
    if (n == 16.0f) {
        n = 8.0f;
        E += 1;
    }
    int field = E + 7;
    if (field > 15 || (field == 15 && n > 14.0f))
        return sign | 0x7E;
    return sign | (uint8_t)((field << 3) | ((int)n - 8));
}

/* ------------------------------------------------------------------ */
/* Per-head RMSNorm                                                    */
/* ------------------------------------------------------------------ */

/* y_i = (x_i * r) * w_i with r = 1 / sqrt(sum_j x_j^2 / D + eps); the sum is taken
 * in index order.  w == NULL means unit weight. */
void oracle_rmsnorm(const float *x, const float *w, int32_t D, float eps, float *y)
{
    float ss = 0.0f;
    for (int32_t i = 0; i < D; ++i)
        ss += x[i] * x[i];
    float r = 1.0f / sqrtf(ss / (float)D + eps);
    for (int32_t i = 0; i < D; ++i)
        y[i] = (x[i] * r) * (w ? w[i] : 1.0f);
}

/* ------------------------------------------------------------------ */
/* Rotary position embedding                                           */
/* ------------------------------------------------------------------ */

/* Frequency k of a rotary block of rd dims: theta^(-2k/rd), evaluated in double
 * and rounded once to single precision. */
static float rope_inv_freq(float theta, int32_t rd, int32_t k)
{
    return (float)(1.0 / pow((double)theta, 2.0 * (double)k / (double)rd));
}

/* Rotates the first rd dims of y (length D) in place for position pos.
 * NeoX: dim k pairs with dim k + rd/2 (k < rd/2), both at frequency k.
 * GPT-J: dim 2k pairs with dim 2k + 1, at frequency k.
 * For a pair (u, v) at angle a: u' = u cos a - v sin a, v' = v cos a + u sin a.
 * Dims at or beyond rd are left as they are. */
void oracle_rope(float *y, int32_t D, int32_t rd, int32_t style, float theta, int32_t pos)
{
    (void)D;
    int32_t half = rd / 2;
    for (int32_t k = 0; k < half; ++k) {
        float a = (float)pos * rope_inv_freq(theta, rd, k);
        float c = (float)cos((double)a);
        float s = (float)sin((double)a);
        int32_t iu = (style == ORACLE_ROPE_GPTJ) ? 2 * k : k;
        int32_t iv = (style == ORACLE_ROPE_GPTJ) ? 2 * k + 1 : k + half;
        float u = y[iu];
        float v = y[iv];
        y[iu] = u * c - v * s;
        y[iv] = v * c + u * s;
    }
}

/* ------------------------------------------------------------------ */
/* Placement: slot -> (page, in-page offset)                           */
/* ------------------------------------------------------------------ */

/* Returns 1 and sets *page, *off when slot ls lands inside a cache of num_pages
 * pages; returns 0 (nothing is written) for a padded slot (ls < 0), a logical
 * block past the page table, a table entry that is negative, or a page at or
 * beyond num_pages.  Without a table the slot is physical: page = ls / P. */
int oracle_place(int64_t ls, int32_t P, const int32_t *page_table, int64_t page_table_len,
                 int64_t num_pages, int64_t *page, int64_t *off)
{
    if (ls < 0 || P <= 0)
        return 0;
    int64_t block = ls / P;
    int64_t pg;
    if (page_table) {
        if (block >= page_table_len)
            return 0;
        pg = (int64_t)page_table[block];
    } else {
        pg = block;
    }
    if (pg < 0 || pg >= num_pages)
        return 0;
    *page = pg;
    *off = ls % P;
    return 1;
}

/* ------------------------------------------------------------------ */
/* The producer                                                        */
/* ------------------------------------------------------------------ */

static void store_cache_row(const oracle_cache *c, int64_t page, int64_t head, int64_t off,
                            const float *vals, int32_t D, float inv_scale)
{
    int64_t elem = page * c->stride_page + head * c->stride_head + off * c->stride_token;
    if (c->dtype == ORACLE_DTYPE_E4M3) {
        uint8_t *dst = c->data + elem;
        for (int32_t d = 0; d < D; ++d)
            dst[d] = oracle_e4m3_encode(vals[d] * inv_scale);
    } else {
        uint8_t *dst = c->data + 2 * elem;
        for (int32_t d = 0; d < D; ++d) {
            uint16_t h = oracle_bf16_encode(vals[d]);
            memcpy(dst + 2 * d, &h, 2);
        }
    }
}

/* Scale for head h of cache `which` (0 = K, 1 = V, 2 = index-K). */
static float cache_scale(const oracle_shape *sh, const float *scales, int which, int64_t h)
{
    if (sh->scale_mode == ORACLE_SCALE_PER_HEAD) {
        int64_t base = 0;
        if (which >= 1)
            base += sh->num_kv_heads;
        if (which >= 2)
            base += sh->num_kv_heads;
        return scales[base + h];
    }
    return scales[which];
}

/* Runs the producer over num_tokens tokens.  Buffers are host memory with the
 * same layouts the device entry point takes: qkv rows of row_stride bf16
 * elements holding [Q | K | V | idx-Q | idx-K], each section head-major [H, D];
 * q_out [T, Hq, D] and idx_q_out [T, Hiq, D] bf16, contiguous; caches addressed
 * by page * stride_page + head * stride_head + off * stride_token + dim.
 * Returns 0, or -1 for an argument the oracle cannot interpret. */
int oracle_forward(const oracle_shape *sh, int64_t num_tokens,
                   const uint16_t *qkv, int64_t row_stride,
                   const int32_t *positions, const int64_t *slot_mapping,
                   const int32_t *page_table, int64_t page_table_len,
                   const uint16_t *q_norm_w, const uint16_t *k_norm_w,
                   const uint16_t *idx_q_norm_w, const uint16_t *idx_k_norm_w,
                   uint16_t *q_out, uint16_t *idx_q_out,
                   const oracle_cache *k_cache, const oracle_cache *v_cache,
                   const oracle_cache *idx_k_cache, const float *scales)
{
    const int32_t D = sh->head_dim;
    const int32_t Hq = sh->num_q_heads, Hkv = sh->num_kv_heads;
    const int32_t Hiq = sh->num_idx_q_heads, Hik = sh->num_idx_k_heads;
    const int32_t rd = sh->rotary_dim;
    if (D <= 0 || rd < 0 || rd > D || (rd & 1) || sh->page_size <= 0)
        return -1;

    float *x = (float *)malloc(sizeof(float) * (size_t)D);
    float *y = (float *)malloc(sizeof(float) * (size_t)D);
    float *w[4];
    const uint16_t *wsrc[4] = {q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w};
    for (int i = 0; i < 4; ++i) {
        w[i] = (float *)malloc(sizeof(float) * (size_t)D);
        for (int32_t d = 0; d < D; ++d)
            w[i][d] = wsrc[i] ? oracle_bf16_decode(wsrc[i][d]) : 1.0f;
    }

    /* section order inside the row */
    const int64_t off_q = 0;
    const int64_t off_k = off_q + (int64_t)Hq * D;
    const int64_t off_v = off_k + (int64_t)Hkv * D;
    const int64_t off_iq = off_v + (int64_t)Hkv * D;
    const int64_t off_ik = off_iq + (int64_t)Hiq * D;

    for (int64_t t = 0; t < num_tokens; ++t) {
        const uint16_t *row = qkv + t * row_stride;
        const int32_t pos = positions[t];
        const int64_t ls = slot_mapping[t];

        /* Q heads: norm, RoPE, bf16, compact output (every token) */
        for (int32_t h = 0; h < Hq; ++h) {
            for (int32_t d = 0; d < D; ++d)
                x[d] = oracle_bf16_decode(row[off_q + (int64_t)h * D + d]);
            oracle_rmsnorm(x, w[0], D, sh->rms_eps, y);
            oracle_rope(y, D, rd, sh->rope_style, sh->rope_theta, pos);
            for (int32_t d = 0; d < D; ++d)
                q_out[(t * Hq + h) * D + d] = oracle_bf16_encode(y[d]);
        }
        /* index-Q heads: the same with their own weight */
        for (int32_t h = 0; h < Hiq; ++h) {
            for (int32_t d = 0; d < D; ++d)
                x[d] = oracle_bf16_decode(row[off_iq + (int64_t)h * D + d]);
            oracle_rmsnorm(x, w[2], D, sh->rms_eps, y);
            oracle_rope(y, D, rd, sh->rope_style, sh->rope_theta, pos);
            for (int32_t d = 0; d < D; ++d)
                idx_q_out[(t * Hiq + h) * D + d] = oracle_bf16_encode(y[d]);
        }

        /* cache writes: each cache takes the token only if its page is inside it */
        int64_t page, off;
        if (k_cache && k_cache->data &&
            oracle_place(ls, sh->page_size, page_table, page_table_len, k_cache->num_pages, &page, &off)) {
            for (int32_t h = 0; h < Hkv; ++h) {
                for (int32_t d = 0; d < D; ++d)
                    x[d] = oracle_bf16_decode(row[off_k + (int64_t)h * D + d]);
                oracle_rmsnorm(x, w[1], D, sh->rms_eps, y);
                oracle_rope(y, D, rd, sh->rope_style, sh->rope_theta, pos);
                store_cache_row(k_cache, page, h, off, y, D, 1.0f / cache_scale(sh, scales, 0, h));
            }
        }
        if (v_cache && v_cache->data &&
            oracle_place(ls, sh->page_size, page_table, page_table_len, v_cache->num_pages, &page, &off)) {
            for (int32_t h = 0; h < Hkv; ++h) {
                for (int32_t d = 0; d < D; ++d)
                    x[d] = oracle_bf16_decode(row[off_v + (int64_t)h * D + d]);
                store_cache_row(v_cache, page, h, off, x, D, 1.0f / cache_scale(sh, scales, 1, h));
            }
        }
        if (idx_k_cache && idx_k_cache->data &&
            oracle_place(ls, sh->page_size, page_table, page_table_len, idx_k_cache->num_pages, &page, &off)) {
            for (int32_t h = 0; h < Hik; ++h) {
                for (int32_t d = 0; d < D; ++d)
                    x[d] = oracle_bf16_decode(row[off_ik + (int64_t)h * D + d]);
                oracle_rmsnorm(x, w[3], D, sh->rms_eps, y);
                oracle_rope(y, D, rd, sh->rope_style, sh->rope_theta, pos);
                store_cache_row(idx_k_cache, page, h, off, y, D, 1.0f / cache_scale(sh, scales, 2, h));
            }
        }
    }

    for (int i = 0; i < 4; ++i)
        free(w[i]);
    free(x);
    free(y);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Indexer: block scores over the index-K cache and top-k block ids    */
/* ------------------------------------------------------------------ */
/*
 * The downstream consumer of the index-K cache ("[None][perf] Fuse MiniMax-M3
 * MSA per-layer KV-cache writes into one kernel", the layer walk-through: the
 * indexer runs a proxy attention over index-K, max-reduces, and selects the top
 * 16 of 128-token blocks; "[None][perf] Fuse MiniMax-M3 QKV and index
 * projection", AFTER diagram: score visible index-K, max-pool scores by block,
 * select top-k block ids).
 *
 * Readings: the score of visible token j for query t is max over index heads h
 * of q[t,h,:] . k[j,:] (k dequantised as code * k_scale for an FP8 cache); a
 * block's score is the max over its visible tokens; a positive softmax scale
 * would change neither max nor order and is left out.  Token j of query t is
 * visible when j < kv_len[t]; its page is page_table[table_offset[t] + j / P];
 * a token whose table entry is outside the table or the cache is skipped.
 * Blocks are block_tokens tokens; scores of blocks at or beyond the visible
 * count (or with no scored token) are -inf.  Top-k: the k highest finite block
 * scores in descending order, ties to the lower block id, padded with -1.
 */
int oracle_indexer(int32_t num_heads, int32_t head_dim, int32_t page_size, int32_t block_tokens,
                   int32_t topk, int64_t num_tokens, const uint16_t *idx_q,
                   const int32_t *kv_len, const int64_t *table_offset,
                   const int32_t *page_table, int64_t page_table_len,
                   const oracle_cache *idx_k_cache, float k_scale, int32_t max_blocks,
                   float *block_scores, int32_t *topk_out)
{
    const int32_t D = head_dim, P = page_size;
    if (D <= 0 || P <= 0 || block_tokens <= 0 || topk < 0 || max_blocks < 0 || num_heads <= 0)
        return -1;
    float *q = (float *)malloc(sizeof(float) * (size_t)num_heads * (size_t)D);
    float *k = (float *)malloc(sizeof(float) * (size_t)D);
    for (int64_t t = 0; t < num_tokens; ++t) {
        float *bs = block_scores + t * max_blocks;
        for (int32_t b = 0; b < max_blocks; ++b)
            bs[b] = -INFINITY;
        for (int32_t h = 0; h < num_heads; ++h)
            for (int32_t d = 0; d < D; ++d)
                q[h * D + d] = oracle_bf16_decode(idx_q[(t * num_heads + h) * D + d]);
        const int64_t L = kv_len[t];
        for (int64_t j = 0; j < L; ++j) {
            const int64_t b = j / block_tokens;
            if (b >= max_blocks)
                break;
            const int64_t ti = table_offset[t] + j / P;
            if (ti < 0 || ti >= page_table_len)
                continue;
            const int64_t page = page_table[ti];
            if (page < 0 || page >= idx_k_cache->num_pages)
                continue;
            const int64_t e = page * idx_k_cache->stride_page + (j % P) * idx_k_cache->stride_token;
            for (int32_t d = 0; d < D; ++d) {
                if (idx_k_cache->dtype == ORACLE_DTYPE_E4M3)
                    k[d] = oracle_e4m3_decode(idx_k_cache->data[e + d]) * k_scale;
                else {
                    uint16_t hbits;
                    memcpy(&hbits, idx_k_cache->data + 2 * (e + d), 2);
                    k[d] = oracle_bf16_decode(hbits);
                }
            }
            for (int32_t h = 0; h < num_heads; ++h) {
                float s = 0.0f;
                for (int32_t d = 0; d < D; ++d)
                    s += q[h * D + d] * k[d];
                if (s > bs[b])
                    bs[b] = s;
            }
        }
        /* top-k by repeated selection: highest score, lowest id among equals */
        int32_t *out = topk_out + t * topk;
        for (int32_t r = 0; r < topk; ++r) {
            int32_t best = -1;
            for (int32_t b = 0; b < max_blocks; ++b) {
                if (!(bs[b] > -INFINITY))
                    continue;
                int taken = 0;
                for (int32_t u = 0; u < r; ++u)
                    if (out[u] == b)
                        taken = 1;
                if (taken)
                    continue;
                if (best < 0 || bs[b] > bs[best])
                    best = b;
            }
            out[r] = best;
        }
    }
    free(q);
    free(k);
    return 0;
}

/*
 * The wide projection that feeds the producer ("[None][perf] Fuse MiniMax-M3 QKV
 * and index projection", Description, AFTER diagram: hidden states -> one wider
 * fused GEMM [Q | K | V | index-Q | index-K] -> one fused producer; the five
 * outputs come from a single quantised projection there).
 *
 *   rows[t, j] = bf16(fp32(hidden_scale[t] * weight_scale[j] *
 *                          sum_k x[t, k] * w[j, k]))            for j < width
 *
 * x and w are the decoded operands: bf16, or FP8 E4M3 codes (dtype 0 / 1, as for
 * the caches).  The weight is stored output-major ([width, hidden_size], row j is
 * the weights of output j).  The scales are the dequantisation factors of a
 * quantised projection: one per token, one per output (NULL: 1).  The sum is
 * accumulated in double in index order (a product of two bf16 or E4M3 values is
 * exact in double), multiplied by the scales in double, rounded once to fp32
 * and then to bf16 with round-to-nearest-even: the row that a GEMM with an fp32
 * accumulator stores, up to the rounding of its own accumulation and scaling.
 *
 * Readings: the pages do not say whether the fused epilogue consumes the fp32
 * accumulator or the bf16 row; the bf16 row is taken, so that projection and
 * producer together equal the unfused GEMM followed by the producer.  The pages
 * name a quantised projection without its format; per-token and per-output
 * scales over E4M3 operands are taken.
 */
static double projection_operand(const uint8_t *base, int32_t dtype, int64_t idx)
{
    if (dtype == ORACLE_DTYPE_E4M3)
        return (double)oracle_e4m3_decode(base[idx]);
    uint16_t h;
    memcpy(&h, base + 2 * idx, 2);
    return (double)oracle_bf16_decode(h);
}

int oracle_projection(int64_t num_tokens, int64_t hidden_size, int32_t dtype, const void *hidden,
                      int64_t hidden_stride, const float *hidden_scales, int64_t width,
                      const void *weight, int64_t weight_stride, const float *weight_scales,
                      uint16_t *rows, int64_t row_stride)
{
    if (num_tokens < 0 || hidden_size < 0 || width < 0 || hidden_stride < hidden_size ||
        weight_stride < hidden_size || row_stride < width ||
        (dtype != ORACLE_DTYPE_BF16 && dtype != ORACLE_DTYPE_E4M3))
        return -1;
    const uint8_t *hx = (const uint8_t *)hidden;
    const uint8_t *hw = (const uint8_t *)weight;
    for (int64_t t = 0; t < num_tokens; ++t) {
        for (int64_t j = 0; j < width; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < hidden_size; ++k)
                acc += projection_operand(hx, dtype, t * hidden_stride + k) *
                       projection_operand(hw, dtype, j * weight_stride + k);
            const double sx = hidden_scales ? (double)hidden_scales[t] : 1.0;
            const double sw = weight_scales ? (double)weight_scales[j] : 1.0;
            rows[t * row_stride + j] = oracle_bf16_encode((float)(acc * sx * sw));
        }
    }
    return 0;
}
