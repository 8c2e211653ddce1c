// Indexer for sm_103a: block scores over the index-K cache and top-k block ids.
//
// What it computes is stated in include/msa_producer.h (msa_indexer_forward),
// after "[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into one
// kernel" (the layer walk-through: proxy attention over index-K, max-reduce,
// top-16 of 128-token blocks) and "[None][perf] Fuse MiniMax-M3 QKV and index
// projection" (AFTER diagram: score visible index-K, max-pool by block, top-k).
//
// Design (decode): each query has only a handful of index heads, too few rows for
// a tensor-core tile, and its visible history is read exactly once, so the work
// is a bandwidth-bound scan on the CUDA cores.
//   * Score kernel: one CTA of 128 threads per (query, block); a thread owns one
//     token at a time, reads its index-K row with 16-byte loads (the 32 rows of a
//     warp are one contiguous run of the page), converts FP8 pairs with
//     cvt.rn.f16x2.e4m3x2, and dots them against every head with paired f32x2
//     FMAs, the query's heads being broadcast from shared memory.  The token's
//     score is the max over heads; the block's score the CTA-wide max.
//   * Top-k kernel: one warp per query; round r picks, among the entries ranked
//     strictly after round r-1's pick (score descending, id ascending), the best
//     one by a warp-wide arg-max, so nothing is marked or sorted in place.
//   * No scratch memory: block_scores is an output of the call.

#include "msa_internal.h"
#include "msa_producer.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

namespace {

constexpr int kMaxHeads = 16;
constexpr int kScoreThreads = 128;
constexpr int kTopkWarps = 4;

struct IndexerParams {
    const uint16_t *idx_q;          // [T, H, D] bf16
    const int32_t *kv_len;
    const int64_t *table_offset;
    const int32_t *page_table;
    int64_t page_table_len;
    const uint8_t *kdata;           // element 0 of the index-K cache
    int64_t num_pages;
    int64_t stride_page;            // elements
    int64_t stride_token;           // elements
    const float *k_scale;
    float *block_scores;            // [T, max_blocks]
    int32_t *topk_ids;              // [T, topk]
    int64_t num_queries;
    int32_t heads;
    int32_t fp8;
    int32_t page_size;
    int32_t page_shift;             // log2(page_size) when a power of two, else -1
    int32_t block_tokens;
    int32_t topk;
    int32_t max_blocks;
    int32_t pad;
};

__device__ __forceinline__ uint4 ldg16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// two E4M3 codes (element 0 in the low byte) -> (element 0, element 1) in fp32
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t two_codes)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_codes));
    float lo, hi;
    asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t v)
{
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// ---------------------------------------------------------------------------
// block scores
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kScoreThreads) msa_index_score_kernel(const __grid_constant__ IndexerParams p)
{
    __shared__ __align__(16) float s_q[kMaxHeads][D];
    __shared__ float s_red[kScoreThreads / 32];

    const int64_t cta = blockIdx.x;
    const int64_t t = cta / p.max_blocks;
    const int b = (int)(cta % p.max_blocks);
    const int tid = threadIdx.x;
    const int H = p.heads;

    const int64_t L = p.kv_len[t] > 0 ? (int64_t)p.kv_len[t] : 0;
    const int64_t j0 = (int64_t)b * p.block_tokens;
    float *out = p.block_scores + t * p.max_blocks + b;
    if (j0 >= L) {
        if (tid == 0)
            *out = -INFINITY;
        return;
    }
    for (int i = tid; i < H * D; i += kScoreThreads)
        s_q[i / D][i % D] = __uint_as_float(((uint32_t)p.idx_q[t * (int64_t)H * D + i]) << 16);
    __syncthreads();

    const float scale = p.fp8 ? __ldg(p.k_scale) : 1.0f;
    const int64_t jend = L < j0 + p.block_tokens ? L : j0 + p.block_tokens;
    const int64_t tbase = p.table_offset[t];
    float best = -INFINITY;
    for (int64_t j = j0 + tid; j < jend; j += kScoreThreads) {
        const int64_t ti = tbase + (p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size);
        if (ti < 0 || ti >= p.page_table_len)
            continue;
        const int64_t page = __ldg(p.page_table + ti);
        if (page < 0 || page >= p.num_pages)
            continue;
        const int64_t off = p.page_shift >= 0 ? (j & (p.page_size - 1)) : j % p.page_size;
        const int64_t e = page * p.stride_page + off * p.stride_token;

        float2 acc[kMaxHeads];
#pragma unroll
        for (int h = 0; h < kMaxHeads; ++h)
            acc[h] = make_float2(0.0f, 0.0f);
        if (p.fp8) {
            const uint8_t *row = p.kdata + e;
#pragma unroll 2
            for (int c = 0; c < D / 16; ++c) {
                const uint4 r = ldg16(row + 16 * c);
                float2 k[8];
                k[0] = e4m3x2_to_f2(r.x & 0xFFFF); k[1] = e4m3x2_to_f2(r.x >> 16);
                k[2] = e4m3x2_to_f2(r.y & 0xFFFF); k[3] = e4m3x2_to_f2(r.y >> 16);
                k[4] = e4m3x2_to_f2(r.z & 0xFFFF); k[5] = e4m3x2_to_f2(r.z >> 16);
                k[6] = e4m3x2_to_f2(r.w & 0xFFFF); k[7] = e4m3x2_to_f2(r.w >> 16);
#pragma unroll
                for (int h = 0; h < kMaxHeads; ++h) {
                    if (h < H) {
                        const float4 *qv = reinterpret_cast<const float4 *>(&s_q[h][16 * c]);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float4 qq = qv[u];
                            acc[h] = __ffma2_rn(make_float2(qq.x, qq.y), k[2 * u], acc[h]);
                            acc[h] = __ffma2_rn(make_float2(qq.z, qq.w), k[2 * u + 1], acc[h]);
                        }
                    }
                }
            }
        } else {
            const uint16_t *row = reinterpret_cast<const uint16_t *>(p.kdata) + e;
#pragma unroll 2
            for (int c = 0; c < D / 8; ++c) {
                const uint4 r = ldg16(row + 8 * c);
                const float2 k[4] = {bf16x2_to_f2(r.x), bf16x2_to_f2(r.y), bf16x2_to_f2(r.z),
                                     bf16x2_to_f2(r.w)};
#pragma unroll
                for (int h = 0; h < kMaxHeads; ++h) {
                    if (h < H) {
                        const float4 *qv = reinterpret_cast<const float4 *>(&s_q[h][8 * c]);
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const float4 qq = qv[u];
                            acc[h] = __ffma2_rn(make_float2(qq.x, qq.y), k[2 * u], acc[h]);
                            acc[h] = __ffma2_rn(make_float2(qq.z, qq.w), k[2 * u + 1], acc[h]);
                        }
                    }
                }
            }
        }
        float s = -INFINITY;
#pragma unroll
        for (int h = 0; h < kMaxHeads; ++h)
            if (h < H)
                s = fmaxf(s, acc[h].x + acc[h].y);
        best = fmaxf(best, s * scale);
    }

#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, o));
    if ((tid & 31) == 0)
        s_red[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
        float m = s_red[0];
#pragma unroll
        for (int w = 1; w < kScoreThreads / 32; ++w)
            m = fmaxf(m, s_red[w]);
        *out = m;
    }
}

// ---------------------------------------------------------------------------
// top-k block ids
// ---------------------------------------------------------------------------
// (a, ia) ranks before (b, ib): higher score first, lower id among equals.
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib)
{
    return a > b || (a == b && ia < ib);
}

__global__ void __launch_bounds__(kTopkWarps * 32) msa_index_topk_kernel(const __grid_constant__ IndexerParams p)
{
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
    if (t >= p.num_queries)
        return;  // uniform across the warp
    const float *row = p.block_scores + t * p.max_blocks;
    int32_t *out = p.topk_ids + t * p.topk;
    float prev_s = INFINITY;
    int prev_i = -1;
    int r = 0;
    for (; r < p.topk; ++r) {
        float bs = -INFINITY;
        int bi = -1;
        for (int b = lane; b < p.max_blocks; b += 32) {
            const float v = row[b];
            if (!(v > -INFINITY))      // -inf: no scored token; NaN: ignored
                continue;
            if (!ranks_before(prev_s, prev_i, v, b))
                continue;              // picked in an earlier round
            if (bi < 0 || ranks_before(v, b, bs, bi)) {
                bs = v;
                bi = b;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(0xffffffffu, bs, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (oi >= 0 && (bi < 0 || ranks_before(os, oi, bs, bi))) {
                bs = os;
                bi = oi;
            }
        }
        if (lane == 0)
            out[r] = bi;
        if (bi < 0)
            break;                     // same on every lane after the butterfly
        prev_s = bs;
        prev_i = bi;
    }
    for (int rr = r + 1 + lane; rr < p.topk; rr += 32)
        out[rr] = -1;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

msa_status fail(msa_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
msa_status fail(msa_status s, const char *fmt, ...)
{
    char buf[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    msa_internal_set_detail(buf);
    return s;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

msa_status validate(const msa_indexer_cfg *cfg, int64_t T, const void *idx_q, const int32_t *kv_len,
                    const int64_t *table_offset, const int32_t *page_table, int64_t page_table_len,
                    const msa_cache_desc *kc, const float *k_scale, float *block_scores,
                    int32_t *topk_ids)
{
    msa_internal_set_detail("");
    if (!cfg)
        return fail(MSA_ERR_INVALID_ARGUMENT, "cfg is NULL");
    if (cfg->num_heads < 1 || cfg->num_heads > kMaxHeads)
        return fail(MSA_ERR_UNSUPPORTED, "num_heads %d (1..%d)", cfg->num_heads, kMaxHeads);
    if (cfg->head_dim != 64 && cfg->head_dim != 128)
        return fail(MSA_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", cfg->head_dim);
    if (cfg->page_size <= 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "page_size %d", cfg->page_size);
    if (cfg->block_tokens < 32 || cfg->block_tokens > 1024 || cfg->block_tokens % 32)
        return fail(MSA_ERR_UNSUPPORTED, "block_tokens %d (multiple of 32, 32..1024)",
                    cfg->block_tokens);
    if (cfg->topk < 1 || cfg->topk > 64)
        return fail(MSA_ERR_UNSUPPORTED, "topk %d (1..64)", cfg->topk);
    if (cfg->max_blocks < 1 || cfg->max_blocks > 65536)
        return fail(MSA_ERR_UNSUPPORTED, "max_blocks %d (1..65536)", cfg->max_blocks);
    if (cfg->reserved[0] || cfg->reserved[1])
        return fail(MSA_ERR_INVALID_ARGUMENT, "reserved fields must be 0");
    if (T < 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "num_queries %lld", (long long)T);
    if (T == 0)
        return MSA_OK;
    if (T > (int64_t)0x7fffffff / cfg->max_blocks)
        return fail(MSA_ERR_UNSUPPORTED, "num_queries x max_blocks exceeds the grid");
    if (!idx_q || !kv_len || !table_offset || !page_table || !block_scores || !topk_ids || !kc)
        return fail(MSA_ERR_INVALID_ARGUMENT, "a required pointer is NULL");
    if (page_table_len <= 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "page_table_len %lld", (long long)page_table_len);
    if (!aligned(idx_q, 16) || !aligned(kv_len, 4) || !aligned(table_offset, 8) ||
        !aligned(page_table, 4) || !aligned(block_scores, 4) || !aligned(topk_ids, 4))
        return fail(MSA_ERR_MISALIGNED, "a buffer is misaligned");
    msa_status s = msa_internal_check_cache("idx_k_cache", kc, 1, cfg->head_dim, cfg->page_size);
    if (s != MSA_OK)
        return s;
    const int64_t es = kc->dtype == MSA_DTYPE_FP8_E4M3 ? 1 : 2;
    if ((kc->stride_page * es) % 16 || (kc->stride_token * es) % 16)
        return fail(MSA_ERR_MISALIGNED, "idx_k_cache rows must start on 16-byte boundaries");
    if (kc->dtype == MSA_DTYPE_FP8_E4M3 && (!k_scale || !aligned(k_scale, 4)))
        return fail(MSA_ERR_INVALID_ARGUMENT, "an FP8 index-K cache needs k_scale");
    return MSA_OK;
}

}  // namespace

extern "C" msa_status msa_indexer_forward(const msa_indexer_cfg *cfg, int64_t num_queries,
                                          const void *idx_q, const int32_t *kv_len,
                                          const int64_t *table_offset, const int32_t *page_table,
                                          int64_t page_table_len, const msa_cache_desc *idx_k_cache,
                                          const float *k_scale, float *block_scores,
                                          int32_t *topk_ids, cudaStream_t stream)
{
    msa_status s = validate(cfg, num_queries, idx_q, kv_len, table_offset, page_table,
                            page_table_len, idx_k_cache, k_scale, block_scores, topk_ids);
    if (s != MSA_OK || num_queries == 0)
        return s;
    IndexerParams p;
    memset(&p, 0, sizeof p);
    p.idx_q = static_cast<const uint16_t *>(idx_q);
    p.kv_len = kv_len;
    p.table_offset = table_offset;
    p.page_table = page_table;
    p.page_table_len = page_table_len;
    p.kdata = static_cast<const uint8_t *>(idx_k_cache->data);
    p.num_pages = idx_k_cache->num_pages;
    p.stride_page = idx_k_cache->stride_page;
    p.stride_token = idx_k_cache->stride_token;
    p.fp8 = idx_k_cache->dtype == MSA_DTYPE_FP8_E4M3;
    p.k_scale = k_scale;
    p.block_scores = block_scores;
    p.topk_ids = topk_ids;
    p.num_queries = num_queries;
    p.heads = cfg->num_heads;
    p.page_size = cfg->page_size;
    p.page_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == cfg->page_size)
            p.page_shift = sh;
    p.block_tokens = cfg->block_tokens;
    p.topk = cfg->topk;
    p.max_blocks = cfg->max_blocks;

    const unsigned grid_a = (unsigned)(num_queries * cfg->max_blocks);
    if (cfg->head_dim == 128)
        msa_index_score_kernel<128><<<grid_a, kScoreThreads, 0, stream>>>(p);
    else
        msa_index_score_kernel<64><<<grid_a, kScoreThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(MSA_ERR_CUDA, "score kernel launch failed: %s", cudaGetErrorString(e));
    const unsigned grid_b = (unsigned)((num_queries + kTopkWarps - 1) / kTopkWarps);
    msa_index_topk_kernel<<<grid_b, kTopkWarps * 32, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(MSA_ERR_CUDA, "top-k kernel launch failed: %s", cudaGetErrorString(e));
    return MSA_OK;
}
