// Indexer for sm_103a: block scores over the index-K cache and top-k block ids.
//
// What it computes is stated in include/msa_producer.h (msa_indexer_forward),
// after "[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into one
// kernel" (the layer walk-through: proxy attention over index-K, max-reduce,
// top-16 of 128-token blocks) and "[None][perf] Fuse MiniMax-M3 QKV and index
// projection" (AFTER diagram: score visible index-K, max-pool by block, top-k).
//
// Design (decode): the score is a small dense contraction per query -- its
// index heads against every visible index-K row -- and the history is read
// exactly once, so the kernel aims at the HBM roofline with the contraction on
// the tensor cores.
//   * Score kernel: a CTA of 4 warps takes 4 consecutive blocks of one query, a
//     warp one block; 8 tokens at a time it issues D/16 mma.sync m16n8k16 (heads
//     as rows, tokens as columns, fp32 accumulation).  Each lane loads one
//     contiguous quarter of its token's row with 16-byte loads; FP8 code pairs
//     become f16x2 operands with one cvt.rn.f16x2.e4m3x2.  Token score = max over
//     real heads; block score = max over visible tokens, times the FP8 scale.
//   * Top-k kernel: a CTA per query, launched programmatically dependent on the
//     score kernel.  Rows up to 1024 blocks are staged in shared memory and every
//     finite entry counts the entries ranked before it (score descending, id
//     ascending), all in parallel.  Longer rows take topk rounds of warp-wide
//     arg-max over the entries ranked after the last pick.  Large batches of short
//     rows rank up to 16 rows per CTA.
//   * No scratch memory: block_scores is an output of the call.
//
// Design (prefill, MSA_LAUNCH_QUERY_RUNS): consecutive queries of a sequence see
// the same blocks, so tiles of 16 queries (8 for more than 8 heads) are scored
// against each 128-token block on the tcgen05 tensor cores by warp-specialised
// persistent kernels with mbarrier hand-offs and bounded waits:
//   * msa_index_runs_tma_kernel (E4M3 keys of 128 dims whose pages lie on one row
//     grid): the query tile, split into E4M3 halves hi | lo, is A and the block's
//     key rows, copied by TMA (whole pages as boxes, or tile::gather4 rows), are B,
//     both in shared memory; four accumulators, two MMA warps, four epilogue groups.
//   * msa_index_runs_kernel (every other layout): the block's keys are written into
//     tensor memory from registers as A, the query tile is B in shared memory.

#include "msa_internal.h"
#include "msa_producer.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

// Groups of 8 tokens whose index-K rows a warp has in flight at once.
#ifndef MSA_INDEX_GROUPS
#define MSA_INDEX_GROUPS 4
#endif
// Resident 128-thread score CTAs per SM the register budget is sized for.
#ifndef MSA_INDEX_MIN_CTAS
#define MSA_INDEX_MIN_CTAS 4
#endif

namespace {

constexpr int kMaxHeads = 16;

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
    int32_t pdl;                    // launched with programmatic dependent launch
    int32_t *counters;              // [T] arrivals per query (single launch), else nullptr
    int32_t topk_rows;              // queries per CTA of the several-rows top-k kernel
    int64_t rows_per_page;          // stride_page / stride_token (query runs with TMA key rows)
    int32_t box_rows;               // rows of the key-row tensor map's box: a page, 128, or 1 (gather4)
};

__device__ __forceinline__ uint4 ldg16(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ---------------------------------------------------------------------------
// block scores on the tensor cores
// ---------------------------------------------------------------------------
//
// One warp scores one block: it walks the block's tokens 8 at a time and, per
// group, computes the [16 heads x 8 tokens] dot products with D/16 mma.sync
// m16n8k16 steps (fp32 accumulation).  Heads are the A rows (padded to 16 and
// masked), tokens the B columns.  Because a dot product may visit the head
// dimension in any order, step s of lane (g, i) takes dims 4s..4s+3 of the
// lane's own contiguous quarter of the row (dims [i*D/4, (i+1)*D/4)): lane i
// reads one contiguous D/4-element piece of token g's index-K row, and the same
// permutation is applied to the query when its A fragments are built.
//   FP8 cache:  two codes convert to one f16x2 operand (cvt.rn.f16x2.e4m3x2); the
//               query is rounded to f16 (exact for |q| < 65504), f16 MMA.
//   bf16 cache: the row's bf16 pairs are the operands as they are; bf16 MMA.
// The token score is the max over the real heads of its column, the block score
// the max over its visible tokens, times the FP8 scale.

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                 "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t f2_to_f16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint32_t f2_to_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// (x0, x1) -> two E4M3 codes, x0 in the low byte; round to nearest even, saturating
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float x0, float x1)
{
    unsigned short c;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(x1), "f"(x0));
    return (uint32_t)c;
}

// an f16 pair -> (low half, high half) as floats
__device__ __forceinline__ float2 f16x2_to_f2(uint32_t h2)
{
    float lo, hi;
    asm("{ .reg .b16 l, h; mov.b32 {l, h}, %2; cvt.f32.f16 %0, l; cvt.f32.f16 %1, h; }"
        : "=f"(lo), "=f"(hi)
        : "r"(h2));
    return make_float2(lo, hi);
}

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)two_codes));
    return h2;
}

// (a, ia) ranks before (b, ib): higher score first, lower id among equals.
__device__ __forceinline__ bool ranks_before(float a, int ia, float b, int ib)
{
    return a > b || (a == b && ia < ib);
}

constexpr int kTopkThreads = 128;
constexpr int kRankMaxBlocks = 1024;   // rows up to this many blocks are ranked in shared memory

// Top-k ids of one row of n block scores, by the kTopkThreads threads of a CTA.
// The row is read from global memory through L2 (ld.global.cg): in the single-launch
// indexer it holds scores that other CTAs of the same kernel wrote.
// Short rows (n <= kRankMaxBlocks) are ranked in shared memory s_row: every finite
// entry counts the entries ranked before it, all threads in parallel, and entries
// with rank < topk write their id at that rank.  When `staged`, s_row already holds
// the row; otherwise it is read from `row`.  Long rows: warp 0 takes topk rounds,
// each an arg-max over the entries ranked after the previous pick, reading `row`.
__device__ __forceinline__ void topk_row(const float *row, float *s_row, int *s_nfin, bool staged,
                                         int n, int topk, int32_t *out)
{
    const int tid = threadIdx.x, lane = tid & 31;
    if (n <= kRankMaxBlocks) {
        if (tid == 0)
            *s_nfin = 0;
        __syncthreads();
        int nfin = 0;
        const int npad = (n + 3) & ~3;
        for (int b = tid; b < npad; b += kTopkThreads) {
            const float v = b < n ? (staged ? s_row[b] : __ldcg(row + b)) : -INFINITY;
            if (!staged || b >= n)
                s_row[b] = v;
            nfin += (v > -INFINITY) ? 1 : 0;   // NaN and -inf are not candidates
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            nfin += __shfl_xor_sync(0xffffffffu, nfin, o);
        if (lane == 0)
            atomicAdd(s_nfin, nfin);
        __syncthreads();
        const float4 *r4 = reinterpret_cast<const float4 *>(s_row);
        for (int b = tid; b < n; b += kTopkThreads) {
            const float v = s_row[b];
            if (!(v > -INFINITY))
                continue;
            int rank = 0;
            for (int u4 = 0; u4 < npad / 4; ++u4) {
                const float4 w = r4[u4];
                const int u = 4 * u4;
                rank += (w.x > v || (w.x == v && u < b)) ? 1 : 0;
                rank += (w.y > v || (w.y == v && u + 1 < b)) ? 1 : 0;
                rank += (w.z > v || (w.z == v && u + 2 < b)) ? 1 : 0;
                rank += (w.w > v || (w.w == v && u + 3 < b)) ? 1 : 0;
            }
            if (rank < topk)
                out[rank] = b;
        }
        for (int r = *s_nfin + tid; r < topk; r += kTopkThreads)
            out[r] = -1;
        return;
    }

    if (tid >= 32)
        return;
    float prev_s = INFINITY;
    int prev_i = -1;
    int r = 0;
    for (; r < topk; ++r) {
        float bs = -INFINITY;
        int bi = -1;
        for (int b = lane; b < n; b += 32) {
            const float v = __ldcg(row + b);
            if (!(v > -INFINITY))
                continue;
            if (!ranks_before(prev_s, prev_i, v, b))
                continue;
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
            break;
        prev_s = bs;
        prev_i = bi;
    }
    for (int rr = r + 1 + lane; rr < topk; rr += 32)
        out[rr] = -1;
}

constexpr int kScoreWarps = 4;   // blocks per CTA (one per warp)
static_assert(kTopkThreads == kScoreWarps * 32, "a score CTA runs the top-k of the single launch");

// The single-launch indexer's top-k: every CTA of query t that scored blocks counts
// itself in counters[t] after its block scores are stored and fenced; the CTA that
// arrives last (the count of such CTAs follows from the query's length) resets the
// counter to zero for the next launch and ranks the row as the top-k kernel would,
// writing -inf past the visible history.  A query without visible tokens has no
// such CTA: its first CTA takes the row alone.  s_row: shared memory for up to
// kRankMaxBlocks scores (the score kernel's query staging, free by then).
__device__ __forceinline__ void fused_topk(const IndexerParams &p, int64_t t, int64_t L, int64_t cpq,
                                           float *s_row)
{
    __shared__ int s_last, s_nfin;
    __syncthreads();   // every warp of this CTA has stored its block score
    if (threadIdx.x == 0) {
        const int64_t span = (int64_t)kScoreWarps * p.block_tokens;
        const int64_t live = (L + span - 1) / span;   // CTAs of the query with blocks to score
        const int n_live = (int)(live < cpq ? live : cpq);
        int last = 1;
        if (n_live > 0) {
            // release: this CTA's block scores (ordered before by the barrier) are
            // visible to whoever acquires the count; acquire: the last CTA sees every
            // other CTA's
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                         : "=r"(old)
                         : "l"(p.counters + t)
                         : "memory");
            last = old == n_live - 1;
            if (last)
                p.counters[t] = 0;
        }
        s_last = last;
    }
    __syncthreads();
    if (!s_last)
        return;
    const int n = p.max_blocks;
    const int64_t nb64 = (L + p.block_tokens - 1) / p.block_tokens;
    const int nb = nb64 < n ? (int)nb64 : n;
    float *row = p.block_scores + t * n;
    for (int b = nb + (int)threadIdx.x; b < n; b += kTopkThreads)
        row[b] = -INFINITY;
    if (n <= kRankMaxBlocks) {   // stage the row, with -inf past the history
        for (int b = threadIdx.x; b < n; b += kTopkThreads)
            s_row[b] = b < nb ? __ldcg(row + b) : -INFINITY;
    } else {
        __syncthreads();   // the -inf above is in place before warp 0 reads the row
    }
    topk_row(row, s_row, &s_nfin, n <= kRankMaxBlocks, n, p.topk, p.topk_ids + t * p.topk);
}


template <int D, bool FP8>
__global__ void __launch_bounds__(kScoreWarps * 32, MSA_INDEX_MIN_CTAS) msa_index_score_kernel(const __grid_constant__ IndexerParams p)
{
    constexpr int KS = D / 16;          // mma k-steps
    __shared__ __align__(16) float s_q[16][D];
    __shared__ __align__(16) uint4 s_af[KS][32];   // A fragments of each k-step, per lane

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, i = lane & 3;
    const int cpq = (p.max_blocks + kScoreWarps - 1) / kScoreWarps;   // CTAs per query
    const int64_t t = (int64_t)blockIdx.x / cpq;
    const int b = (int)((int64_t)blockIdx.x % cpq) * kScoreWarps + warp;
    const int H = p.heads;
    // Metadata first, in one round of independent loads: under programmatic
    // dependent launch it is read before waiting on the previous kernel (kv_len,
    // table_offset and page_table must not be written by it); the query, the
    // index-K rows and every output are touched only after the wait.
    const int32_t len_raw = __ldg(p.kv_len + t);
    const int64_t tbase = __ldg(p.table_offset + t);
    const int64_t L = len_raw > 0 ? (int64_t)len_raw : 0;
    const int64_t cta_j0 = (int64_t)((int64_t)blockIdx.x % cpq) * kScoreWarps * p.block_tokens;
    // Every block of this CTA is past the visible tokens: nothing to score, and the
    // top-k writes these blocks' -inf, so the CTA leaves at once -- before the wait,
    // freeing its slot for the CTAs with work (the grid is sized for the longest
    // history).  In the single launch, a query without visible tokens has its first
    // CTA stay to write its row and ids.
    const int cta = (int)((int64_t)blockIdx.x % cpq);
    if (cta_j0 >= L && !(p.counters && L == 0 && cta == 0))
        return;
    // This warp's block, and its page-table entries, one per lane, requested before
    // the query (when the block spans at most 32 pages; otherwise each token looks
    // its page up itself).
    const int64_t j0 = (int64_t)b * p.block_tokens;
    const int64_t jend = L < j0 + p.block_tokens ? L : j0 + p.block_tokens;
    const int64_t blk0 = p.page_shift >= 0 ? (j0 >> p.page_shift) : j0 / p.page_size;
    const int64_t jlast = jend > j0 ? jend - 1 : j0;
    const int64_t blk1 = p.page_shift >= 0 ? (jlast >> p.page_shift) : jlast / p.page_size;
    const bool pages_in_lanes = blk1 - blk0 < 32;
    int64_t lane_page = -1;
    if (b < p.max_blocks && pages_in_lanes && blk0 + lane <= blk1) {
        const int64_t ti = tbase + blk0 + lane;
        if (ti >= 0 && ti < p.page_table_len)
            lane_page = __ldg(p.page_table + ti);
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // the query's heads (rows >= H zero): one 16-byte load of 8 bf16 per chunk
    constexpr int NCH = 16 * D / 8, CPT = (NCH + kScoreWarps * 32 - 1) / (kScoreWarps * 32);
    uint4 qraw[CPT];
#pragma unroll
    for (int u = 0; u < CPT; ++u) {
        const int ch = tid + u * kScoreWarps * 32;
        const int h = ch * 8 / D;
        qraw[u] = (ch < NCH && h < H) ? ldg16(p.idx_q + (t * H + h) * D + (ch * 8) % D)
                                      : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < CPT; ++u) {
        const int ch = tid + u * kScoreWarps * 32;
        if (ch < NCH) {
            float *dst = &s_q[ch * 8 / D][(ch * 8) % D];
            const uint32_t wv[4] = {qraw[u].x, qraw[u].y, qraw[u].z, qraw[u].w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                dst[2 * k] = __uint_as_float(wv[k] << 16);
                dst[2 * k + 1] = __uint_as_float(wv[k] & 0xFFFF0000u);
            }
        }
    }
    asm volatile("griddepcontrol.launch_dependents;" :::);
    __syncthreads();

    // A fragments, built once per CTA: k-step st of lane (g, i) holds rows g and g+8
    // at dims i*D/4 + 4st + {0,1} and {2,3}; warp w builds the steps st = w mod 4
    for (int st = warp; st < KS; st += kScoreWarps) {
        const int d = i * (D / 4) + 4 * st;
        const float *r0 = &s_q[g][d], *r1 = &s_q[g + 8][d];
        uint4 f;
        if (FP8) {
            f.x = f2_to_f16x2(r0[0], r0[1]);
            f.y = f2_to_f16x2(r1[0], r1[1]);
            f.z = f2_to_f16x2(r0[2], r0[3]);
            f.w = f2_to_f16x2(r1[2], r1[3]);
        } else {
            f.x = f2_to_bf16x2(r0[0], r0[1]);
            f.y = f2_to_bf16x2(r1[0], r1[1]);
            f.z = f2_to_bf16x2(r0[2], r0[3]);
            f.w = f2_to_bf16x2(r1[2], r1[3]);
        }
        s_af[st][lane] = f;
    }
    __syncthreads();
    if (b < p.max_blocks) {
        const bool row0_real = g < H, row1_real = g + 8 < H;
        if (lane_page >= p.num_pages)
            lane_page = -1;


        constexpr int NG = MSA_INDEX_GROUPS;        // token groups whose rows are in flight together
        constexpr int NWL = FP8 ? (D / 4) / 16 : (D / 4) / 8;   // 16-byte loads per lane and token
        float best = -INFINITY;
        for (int64_t jb = j0; jb < jend; jb += 8 * NG) {
            uint4 w[NG][NWL];
            bool okg[NG];
    #pragma unroll
            for (int u = 0; u < NG; ++u) {
                // this lane loads token g of group u; its columns are tokens 2i, 2i+1
                const int64_t j = jb + 8 * u + g;
                bool ok = j < jend;
                int64_t page = -1;
                if (ok) {
                    const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                    if (!pages_in_lanes) {
                        const int64_t ti = tbase + blk;
                        if (ti >= 0 && ti < p.page_table_len) {
                            const int64_t pg = __ldg(p.page_table + ti);
                            page = (pg >= 0 && pg < p.num_pages) ? pg : -1;
                        }
                    }
                    (void)blk;
                }
                if (pages_in_lanes) {
                    const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                    const int src = (int)(blk - blk0) & 31;
                    const long long pg = __shfl_sync(0xffffffffu, (long long)lane_page, src);
                    page = ok ? pg : -1;
                }
                ok = ok && page >= 0;
                okg[u] = ok;
                const int64_t off = p.page_shift >= 0 ? (j & (p.page_size - 1)) : j % p.page_size;
                const int64_t e = ok ? page * p.stride_page + off * p.stride_token : 0;
                if (FP8) {
    #pragma unroll
                    for (int v = 0; v < NWL; ++v)
                        w[u][v] = ok ? ldg16(p.kdata + e + i * (D / 4) + 16 * v) : make_uint4(0, 0, 0, 0);
                } else {
                    const uint16_t *row = reinterpret_cast<const uint16_t *>(p.kdata) + e;
    #pragma unroll
                    for (int v = 0; v < NWL; ++v)
                        w[u][v] = ok ? ldg16(row + i * (D / 4) + 8 * v) : make_uint4(0, 0, 0, 0);
                }
            }
            // the k-steps are issued step-major over the NG groups, so that consecutive
            // mma.sync are independent (group-major order would chain each on the last)
            float cc[NG][4];
    #pragma unroll
            for (int u = 0; u < NG; ++u)
                cc[u][0] = cc[u][1] = cc[u][2] = cc[u][3] = 0.0f;
    #pragma unroll
            for (int st = 0; st < KS; ++st) {
                const uint4 f = s_af[st][lane];
                const uint32_t a[4] = {f.x, f.y, f.z, f.w};
    #pragma unroll
                for (int u = 0; u < NG; ++u) {
                    const uint32_t *words = reinterpret_cast<const uint32_t *>(w[u]);
                    if (FP8)
                        mma_f16(cc[u], a, e4m3x2_to_f16x2(words[st] & 0xFFFF), e4m3x2_to_f16x2(words[st] >> 16));
                    else
                        mma_bf16(cc[u], a, words[2 * st], words[2 * st + 1]);
                }
            }
    #pragma unroll
            for (int u = 0; u < NG; ++u) {
                const float *c = cc[u];
                // columns 2i, 2i+1: max over the real heads (rows g, g+8 across lane groups)
                float m0 = fmaxf(row0_real ? c[0] : -INFINITY, row1_real ? c[2] : -INFINITY);
                float m1 = fmaxf(row0_real ? c[1] : -INFINITY, row1_real ? c[3] : -INFINITY);
    #pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    m0 = fmaxf(m0, __shfl_xor_sync(0xffffffffu, m0, o));
                    m1 = fmaxf(m1, __shfl_xor_sync(0xffffffffu, m1, o));
                }
                // a column counts only if its token was loaded (lane 8i loaded token 2i)
                const bool ok0 = __shfl_sync(0xffffffffu, okg[u], 8 * i);
                const bool ok1 = __shfl_sync(0xffffffffu, okg[u], 8 * i + 4);
                float m = fmaxf(ok0 ? m0 : -INFINITY, ok1 ? m1 : -INFINITY);
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
                best = fmaxf(best, m);
            }
        }
        if (lane == 0)
            p.block_scores[t * p.max_blocks + b] = best * (FP8 ? __ldg(p.k_scale) : 1.0f);
    }
    if (p.counters)
        fused_topk(p, t, L, cpq, &s_q[0][0]);
}

// ---------------------------------------------------------------------------
// tensor-core and barrier helpers of the query-run kernel
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// true once the phase with the given parity has completed; false after the limit
// (MSA_WAIT_LIMIT_NS, 2 s)
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try(bar, parity))
            return true;
        if ((n & 63) == 0 && globaltimer() - t0 > MSA_WAIT_LIMIT_NS)
            return false;
    }
}

// mbar_wait with the common case (the phase has already completed) inline
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity)
{
    return mbar_try(bar, parity) || mbar_wait(bar, parity);
}

// K-major operand tile in the 128-byte swizzle layout: 16-byte chunk c of row r (of
// 128 rows) at atom c / 8, row r, slot (c % 8) ^ (r % 8)
__device__ __forceinline__ uint32_t swz(uint32_t base, int r, int c)
{
    return base + (uint32_t)(c >> 3) * (128u * 128u) + (uint32_t)r * 128u +
           (uint32_t)(((c & 7) ^ (r & 7)) << 4);
}

__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;            // leading byte offset (unused with the swizzle)
    d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: 8 rows x 128 bytes
    d |= (uint64_t)1 << 46;            // descriptor version
    d |= (uint64_t)2 << 61;            // 128-byte swizzle
    return d;
}

constexpr int kTileKeys = 128;   // keys per MMA tile: the 128-token blocks of the pages

// ---------------------------------------------------------------------------
// block scores of query runs, warp-specialised (prefill)
// ---------------------------------------------------------------------------
//
// When queries come in runs of one sequence (a prefill chunk), the queries of a run
// share every index-K block they see, so a CTA scores a tile of QT consecutive
// queries (QT = 128 / HP, HP = 8 rows per query for up to 8 heads, else 16) against
// each 128-token block at once on the tcgen05 tensor cores; a tile whose queries
// belong to several sequences (different table rows) is scored one sequence at a
// time.  The FP8 keys become f16 exactly and the queries are rounded to f16, as in
// the per-query kernel; bf16 stays bf16.  The operands:
//   A (M = 128)  the 128 keys of a block: FP8 codes converted to f16 (bf16 rows as
//                they are) by the gather warps and written from registers straight
//                into tensor memory (tcgen05.st) -- no shared-memory round trip;
//   B (N = 128)  the tile's query heads (row = query * HP + head), K-major in shared
//                memory with the 128-byte swizzle, loaded once per tile;
//   D            fp32 [key, query-head] in tensor memory.
// The only shared-memory traffic per block is the MMA reading B (32 KB for D = 128);
// the earlier arrangement (queries as A, keys gathered into shared memory as B, the
// CTA's phases in lockstep) needed 96 KB per block and ran at 0.27 of the bf16 peak.
// Warps: 0 allocates tensor memory and issues the MMAs (the whole warp runs the
// loop, one elected lane issues each tcgen05 instruction); 1-8 gather
// (warps w and w + 4 share tensor-memory lane quarter w & 3 and take one half of
// the head dimension each; the rows of the next block are in flight in registers
// while the current one is converted); 9-16 epilogue, two groups of four that take
// alternate blocks, group g always reading accumulator g (thread = key of its lane
// quarter: per query, the max over its heads of the key's scores, masked by the
// key's page and the query's visible length; then the max over the block's keys,
// by a shuffle butterfly inside the warp and across the group's four warps through
// shared memory).  CTAs are persistent over the tiles.  Hand-offs are mbarriers: key
// stages (A) full / empty, accumulators full / empty, query tiles (B) full / empty.
// Every wait is bounded: after a timeout the CTA stops issuing copies and MMAs, and
// the epilogue scores every remaining visible block NaN (never selected).

constexpr int kRunsNSA = 3;            // key stages (A) in tensor memory
constexpr int kRunsNSATma = 8;         // key stages (B) in shared memory (TMA kernel): one per gather warp
constexpr int kRunsNACC = 2;           // accumulators
constexpr int kRunsThreads = 17 * 32;  // 1 MMA + 8 gather + 2 x 4 epilogue warps
constexpr uint32_t kRunsTmemCols = 512;
constexpr int kRunsDynSmem = 120 * 1024;  // two query tiles; more than half an SM: one CTA per SM
constexpr int kRunsStageBytes = 128 * 128;  // one key stage in shared memory: 128 rows of 128 E4M3 codes
constexpr int kRunsDynSmemTma = 1024 + 2 * 2 * 128 * 128 + kRunsNSATma * kRunsStageBytes;
constexpr int kRunsTmaThreads = 26 * 32;  // 2 MMA + 8 gather + 4 x 4 epilogue warps

template <int QT>
__device__ __forceinline__ float butterfly_max(float (&v)[QT], int lane)
{
    // after the level with offset o, a lane keeps the half of its values selected by
    // bit o of its lane id, combined with its partner's copy of that half
    static_assert(QT == 8 || QT == 16, "queries per tile");
#pragma unroll
    for (int o = 16, n = QT; o >= 1; o >>= 1) {
        if (n > 1) {
            const bool hi = (lane & o) != 0;
#pragma unroll
            for (int i = 0; i < QT / 2; ++i) {
                if (i < n / 2) {
                    const float send = hi ? v[i] : v[i + n / 2];
                    const float keep = hi ? v[i + n / 2] : v[i];
                    v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
                }
            }
            n /= 2;
        } else {
            v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
        }
    }
    return v[0];   // the max of query (lane >> 1) & 15 (QT 16) or (lane >> 2) & 7 (QT 8)
}

__device__ __forceinline__ void tmem_st16x(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Four rows of a byte-row tensor map (one-row boxes of 128 bytes, 128-byte swizzle)
// into four consecutive 128-byte rows of shared memory; the bytes are counted on `bar`.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, const int32_t (&row)[4],
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(map), "r"(0), "r"(row[0]), "r"(row[1]), "r"(row[2]), "r"(row[3]), "r"(bar)
        : "memory");
}

// A box of consecutive rows of a byte-row tensor map from row `row` into shared
// memory; the bytes are counted on `bar`.
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap *map, int32_t row, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(0), "r"(row), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// The segments and blocks of a tile, in the order every role walks them: one
// sequence (table row) at a time, first the one of the lowest unscored query;
// fn(seg_mask, toff, seg_len, nb) per segment.
template <int QT, typename Fn>
__device__ __forceinline__ void for_each_segment(const int32_t *len, const int64_t *toff,
                                                 int max_blocks, Fn &&fn)
{
    constexpr uint32_t all = (QT == 32) ? 0xffffffffu : ((1u << QT) - 1u);
    uint32_t done = 0;
    while (done != all) {
        const int q0 = __ffs(~done & all) - 1;
        const int64_t to = toff[q0];
        uint32_t seg = 0;
        int32_t seg_len = 0;
#pragma unroll
        for (int q = 0; q < QT; ++q)
            if (!((done >> q) & 1) && toff[q] == to) {
                seg |= 1u << q;
                seg_len = len[q] > seg_len ? len[q] : seg_len;
            }
        int nb = to == INT64_MIN ? 0 : (int)((seg_len + kTileKeys - 1) / kTileKeys);
        nb = nb > max_blocks ? max_blocks : nb;
        fn(seg, to, seg_len, nb);
        done |= seg;
    }
}

template <int D, bool FP8, int HP>
__global__ void __launch_bounds__(kRunsThreads, 1)
msa_index_runs_kernel(const __grid_constant__ IndexerParams p)
{
    constexpr int QT = 128 / HP;                           // queries per tile
    // E4M3 keys of 128 dims: the MMA takes them as stored (kind::f8f6f4, A = the raw
    // codes in tensor memory) against each query split into two E4M3 halves
    constexpr bool F8 = FP8 && D == 128;
    constexpr int NSA = kRunsNSA;
    constexpr uint32_t kBBytes = 128u * D * 2u;            // one query tile (B): f16/bf16, or E4M3 hi | lo
    constexpr int CH = D / 8;                              // 16-byte chunks of a 2-byte row
    constexpr uint32_t kACols = F8 ? D / 4 : D / 2;        // tensor-memory columns of a key stage
    constexpr uint32_t kAccCols = 128;
    constexpr uint32_t kACol0 = kRunsNACC * kAccCols;      // first key-stage column
    static_assert(kACol0 + NSA * kACols <= kRunsTmemCols, "tensor memory budget");
    constexpr uint32_t kIdesc = (1u << 4) | ((FP8 ? 0u : 1u) << 7) | ((FP8 ? 0u : 1u) << 10) |
                                ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_tile_full[2], bar_tile_empty[2];
    __shared__ __align__(8) uint64_t bar_a_full[NSA], bar_a_empty[NSA];
    __shared__ __align__(8) uint64_t bar_acc_full[kRunsNACC], bar_acc_empty[kRunsNACC];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ float s_qinv[2][QT];        // E4M3 split: 2^-e of each query's scale
    __shared__ int32_t g_len[2][QT];       // gather side's tile metadata (also read by the MMA)
    __shared__ int64_t g_toff[2][QT];
    __shared__ int32_t e_len[2][2][QT];    // each epilogue group's own copy
    __shared__ int64_t e_toff[2][2][QT];
    __shared__ float s_red[2][2][4][QT];   // [group][block parity][warp][query]
    __shared__ int s_red_ok[2][2][4];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int64_t num_tiles = (p.num_queries + QT - 1) / QT;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(smem_u32(&bar_tile_full[i])));
            // released by the eight epilogue warps and the MMA thread
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 9;" ::"r"(smem_u32(&bar_tile_empty[i])));
        }
        for (int i = 0; i < NSA; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(smem_u32(&bar_a_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_a_empty[i])));
        }
        for (int i = 0; i < kRunsNACC; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_acc_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(smem_u32(&bar_acc_empty[i])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_drain)));
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(kRunsTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;
    volatile int *abort_flag = &s_abort;

    if (warp == 0) {
        // ---------------- MMA issuer ----------------
        // The whole warp runs the loop, so that the operands stay warp-uniform, and
        // one elected lane issues each tcgen05 instruction; every wait result and
        // abort-flag read is made warp-uniform before it steers control flow.
        uint32_t tile_it = 0;
        uint32_t s = 0, ph = 0, a = 0, pa = 0;   // key stage and accumulator of the next block, with parities
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < num_tiles && ok; ti += gridDim.x, ++tile_it) {
            const uint32_t tb = tile_it & 1;
            if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                !__all_sync(0xffffffffu, mbar_wait_fast(smem_u32(&bar_tile_full[tb]), (tile_it >> 1) & 1))) {
                ok = false;
                break;
            }
            // the query tile's B descriptors, one per K step
            const uint32_t bt = bbase + tb * kBBytes;
            uint64_t bd[D / 16];
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                bd[ks] = sw128_desc(bt + (uint32_t)(ks >> 2) * (128u * 128u) + (uint32_t)(ks & 3) * 32u);
            for_each_segment<QT>(g_len[tb], g_toff[tb], p.max_blocks,
                                 [&](uint32_t, int64_t, int32_t, int nb) {
                for (int b = 0; b < nb && ok; ++b) {
                    // the abort flag is read only when a stage or accumulator is not
                    // ready yet: the ready path stays short
                    if (!__all_sync(0xffffffffu, mbar_try(smem_u32(&bar_a_full[s]), ph) &&
                                                     mbar_try(smem_u32(&bar_acc_empty[a]), pa ^ 1)) &&
                        (__any_sync(0xffffffffu, *abort_flag != 0) ||
                         !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_a_full[s]), ph) &&
                                                      mbar_wait(smem_u32(&bar_acc_empty[a]), pa ^ 1)))) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t d = tmem + a * kAccCols;
#ifndef MSA_STARVE
                    const uint32_t at0 = tmem + kACol0 + s * kACols;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        if (F8)   // K steps 0-3 against the hi halves, 4-7 against the lo halves
                            asm volatile(
                                "{\n\t.reg .pred pp, pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
                                "setp.ne.b32 pp, %4, 0;\n\t"
                                "@pe tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, pp;\n\t}" ::"r"(d),
                                "r"(at0 + (uint32_t)(ks & 3) * 8u), "l"(bd[ks]), "r"(kIdesc), "r"((uint32_t)ks)
                                : "memory");
                        else
                            asm volatile(
                                "{\n\t.reg .pred pp, pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
                                "setp.ne.b32 pp, %4, 0;\n\t"
                                "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pp;\n\t}" ::"r"(d),
                                "r"(at0 + (uint32_t)ks * 8u), "l"(bd[ks]), "r"(kIdesc), "r"((uint32_t)ks)
                                : "memory");
                    }
                    asm volatile(
                        "{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
                        "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t"
                        "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}" ::"r"(
                            smem_u32(&bar_a_empty[s])),
                        "r"(smem_u32(&bar_acc_full[a]))
                        : "memory");
#else
                    (void)d;
#endif
                    if (++s == (uint32_t)NSA) { s = 0; ph ^= 1u; }
                    if (++a == (uint32_t)kRunsNACC) { a = 0; pa ^= 1u; }
                }
            });
            __syncwarp();
            if (ok && lane == 0)   // this warp is done with the tile (its MMAs may still run)
                mbar_arrive_local(smem_u32(&bar_tile_empty[tb]));
        }
        if (!ok && lane == 0)
            *abort_flag = 1;
        // every MMA has completed before tensor memory is released
        asm volatile(
            "{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
            "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                smem_u32(&bar_drain))
            : "memory");
        (void)mbar_wait_fast(smem_u32(&bar_drain), 0);
        __syncwarp();
    } else if (warp <= 8) {
        // ---------------- gather ----------------
        const int gt = tid - 32;                    // 0..255
        const int quarter = warp & 3, half = (warp - 1) >> 2;
        const int key = quarter * 32 + lane;        // tensor-memory lane = key of the block
        constexpr int NV = FP8 ? D / 32 : D / 16;   // 16-byte pieces of half a key row
        const uint32_t a_lane = (uint32_t)(quarter * 32) << 16;
        uint32_t it = 0, tile_it = 0;
        bool stop = false;
        for (int64_t ti = blockIdx.x; ti < num_tiles; ti += gridDim.x, ++tile_it) {
            const uint32_t tb = tile_it & 1;
            stop = stop || *abort_flag ||
                   !__any_sync(0xffffffffu, mbar_wait_fast(smem_u32(&bar_tile_empty[tb]), ((tile_it >> 1) & 1) ^ 1));
            const int64_t t0 = ti * QT;
            if (!stop && gt < QT) {
                const int64_t t = t0 + gt;
                const int32_t len = t < p.num_queries ? __ldg(p.kv_len + t) : 0;
                g_len[tb][gt] = len > 0 ? len : 0;
                g_toff[tb][gt] = t < p.num_queries ? __ldg(p.table_offset + t) : INT64_MIN;
            }
            {   // the query tile: row r = (query r / HP, head r % HP), this thread's half.
                // Rows of heads past num_heads repeat head 0, so that the max over a
                // query's HP columns equals the max over its real heads.
                const int r = gt >> 1, hh = gt & 1;
                const int q = r / HP, h = r % HP;
                const int64_t t = t0 + q;
                const bool real = t < p.num_queries;
                const uint16_t *src = p.idx_q + (t * p.heads + (h < p.heads ? h : 0)) * D;
                const uint32_t bt = bbase + tb * kBBytes;
                if (F8) {
                    // The query in two E4M3 halves: x * 2^e = hi + lo, e chosen so that the
                    // query's largest |x| (over its heads and dims) lands in [128, 256), hi
                    // = x * 2^e rounded to E4M3 and lo = the remainder rounded to E4M3 (the
                    // sum is exact unless an element is below 2^-2 after scaling).  Byte d
                    // of a tile row is dim d: hi in the first 16 KB, lo in the second.
                    uint4 v[CH / 2];
                    float amax = 0.0f;
#pragma unroll
                    for (int k = 0; k < CH / 2; ++k) {
                        v[k] = (real && !stop) ? ldg16(src + 8 * (hh * (CH / 2) + k)) : make_uint4(0, 0, 0, 0);
                        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                                     fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
                    }
#pragma unroll
                    for (int o = 1; o < 2 * HP; o <<= 1)   // the query's 2 * HP threads are consecutive lanes
                        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                    int e = 0;
                    if (amax > 0.0f) {
                        e = 7 - ((int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127);   // 7 - floor(log2 amax)
                        e = e > 126 ? 126 : e;
                    }
                    const float sc = __int_as_float((e + 127) << 23);   // 2^e, e in [-120, 126]
                    if (h == 0 && hh == 0)
                        s_qinv[tb][q] = __int_as_float((127 - e) << 23);
                    uint32_t hw[16], lw[16];
#pragma unroll
                    for (int k = 0; k < CH / 2; ++k) {   // 8 dims a chunk -> 2 words of hi, 2 of lo
                        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                        for (int j = 0; j < 4; j += 2) {
                            const float x0 = __uint_as_float(w[j] << 16) * sc, x1 = __uint_as_float(w[j] & 0xFFFF0000u) * sc;
                            const float x2 = __uint_as_float(w[j + 1] << 16) * sc,
                                        x3 = __uint_as_float(w[j + 1] & 0xFFFF0000u) * sc;
                            const uint32_t h01 = e4m3x2_from_f32(x0, x1), h23 = e4m3x2_from_f32(x2, x3);
                            const float2 d01 = f16x2_to_f2(e4m3x2_to_f16x2(h01)), d23 = f16x2_to_f2(e4m3x2_to_f16x2(h23));
                            hw[2 * k + j / 2] = h01 | (h23 << 16);
                            lw[2 * k + j / 2] = e4m3x2_from_f32(x0 - d01.x, x1 - d01.y) |
                                                (e4m3x2_from_f32(x2 - d23.x, x3 - d23.y) << 16);
                        }
                    }
                    if (!stop) {
#pragma unroll
                        for (int m = 0; m < 4; ++m) {
                            sts128(swz(bt, r, 4 * hh + m), hw[4 * m], hw[4 * m + 1], hw[4 * m + 2], hw[4 * m + 3]);
                            sts128(swz(bt + 16384u, r, 4 * hh + m), lw[4 * m], lw[4 * m + 1], lw[4 * m + 2],
                                   lw[4 * m + 3]);
                        }
                    }
                } else
#pragma unroll
                for (int c = hh * (CH / 2); c < (hh + 1) * (CH / 2); ++c) {
                    if (stop)
                        break;
                    uint4 v = real ? ldg16(src + 8 * c) : make_uint4(0, 0, 0, 0);
                    if (FP8) {   // bf16 -> f16 (exact for the normal f16 range)
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                        uint32_t o[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            o[k] = f2_to_f16x2(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
                        v = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    sts128(swz(bt, r, c), v.x, v.y, v.z, v.w);
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            // publishes the tile's metadata to every gather thread and takes one stop
            // decision for all eight gather warps (a warp that stopped on its own,
            // after a wait ran out, stops them all here)
            {
                uint32_t any;
                asm volatile(
                    "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, 256, p; selp.u32 %0, 1, 0, q; }"
                    : "=r"(any)
                    : "r"((uint32_t)stop)
                    : "memory");
                if (any) {
                    *abort_flag = 1;
                    break;
                }
            }
            if (lane == 0)
                mbar_arrive_local(smem_u32(&bar_tile_full[tb]));

            for_each_segment<QT>(g_len[tb], g_toff[tb], p.max_blocks,
                                 [&](uint32_t, int64_t toff, int32_t seg_len, int nb) {
                // this thread's half row of key `key` of block bb, fetched into registers
                auto fetch = [&](int bb, uint4 (&raw)[NV]) {
                    const int64_t j = (int64_t)bb * kTileKeys + key;
                    bool okr = bb < nb && j < seg_len;
                    int64_t page = -1;
                    if (okr) {
                        const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                        const int64_t ti2 = toff + blk;
                        page = (ti2 >= 0 && ti2 < p.page_table_len) ? (int64_t)__ldg(p.page_table + ti2) : -1;
                        okr = page >= 0 && page < p.num_pages;
                    }
                    const int64_t off = p.page_shift >= 0 ? (j & (p.page_size - 1)) : j % p.page_size;
                    const uint8_t *row = okr ? p.kdata + (page * p.stride_page + off * p.stride_token) * (FP8 ? 1 : 2) +
                                                   (size_t)half * (D / 2) * (FP8 ? 1 : 2)
                                             : nullptr;
#pragma unroll
                    for (int v = 0; v < NV; ++v)
                        raw[v] = okr ? ldg16(row + 16 * v) : make_uint4(0, 0, 0, 0);
                };
                auto store = [&](const uint4 (&raw)[NV]) -> bool {
                    const uint32_t s = it % NSA, ph = (it / NSA) & 1;
                    // the abort flag is read only when the stage is not free yet
                    if (!__all_sync(0xffffffffu, mbar_try(smem_u32(&bar_a_empty[s]), ph ^ 1)) &&
                        (__any_sync(0xffffffffu, *abort_flag != 0) ||
                         !__any_sync(0xffffffffu, mbar_wait(smem_u32(&bar_a_empty[s]), ph ^ 1)))) {
                        *abort_flag = 1;
                        return false;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t taddr = tmem + a_lane + kACol0 + s * kACols + (uint32_t)half * (kACols / 2);
                    // 16 columns (32 elements) at a time, to keep few registers live
#pragma unroll
                    for (int q16 = 0; q16 < (int)(kACols / 2) / 16; ++q16) {
                        uint32_t w[32];
                        if (FP8 && !F8) {   // two 16-code pieces -> 16 f16x2 words
#pragma unroll
                            for (int vv = 0; vv < 2; ++vv) {
                                const uint4 rv = raw[2 * q16 + vv];
                                const uint32_t x[4] = {rv.x, rv.y, rv.z, rv.w};
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    w[8 * vv + 2 * k] = e4m3x2_to_f16x2(x[k] & 0xFFFF);
                                    w[8 * vv + 2 * k + 1] = e4m3x2_to_f16x2(x[k] >> 16);
                                }
                            }
                        } else {     // four pieces are 16 words already (bf16 pairs or E4M3 quads)
#pragma unroll
                            for (int vv = 0; vv < 4; ++vv) {
                                const uint4 rv = raw[4 * q16 + vv];
                                w[4 * vv] = rv.x;
                                w[4 * vv + 1] = rv.y;
                                w[4 * vv + 2] = rv.z;
                                w[4 * vv + 3] = rv.w;
                            }
                        }
                        tmem_st16x(taddr + 16u * (uint32_t)q16, w);
                    }
                    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_local(smem_u32(&bar_a_full[s]));
                    ++it;
                    return true;
                };
                if (stop || nb == 0)
                    return;
                // two register sets: the rows of block b + 1 are in flight while block b
                // is converted and stored
                uint4 ra[NV], rb[NV];
                fetch(0, ra);
                if (nb > 1)
                    fetch(1, rb);
                for (int b = 0; b < nb; b += 2) {
                    if (!store(ra)) { stop = true; return; }
                    if (b + 2 < nb)
                        fetch(b + 2, ra);
                    if (b + 1 < nb) {
                        if (!store(rb)) { stop = true; return; }
                        if (b + 3 < nb)
                            fetch(b + 3, rb);
                    }
                }
            });
        }
    } else {
        // ---------------- epilogue: two groups, alternate blocks ----------------
        const int grp = (warp - 9) >> 2;            // takes the blocks with item parity grp
        const int et = tid - (9 + 4 * grp) * 32;    // 0..127 within the group
        const int quarter = warp & 3;
        const int key = quarter * 32 + lane;
        const uint32_t d_lane = (uint32_t)(quarter * 32) << 16;
        const uint32_t acc_col = (uint32_t)grp * kAccCols;   // item parity grp -> accumulator grp
        const float kscale = FP8 ? __ldg(p.k_scale) : 1.0f;
        auto group_sync = [&]() {
            if (grp == 0)
                asm volatile("bar.sync 2, 128;" ::: "memory");
            else
                asm volatile("bar.sync 3, 128;" ::: "memory");
        };
        uint32_t it = 0, tile_it = 0;
        bool aborted = false;
        for (int64_t ti = blockIdx.x; ti < num_tiles; ti += gridDim.x, ++tile_it) {
            const uint32_t tb = tile_it & 1;
            const int64_t t0 = ti * QT;
            int32_t *elen = e_len[grp][tb];
            int64_t *etoff = e_toff[grp][tb];
            if (et < QT) {
                const int64_t t = t0 + et;
                const int32_t len = t < p.num_queries ? __ldg(p.kv_len + t) : 0;
                elen[et] = len > 0 ? len : 0;
                etoff[et] = t < p.num_queries ? __ldg(p.table_offset + t) : INT64_MIN;
            }
            if (F8 && !aborted) {
                // the query scales s_qinv[tb] are written before the gather releases the
                // tile; the tile is not reused before this group releases it
                const uint32_t par = (tile_it >> 1) & 1;
                bool ok = __all_sync(0xffffffffu, mbar_try(smem_u32(&bar_tile_full[tb]), par));
                if (!ok && !__any_sync(0xffffffffu, *abort_flag != 0))
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_tile_full[tb]), par));
                if (!ok) {
                    aborted = true;
                    *abort_flag = 1;
                }
            }
            group_sync();
            for_each_segment<QT>(elen, etoff, p.max_blocks,
                                 [&](uint32_t seg, int64_t toff, int32_t, int nb) {
                int32_t minlen = 0x7fffffff;
#pragma unroll
                for (int q = 0; q < QT; ++q)
                    if ((seg >> q) & 1)
                        minlen = elen[q] < minlen ? elen[q] : minlen;
                // this key's table entry for block bb (raw; -1 outside the table)
                auto entry = [&](int bb) -> int64_t {
                    const int64_t j = (int64_t)bb * kTileKeys + key;
                    const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                    const int64_t ti2 = toff + blk;
                    return (ti2 >= 0 && ti2 < p.page_table_len) ? (int64_t)__ldg(p.page_table + ti2) : -1;
                };
                int b = ((it & 1) == (uint32_t)grp) ? 0 : 1;     // this group's first block
                int64_t pg = b < nb ? entry(b) : -1;
                for (; b < nb; b += 2) {
                    const uint32_t its = it + (uint32_t)b;          // global item index
                    const int64_t pg_next = b + 2 < nb ? entry(b + 2) : -1;   // in flight meanwhile
                    const uint32_t pa = (its / kRunsNACC) & 1;
                    const int64_t j = (int64_t)b * kTileKeys + key;
                    const bool kvalid = pg >= 0 && pg < p.num_pages;
                    // The abort flag is read only when the accumulator is not ready yet:
                    // after an abort the MMA completes no further phase, so the first
                    // wait that follows fails and sees the flag, and `aborted` keeps
                    // every later block from trying (a later try could find an older
                    // phase of the same parity complete).
                    bool got = false;
                    if (!aborted) {
                        got = __all_sync(0xffffffffu, mbar_try(smem_u32(&bar_acc_full[grp]), pa));
                        if (!got && !__any_sync(0xffffffffu, *abort_flag != 0))
                            got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_acc_full[grp]), pa));
                        if (!got) {
                            aborted = true;
                            *abort_flag = 1;
                        }
                    }
                    float m[QT];
#pragma unroll
                    for (int q = 0; q < QT; ++q)
                        m[q] = -INFINITY;
                    if (got) {
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        // the max over a query's HP columns (padded heads repeat head 0)
#pragma unroll
                        for (int c0 = 0; c0 < 128; c0 += 32) {
                            uint32_t r[32];
                            tmem_ld32_nowait(tmem + d_lane + acc_col + (uint32_t)c0, r);
                            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
                            for (int qq = 0; qq < 32 / HP; ++qq) {
                                float x[HP];
#pragma unroll
                                for (int h = 0; h < HP; ++h)
                                    x[h] = __uint_as_float(r[qq * HP + h]);
#pragma unroll
                                for (int w2 = HP / 2; w2 > 0; w2 >>= 1)
#pragma unroll
                                    for (int h = 0; h < w2; ++h)
                                        x[h] = fmaxf(x[h], x[h + w2]);
                                m[c0 / HP + qq] = x[0];
                            }
                        }
                        // keys without a page, or not visible to a query, take no part
                        if (!__all_sync(0xffffffffu, kvalid && j < minlen)) {
#pragma unroll
                            for (int q = 0; q < QT; ++q)
                                if (!(kvalid && j < elen[q]))
                                    m[q] = -INFINITY;
                        }
                    }
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_local(smem_u32(&bar_acc_empty[grp]));
                    const float wm = butterfly_max<QT>(m, lane);
                    const int qo = QT == 16 ? ((lane >> 1) & 15) : ((lane >> 2) & 7);
                    const int rp = (int)((its >> 1) & 1);           // this group's block parity
                    if ((lane & (QT == 16 ? 1 : 3)) == 0)
                        s_red[grp][rp][quarter][qo] = wm;
                    if (lane == 0)
                        s_red_ok[grp][rp][quarter] = got ? 1 : 0;
                    group_sync();
                    if (et < QT && ((seg >> et) & 1) && t0 + et < p.num_queries) {
                        const float *rr = &s_red[grp][rp][0][0];
                        const float v = fmaxf(fmaxf(rr[et], rr[QT + et]), fmaxf(rr[2 * QT + et], rr[3 * QT + et]));
                        const int *ok4 = s_red_ok[grp][rp];
                        const bool all_got = ok4[0] & ok4[1] & ok4[2] & ok4[3];
                        const float sc = F8 ? kscale * s_qinv[tb][et] : kscale;
                        p.block_scores[(t0 + et) * p.max_blocks + b] =
                            all_got ? (v > -INFINITY ? v * sc : -INFINITY) : __int_as_float(0x7fc00000);
                    }
                    pg = pg_next;
                }
                it += (uint32_t)nb;
                // blocks the segment's queries do not reach (the two groups share them)
                const int rest = p.max_blocks - nb;
                for (int idx = et + 128 * grp; idx < QT * rest; idx += 256) {
                    const int q = idx / rest, bb = nb + idx % rest;
                    if ((seg >> q) & 1 && t0 + q < p.num_queries)
                        p.block_scores[(t0 + q) * p.max_blocks + bb] = -INFINITY;
                }
            });
            __syncwarp();
            if (lane == 0)
                mbar_arrive_local(smem_u32(&bar_tile_empty[tb]));
        }
    }

    asm volatile("griddepcontrol.launch_dependents;" :::);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kRunsTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// block scores of query runs on E4M3 keys of 128 dims, key rows gathered by TMA
// ---------------------------------------------------------------------------
//
// The tiles and segments of msa_index_runs_kernel, with the operands the other way
// round and both in shared memory (128-byte swizzle, K-major):
//   A (M = 128)  the tile's query heads (row = query * HP + head), each query split
//                into E4M3 halves hi | lo under a power-of-two scale (K steps 0-3
//                read hi, 4-7 lo), written once per tile by the gather warps;
//   B (N = 128)  the block's 128 key rows as stored (E4M3 codes), gathered into a
//                key stage by tile::gather4 copies (no register staging);
//   D            fp32 [query head, key] in tensor memory: four accumulators, block i
//                in accumulator i mod 4.
// Warps: 0 and 25 issue the MMAs of the even and the odd blocks (one elected lane of
// the whole warp issues; one warp's waits overlap the other's MMAs); 1-8 gather: the
// query tile, then key stage w - 1 each, filled with the blocks whose item index is
// w - 1 mod 8 (lane l gathers keys 4l .. 4l + 3); 9-24 epilogue, four groups of four,
// group g reading accumulator g.  Each barrier phase is waited on by one warp or
// group that also waited on the phase before it (a parity wait two phases ahead would
// see the older phase complete): stage s is consumed by MMA warp s mod 2 and
// accumulator a issued by MMA warp a mod 2 and read by epilogue group a.  An epilogue thread holds one query head's row of D: the
// max over the block's visible keys in registers, then over the query's HP heads by
// shuffles, and the query's head-0 lane writes the block score.  Key validity (a page
// in range) is a 128-bit mask each epilogue warp builds by ballot; keys past a
// query's history are cut by its length.
template <int HP>
__global__ void __launch_bounds__(kRunsTmaThreads, 1)
msa_index_runs_tma_kernel(const __grid_constant__ IndexerParams p, const __grid_constant__ CUtensorMap kmap)
{
    constexpr int QT = 128 / HP;                           // queries per tile
    constexpr int NSA = kRunsNSATma;
    constexpr int NACC = 4;
    constexpr uint32_t kAccCols = 128;
    constexpr uint32_t kQBytes = 2u * 128u * 128u;         // one query tile: hi atom | lo atom
    static_assert(NACC * kAccCols <= kRunsTmemCols, "tensor memory budget");
    // E4M3 x E4M3 -> fp32, both K-major, N = 128, M = 128
    constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_tile_full[2], bar_tile_empty[2];
    __shared__ __align__(8) uint64_t bar_k_full[NSA], bar_k_empty[NSA];
    __shared__ __align__(8) uint64_t bar_acc_full[NACC], bar_acc_empty[NACC];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ float s_qinv[2][QT];        // 2^-e of each query's scale
    __shared__ float s_amax[2][QT];        // max |x| of each query over one half of the dims
    __shared__ int32_t g_len[2][QT];       // gather side's tile metadata (also read by the MMA)
    __shared__ int64_t g_toff[2][QT];
    __shared__ int32_t e_len[4][2][QT];    // each epilogue group's own copy
    __shared__ int64_t e_toff[4][2][QT];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t qbase = (smem_u32(smem_raw) + 1023u) & ~1023u;   // two query tiles, 1024-byte aligned
    const uint32_t kbase = qbase + 2u * kQBytes;                     // the key stages
    const int64_t num_tiles = (p.num_queries + QT - 1) / QT;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(smem_u32(&bar_tile_full[i])));
            // released by the sixteen epilogue warps and the two MMA warps
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 18;" ::"r"(smem_u32(&bar_tile_empty[i])));
        }
        for (int i = 0; i < NSA; ++i) {
            // one expect-tx arrival and the copies' bytes; the MMA's commit
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_k_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_k_empty[i])));
        }
        for (int i = 0; i < NACC; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_acc_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(smem_u32(&bar_acc_empty[i])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;" ::"r"(smem_u32(&bar_drain)));
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(kRunsTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = s_tmem;
    volatile int *abort_flag = &s_abort;

    if (warp == 0 || warp == 25) {
        // ---------------- MMA issuers: warp 0 the even blocks, warp 25 the odd ones ----------------
        const uint32_t g = warp == 0 ? 0u : 1u;
        uint32_t tile_it = 0, it = 0;
        bool ok = true;
        for (int64_t ti = blockIdx.x; ti < num_tiles && ok; ti += gridDim.x, ++tile_it) {
            const uint32_t tb = tile_it & 1;
            if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                !__all_sync(0xffffffffu, mbar_wait_fast(smem_u32(&bar_tile_full[tb]), (tile_it >> 1) & 1))) {
                ok = false;
                break;
            }
            const uint64_t qd = sw128_desc(qbase + tb * kQBytes);
            for_each_segment<QT>(g_len[tb], g_toff[tb], p.max_blocks,
                                 [&](uint32_t, int64_t, int32_t, int nb) {
                for (int b = (int)((g ^ it) & 1u); b < nb && ok; b += 2) {
                    const uint32_t its = it + (uint32_t)b;   // global item index
                    const uint32_t s = its % (uint32_t)NSA, ph = (its / (uint32_t)NSA) & 1u;
                    const uint32_t a = its % (uint32_t)NACC, pa = (its / (uint32_t)NACC) & 1u;
                    if (!__all_sync(0xffffffffu, mbar_try(smem_u32(&bar_k_full[s]), ph) &&
                                                     mbar_try(smem_u32(&bar_acc_empty[a]), pa ^ 1)) &&
                        (__any_sync(0xffffffffu, *abort_flag != 0) ||
                         !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_k_full[s]), ph) &&
                                                      mbar_wait(smem_u32(&bar_acc_empty[a]), pa ^ 1)))) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    const uint32_t d = tmem + a * kAccCols;
#ifndef MSA_STARVE
                    const uint64_t kd = sw128_desc(kbase + s * (uint32_t)kRunsStageBytes);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)   // K steps 0-3: hi x keys, 4-7: lo x keys (32 bytes each)
                        asm volatile(
                            "{\n\t.reg .pred pp, pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
                            "setp.ne.b32 pp, %4, 0;\n\t"
                            "@pe tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, pp;\n\t}" ::"r"(d),
                            "l"(qd + (uint64_t)((ks >> 2) * 1024 + (ks & 3) * 2)), "l"(kd + (uint64_t)((ks & 3) * 2)),
                            "r"(kIdesc), "r"((uint32_t)ks)
                            : "memory");
                    asm volatile(
                        "{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
                        "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t"
                        "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}" ::"r"(
                            smem_u32(&bar_k_empty[s])),
                        "r"(smem_u32(&bar_acc_full[a]))
                        : "memory");
#else
                    (void)d;
#endif
                }
                it += (uint32_t)nb;
            });
            __syncwarp();
            if (ok && lane == 0)   // this warp is done with the tile (its MMAs may still run)
                mbar_arrive_local(smem_u32(&bar_tile_empty[tb]));
        }
        if (!ok && lane == 0)
            *abort_flag = 1;
        // every MMA of both warps has completed before tensor memory is released
        asm volatile(
            "{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
            "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                smem_u32(&bar_drain))
            : "memory");
        (void)mbar_wait_fast(smem_u32(&bar_drain), 0);
        __syncwarp();
    } else if (warp <= 8) {
        // ---------------- gather: query tiles into tensor memory, key rows by TMA ----------------
        const int gt = tid - 32;                    // 0..255
        const int gw = warp - 1;                    // this warp's key stage
        const int quarter = warp & 3, half = (warp - 1) >> 2;
        const int r = quarter * 32 + lane;          // tensor-memory lane = query-tile row
        const int q = r / HP, h = r % HP;
        uint32_t it = 0, tile_it = 0, uses = 0;
        bool stop = false;
        for (int64_t ti = blockIdx.x; ti < num_tiles; ti += gridDim.x, ++tile_it) {
            const uint32_t tb = tile_it & 1;
            stop = stop || *abort_flag ||
                   !__any_sync(0xffffffffu, mbar_wait_fast(smem_u32(&bar_tile_empty[tb]), ((tile_it >> 1) & 1) ^ 1));
            const int64_t t0 = ti * QT;
            if (gt == 0 && ti + gridDim.x < num_tiles) {
                // the next tile's query rows (contiguous) into L2 while this tile runs
                const int64_t n0 = (ti + gridDim.x) * QT;
                const int64_t nq = p.num_queries - n0 < QT ? p.num_queries - n0 : QT;
                asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.idx_q + n0 * p.heads * 128),
                             "r"((uint32_t)(nq * p.heads * 256))
                             : "memory");
            }
            if (!stop && gt < QT) {
                const int64_t t = t0 + gt;
                const int32_t len = t < p.num_queries ? __ldg(p.kv_len + t) : 0;
                g_len[tb][gt] = len > 0 ? len : 0;
                g_toff[tb][gt] = t < p.num_queries ? __ldg(p.table_offset + t) : INT64_MIN;
            }
            {
                // Row r = (query q, head h), this warp's half of the dims.  Rows of heads
                // past num_heads repeat head 0, so that the max over a query's HP rows
                // equals the max over its real heads.  x * 2^e = hi + lo with e chosen so
                // that the query's largest |x| (over its heads and dims) lies in
                // [128, 256), hi = x * 2^e rounded to E4M3, lo = the remainder rounded
                // to E4M3 (exact unless an element is below 2^-2 after scaling).
                const int64_t t = t0 + q;
                const bool real = t < p.num_queries && !stop;
                const uint16_t *src = p.idx_q + (t * p.heads + (h < p.heads ? h : 0)) * 128 + half * 64;
                uint4 v[8];
                float amax = 0.0f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    v[k] = real ? ldg16(src + 8 * k) : make_uint4(0, 0, 0, 0);
                    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                                 fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
                }
#pragma unroll
                for (int o = 1; o < HP; o <<= 1)   // the query's HP rows are consecutive lanes
                    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                if (h == 0)
                    s_amax[half][q] = amax;
                asm volatile("bar.sync 1, 256;" ::: "memory");
                amax = fmaxf(s_amax[0][q], s_amax[1][q]);
                int e = 0;
                if (amax > 0.0f) {
                    e = 7 - ((int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127);   // 7 - floor(log2 amax)
                    e = e > 126 ? 126 : e;
                }
                const float sc = __int_as_float((e + 127) << 23);   // 2^e, e in [-120, 126]
                if (h == 0 && half == 0)
                    s_qinv[tb][q] = __int_as_float((127 - e) << 23);
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int k = 0; k < 8; ++k) {   // 8 dims a chunk -> 2 words of hi, 2 of lo
                    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int j = 0; j < 4; j += 2) {
                        const float x0 = __uint_as_float(w[j] << 16) * sc, x1 = __uint_as_float(w[j] & 0xFFFF0000u) * sc;
                        const float x2 = __uint_as_float(w[j + 1] << 16) * sc,
                                    x3 = __uint_as_float(w[j + 1] & 0xFFFF0000u) * sc;
                        const uint32_t h01 = e4m3x2_from_f32(x0, x1), h23 = e4m3x2_from_f32(x2, x3);
                        const float2 d01 = f16x2_to_f2(e4m3x2_to_f16x2(h01)), d23 = f16x2_to_f2(e4m3x2_to_f16x2(h23));
                        hw[2 * k + j / 2] = h01 | (h23 << 16);
                        lw[2 * k + j / 2] = e4m3x2_from_f32(x0 - d01.x, x1 - d01.y) |
                                            (e4m3x2_from_f32(x2 - d23.x, x3 - d23.y) << 16);
                    }
                }
                if (!stop) {
                    // 64 dims = 16-byte chunks 4 half .. 4 half + 3 of row r, hi atom and lo atom
                    const uint32_t bt = qbase + tb * kQBytes;
#pragma unroll
                    for (int m = 0; m < 4; ++m) {
                        sts128(swz(bt, r, 4 * half + m), hw[4 * m], hw[4 * m + 1], hw[4 * m + 2], hw[4 * m + 3]);
                        sts128(swz(bt + 16384u, r, 4 * half + m), lw[4 * m], lw[4 * m + 1], lw[4 * m + 2],
                               lw[4 * m + 3]);
                    }
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            // publishes the tile's metadata to every gather thread and takes one stop
            // decision for all eight gather warps
            {
                uint32_t any;
                asm volatile(
                    "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.or.pred q, 1, 256, p; selp.u32 %0, 1, 0, q; }"
                    : "=r"(any)
                    : "r"((uint32_t)stop)
                    : "memory");
                if (any) {
                    *abort_flag = 1;
                    break;
                }
            }
            if (lane == 0)
                mbar_arrive_local(smem_u32(&bar_tile_full[tb]));

            // Key rows.  When pages are whole boxes of p.box_rows rows (a page size that
            // divides 128, or a multiple of 128), lane l < 128 / box_rows copies box l of
            // the block with one tiled copy; otherwise lane l gathers keys 4l .. 4l + 3
            // with one tile::gather4 copy.  A box or key without a page, or wholly past
            // the segment's history, reads from row 0 of the cache; the epilogue masks
            // it.  The next block's page entries load while the stage wait runs.
            const int BR = p.box_rows;
            for_each_segment<QT>(g_len[tb], g_toff[tb], p.max_blocks,
                                 [&](uint32_t, int64_t toff, int32_t seg_len, int nb) {
                if (stop)
                    return;
                // the first key of this lane's box (k = 0), or its key k, in block bb
                auto key_of = [&](int bb, int k) -> int64_t {
                    return (int64_t)bb * kTileKeys + (BR > 1 ? (int64_t)lane * BR : (int64_t)(4 * lane + k));
                };
                auto entries = [&](int bb, int32_t (&e)[4]) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int64_t j = key_of(bb, k);
                        e[k] = -1;
                        if (bb < nb && j < seg_len && (BR > 1 ? (k == 0 && lane * BR < kTileKeys) : true)) {
                            const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                            const int64_t ti2 = toff + blk;
                            if (ti2 >= 0 && ti2 < p.page_table_len)
                                e[k] = __ldg(p.page_table + ti2);
                        }
                    }
                };
                int b = (int)(((uint32_t)gw - it) & 7u);
                int32_t ec[4];
                entries(b, ec);
                for (; b < nb; b += 8) {
                    int32_t en[4];
                    entries(b + 8, en);
                    int32_t row[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int64_t j = key_of(b, k);
                        const int64_t off = p.page_shift >= 0 ? (j & (p.page_size - 1)) : j % p.page_size;
                        row[k] = (ec[k] >= 0 && (int64_t)ec[k] < p.num_pages)
                                     ? (int32_t)((int64_t)ec[k] * p.rows_per_page + off)
                                     : 0;
                    }
                    const uint32_t par = (uses & 1u) ^ 1u;
                    const uint32_t empty = smem_u32(&bar_k_empty[gw]), full = smem_u32(&bar_k_full[gw]);
                    if (!__all_sync(0xffffffffu, mbar_try(empty, par)) &&
                        (__any_sync(0xffffffffu, *abort_flag != 0) ||
                         !__all_sync(0xffffffffu, mbar_wait(empty, par)))) {
                        *abort_flag = 1;
                        stop = true;
                        return;
                    }
                    if (lane == 0)
                        mbar_expect_tx(full, (uint32_t)kRunsStageBytes);
                    __syncwarp();
                    const uint32_t st = kbase + (uint32_t)gw * (uint32_t)kRunsStageBytes;
                    if (BR > 1) {
                        if (lane * BR < kTileKeys)
                            tma_load_rows(st + (uint32_t)(lane * BR) * 128u, &kmap, row[0], full);
                    } else {
                        tma_gather4(st + (uint32_t)lane * 512u, &kmap, row, full);
                    }
                    ++uses;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ec[k] = en[k];
                }
                it += (uint32_t)nb;
            });
        }
        // this warp's copies have landed before the CTA can finish (they complete
        // whether or not the MMA consumes them)
        if (uses > 0)
            (void)__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_k_full[gw]), (uses - 1u) & 1u));
    } else {
        // ---------------- epilogue: four groups, group g the blocks in accumulator g ----------------
        const int grp = (warp - 9) >> 2;            // takes the blocks with item index grp mod 4
        const int et = tid - (9 + 4 * grp) * 32;    // 0..127 within the group
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;          // the query-tile row of this thread
        const int q = r / HP, h = r % HP;
        const uint32_t d_lane = (uint32_t)(quarter * 32) << 16;
        const float kscale = __ldg(p.k_scale);
        auto group_sync = [&]() {
            if (grp == 0)
                asm volatile("bar.sync 2, 128;" ::: "memory");
            else if (grp == 1)
                asm volatile("bar.sync 3, 128;" ::: "memory");
            else if (grp == 2)
                asm volatile("bar.sync 4, 128;" ::: "memory");
            else
                asm volatile("bar.sync 5, 128;" ::: "memory");
        };
        uint32_t it = 0, tile_it = 0;
        bool aborted = false;
        for (int64_t ti = blockIdx.x; ti < num_tiles; ti += gridDim.x, ++tile_it) {
            const uint32_t tb = tile_it & 1;
            const int64_t t0 = ti * QT;
            int32_t *elen = e_len[grp][tb];
            int64_t *etoff = e_toff[grp][tb];
            if (et < QT) {
                const int64_t t = t0 + et;
                const int32_t len = t < p.num_queries ? __ldg(p.kv_len + t) : 0;
                elen[et] = len > 0 ? len : 0;
                etoff[et] = t < p.num_queries ? __ldg(p.table_offset + t) : INT64_MIN;
            }
            if (!aborted) {
                // the query scales s_qinv[tb] are written before the gather releases the
                // tile; the tile is not reused before this group releases it
                const uint32_t par = (tile_it >> 1) & 1;
                bool ok = __all_sync(0xffffffffu, mbar_try(smem_u32(&bar_tile_full[tb]), par));
                if (!ok && !__any_sync(0xffffffffu, *abort_flag != 0))
                    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_tile_full[tb]), par));
                if (!ok) {
                    aborted = true;
                    *abort_flag = 1;
                }
            }
            group_sync();
            const float qscale = kscale * s_qinv[tb][q];
            for_each_segment<QT>(elen, etoff, p.max_blocks,
                                 [&](uint32_t seg, int64_t toff, int32_t, int nb) {
                const bool mine = ((seg >> q) & 1) && t0 + q < p.num_queries;
                const int32_t lenq = elen[q];
                // the page entries of keys 4 lane .. 4 lane + 3 of block bb (-1: none)
                auto kload = [&](int bb, int32_t (&e)[4]) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int64_t j = (int64_t)bb * kTileKeys + 4 * lane + k;
                        const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                        const int64_t ti2 = toff + blk;
                        e[k] = (bb < nb && ti2 >= 0 && ti2 < p.page_table_len) ? __ldg(p.page_table + ti2) : -1;
                    }
                };
                int b = (int)(((uint32_t)grp - it) & 3u);         // this group's first block
                int32_t ec[4];
                kload(b, ec);
                for (; b < nb; b += 4) {
                    const uint32_t its = it + (uint32_t)b;          // global item index
                    const uint32_t acc = (uint32_t)grp, pa = (its / (uint32_t)NACC) & 1u;
                    int32_t en[4];
                    kload(b + 4, en);                               // in flight meanwhile
                    // bit `lane` of word k: key 4 lane + k has a page
                    uint32_t km[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        km[k] = __ballot_sync(0xffffffffu, ec[k] >= 0 && (int64_t)ec[k] < p.num_pages);
                    // the abort flag is read only when the accumulator is not ready yet
                    bool got = false;
                    if (!aborted) {
                        got = __all_sync(0xffffffffu, mbar_try(smem_u32(&bar_acc_full[acc]), pa));
                        if (!got && !__any_sync(0xffffffffu, *abort_flag != 0))
                            got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_acc_full[acc]), pa));
                        if (!got) {
                            aborted = true;
                            *abort_flag = 1;
                        }
                    }
                    float m = -INFINITY;
                    if (got) {
                        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                        // keys of this block inside the query's history
                        const int cut = lenq - b * kTileKeys;
                        const bool all_pages = (km[0] & km[1] & km[2] & km[3]) == 0xffffffffu;
                        const bool plain = all_pages && cut >= kTileKeys;
#pragma unroll
                        for (int c0 = 0; c0 < 128; c0 += 32) {
                            uint32_t v[32];
                            tmem_ld32_nowait(tmem + d_lane + acc * kAccCols + (uint32_t)c0, v);
                            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                            if (plain) {
                                float m2[4] = {m, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    m2[i & 3] = fmaxf(m2[i & 3], __uint_as_float(v[i]));
                                m = fmaxf(fmaxf(m2[0], m2[1]), fmaxf(m2[2], m2[3]));
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    const int c = c0 + i;   // key c: word c % 4, bit c / 4
                                    if (c < cut && ((km[c & 3] >> (c >> 2)) & 1u))
                                        m = fmaxf(m, __uint_as_float(v[i]));
                                }
                            }
                        }
                    }
                    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_local(smem_u32(&bar_acc_empty[acc]));
#pragma unroll
                    for (int o = 1; o < HP; o <<= 1)   // over the query's heads
                        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (h == 0 && mine)
                        p.block_scores[(t0 + q) * p.max_blocks + b] =
                            got ? (m > -INFINITY ? m * qscale : -INFINITY) : __int_as_float(0x7fc00000);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        ec[k] = en[k];
                }
                it += (uint32_t)nb;
                // blocks the segment's queries do not reach (the four groups share them)
                const int rest = p.max_blocks - nb;
                for (int idx = et + 128 * grp; idx < QT * rest; idx += 512) {
                    const int qq = idx / rest, bb = nb + idx % rest;
                    if ((seg >> qq) & 1 && t0 + qq < p.num_queries)
                        p.block_scores[(t0 + qq) * p.max_blocks + bb] = -INFINITY;
                }
            });
            __syncwarp();
            if (lane == 0)
                mbar_arrive_local(smem_u32(&bar_tile_empty[tb]));
        }
    }

    asm volatile("griddepcontrol.launch_dependents;" :::);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 0) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kRunsTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// decode block scores on the tensor cores over a flat list of (query, block) items
// ---------------------------------------------------------------------------
//
// For E4M3 keys of 128 dims whose pages are whole TMA boxes, and batches of up to
// kDecMaxQueries queries of up to 16 index heads: one persistent CTA per SM takes an
// equal share of the batch's (query, block) items, the queries' visible blocks laid
// end to end.  Per item the MMA takes
//   A (M = 128)  the block's key rows as stored, copied by TMA into a 16 KB stage
//                (one box per page, 128-byte swizzle; a box without a page, or past
//                the history, from row 0 and masked);
//   B (N = 16)   the query's heads (rows past num_heads repeat head 0), split into
//                E4M3 halves hi | lo under a power-of-two scale as in the query-run
//                kernel: K steps 0-3 read hi, 4-7 lo;
//   D            fp32 [key, head] in 16 tensor-memory columns, eight accumulators.
// Warps: 0 copies the keys (page entries of up to 32 boxes looked up together, the
// first chunk's before waiting on the previous kernel); 1 builds the query tiles
// (three slots, one query ahead); 2 and 3 issue the MMAs of the even and the odd
// items; 4-19 are four epilogue groups, group g taking the items k with k mod 4 == g
// (and so the accumulators g and g + 4): a thread holds one key's row of 16 heads,
// its max masked by the key's page and the query's length, then the max over the
// block's keys by shuffles and across the group's four warps through shared memory.  Each barrier phase is waited on by one warp or group that also
// waited on the phase before it.  A wait that runs out scores the CTA's remaining
// items NaN.
constexpr int kDecStages = 8;
constexpr int kDecAcc = 8;
constexpr int kDecQSlots = 3;
constexpr int kDecThreads = 20 * 32;   // key-copy, query-tile, 2 MMA, 4 x 4 epilogue warps
constexpr int kDecMaxQueries = 1024;
constexpr uint32_t kDecTmemCols = 128;
constexpr int kDecQBytes = 2 * 16 * 128;   // one query tile: hi rows | lo rows
constexpr int kDecDynSmem = 1024 + kDecStages * 128 * 128 + kDecQSlots * kDecQBytes;
// the prefix scan: each thread holds kDecPasses queries, each warp scans 32 of them per pass
constexpr int kDecPasses = (kDecMaxQueries + kDecThreads - 1) / kDecThreads;
constexpr int kDecWarps = kDecThreads / 32;
static_assert(kDecThreads % 32 == 0, "whole warps");
static_assert(kDecMaxQueries <= 32 * 32, "one warp scans the chunk totals, one chunk a lane");

__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__global__ void __launch_bounds__(kDecThreads, 1)
msa_index_decode_tc_kernel(const __grid_constant__ IndexerParams p, const __grid_constant__ CUtensorMap kmap)
{
    constexpr int S = kDecStages, NA = kDecAcc, QS = kDecQSlots;
    // E4M3 x E4M3 -> fp32, both K-major, N = 16, M = 128
    constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(16 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_k_full[S], bar_k_empty[S];
    __shared__ __align__(8) uint64_t bar_acc_full[NA], bar_acc_empty[NA];
    __shared__ __align__(8) uint64_t bar_q_ready[QS], bar_q_free[QS];
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ int32_t s_pre[kDecMaxQueries + 1];   // items of the queries before q
    __shared__ int32_t s_len[kDecMaxQueries];       // kv_len, table_offset: read once, together
    __shared__ int64_t s_toff[kDecMaxQueries];
    __shared__ int32_t s_csum[kDecPasses * kDecWarps];   // items of each chunk of 32 queries
    __shared__ int64_t s_irange[2];                 // this CTA's items [i0, i1)
    __shared__ int s_qrange[2];                     // the queries of its first and last item
    __shared__ float s_qinv[QS];
    __shared__ float s_part[4][2][4];               // [group][item parity][warp of the group]
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t kbase = (smem_u32(smem_raw) + 1023u) & ~1023u;          // key stages
    const uint32_t qbase = kbase + (uint32_t)(S * kRunsStageBytes);          // query slots
    const int nq = (int)p.num_queries;                                       // <= kDecMaxQueries
    const int n = p.max_blocks;
    volatile int *abort_flag = &s_abort;

    if (tid == 0) {
        // the key map's descriptor is fetched while the lengths are read
        asm volatile("prefetch.tensormap [%0];" ::"l"(&kmap) : "memory");
        for (int i = 0; i < S; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_k_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_k_empty[i])));
        }
        for (int i = 0; i < NA; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_acc_full[i])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(smem_u32(&bar_acc_empty[i])));
        }
        for (int i = 0; i < QS; ++i) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar_q_ready[i])));
            // released by the sixteen epilogue warps and the two MMA warps (every waiter
            // of the slot's ready phase is past it before the slot is rebuilt)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 18;" ::"r"(smem_u32(&bar_q_free[i])));
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 2;" ::"r"(smem_u32(&bar_drain)));
        s_abort = 0;
        s_pre[0] = 0;
        s_qrange[0] = 0;
        s_qrange[1] = -1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(kDecTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Blocks per query and their prefix sums s_pre, in registers: thread t holds the
    // queries t and t + kDecThreads, so each warp scans 32 consecutive queries per pass
    // with shuffles and publishes the total of its chunk (chunk c = queries 32c ..
    // 32c + 31).  Lengths and table offsets are read before waiting on the previous
    // kernel, in one round of loads: every page lookup after this is one load.
    constexpr int kPasses = kDecPasses, kWarps = kDecWarps;
    int32_t nbq[kPasses], inc[kPasses];
#pragma unroll
    for (int r = 0; r < kPasses; ++r) {
        const int q = tid + r * kDecThreads;
        int32_t nb = 0;
        if (q < nq) {
            const int32_t len = __ldg(p.kv_len + q);
            s_toff[q] = __ldg(p.table_offset + q);
            s_len[q] = len;
            const int64_t nb64 = len > 0 ? ((int64_t)len + kTileKeys - 1) / kTileKeys : 0;
            nb = (int32_t)(nb64 < n ? nb64 : n);
        }
        int32_t x = nb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o)
                x += v;
        }
        nbq[r] = nb;
        inc[r] = x;
        if (lane == 31)
            s_csum[r * kWarps + warp] = x;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    {
        // every warp: the chunks' prefix (lane c holds chunk c, at most 32 chunks), the
        // total, this CTA's equal share [c0, c1) of the items; then each thread's
        // queries' bounds, and the queries holding the share's first and last item
        // (query q holds item it when s_pre[q] <= it < s_pre[q + 1])
        const int nch = (nq + 31) >> 5;
        const int32_t cs = lane < nch ? s_csum[lane] : 0;
        int32_t cinc = cs;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, cinc, o);
            if (lane >= o)
                cinc += v;
        }
        const int64_t total = __shfl_sync(0xffffffffu, cinc, 31);
        const uint64_t m0 = (uint64_t)total * blockIdx.x, m1 = m0 + (uint64_t)total;
        int64_t c0, c1;
        if (m1 <= 0xffffffffull) {   // the common case, in 32-bit arithmetic
            c0 = (uint32_t)m0 / gridDim.x;
            c1 = (uint32_t)m1 / gridDim.x;
        } else {
            c0 = (int64_t)(m0 / gridDim.x);
            c1 = (int64_t)(m1 / gridDim.x);
        }
#pragma unroll
        for (int r = 0; r < kPasses; ++r) {
            const int q = tid + r * kDecThreads;
            const int32_t pc = __shfl_sync(0xffffffffu, cinc - cs, (r * kWarps + warp) & 31);
            if (q < nq) {   // then its chunk is below nch <= 32
                const int32_t hi = pc + inc[r], lo = hi - nbq[r];
                s_pre[q + 1] = hi;
                if (c1 > c0) {
                    if (lo <= c0 && c0 < hi)
                        s_qrange[0] = q;
                    if (lo <= c1 - 1 && c1 - 1 < hi)
                        s_qrange[1] = q;
                }
            }
        }
        if (tid == 0) {
            s_irange[0] = c0;
            s_irange[1] = c1;
        }
    }
    __syncthreads();
    const uint32_t tmem = s_tmem;
    const int64_t i0 = s_irange[0], i1 = s_irange[1];
    const int q_lo = s_qrange[0], q_hi = s_qrange[1];
    // Every role waits on the previous kernel (which writes the keys and the queries)
    // before touching them; lengths, table offsets and page entries may be read before.
    auto wait_previous = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" :::);
    };

    if (warp == 0) {
        // ---------------- key copies ----------------
        // The page entries of a chunk of items are looked up together, one box per lane
        // (lane l: item l / nbox of the chunk, box l mod nbox).
        // a box is a whole page whose rows divide 128, or 128 rows: BR is a power of two
        const int BR = p.box_rows, lb = __ffs(BR) - 1, nbox = kTileKeys >> lb, ipc = 32 >> (7 - lb);
        int qc = q_lo;   // the query of the chunk's first item (items run in query order)
        // the rows of this lane's box in the chunk of items starting at c0
        auto chunk_rows = [&](int64_t c0) -> int32_t {
            while (qc + 1 < nq && s_pre[qc + 1] <= c0)
                ++qc;
            const int64_t itl = c0 + (lane >> (7 - lb));
            const int bx = lane & (nbox - 1);
            int32_t rowl = 0;
            if (itl < i1) {
                int q = qc;
                while (q + 1 < nq && s_pre[q + 1] <= itl)
                    ++q;
                const int b = (int)(itl - s_pre[q]);
                const int32_t len = s_len[q];
                const int64_t j = (int64_t)b * kTileKeys + (int64_t)bx * BR;
                if (j < len) {
                    const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                    const int64_t off = p.page_shift >= 0 ? (j & (p.page_size - 1)) : j % p.page_size;
                    const int64_t ti2 = s_toff[q] + blk;
                    if (ti2 >= 0 && ti2 < p.page_table_len) {
                        const int64_t pg = __ldg(p.page_table + ti2);
                        if (pg >= 0 && pg < p.num_pages)
                            rowl = (int32_t)(pg * p.rows_per_page + off);
                    }
                }
            }
            return rowl;
        };
        int32_t rowl = chunk_rows(i0);
        wait_previous();
        uint32_t k = 0;
        bool stop = false;
        for (int64_t c0 = i0; c0 < i1 && !stop; c0 += ipc) {
            if (c0 != i0)
                rowl = chunk_rows(c0);
            for (int x = 0; x < ipc && c0 + x < i1; ++x, ++k) {
                const uint32_t s = k % S, par = ((k / S) & 1u) ^ 1u;
                const int32_t row = __shfl_sync(0xffffffffu, rowl, (x * nbox + lane) & 31);
                const uint32_t empty = smem_u32(&bar_k_empty[s]), full = smem_u32(&bar_k_full[s]);
                if (!__all_sync(0xffffffffu, mbar_try(empty, par)) &&
                    (__any_sync(0xffffffffu, *abort_flag != 0) ||
                     !__all_sync(0xffffffffu, mbar_wait(empty, par)))) {
                    *abort_flag = 1;
                    stop = true;
                    break;
                }
                if (lane == 0)
                    mbar_expect_tx(full, (uint32_t)kRunsStageBytes);
                __syncwarp();
                if (lane < nbox)
                    tma_load_rows(kbase + s * (uint32_t)kRunsStageBytes + (uint32_t)(lane * BR) * 128u, &kmap,
                                  row, full);
            }
        }
        // every copy this warp issued has landed before the CTA finishes
        for (uint32_t s = 0; s < (uint32_t)S && s < k; ++s) {
            const uint32_t uses = (k - s + S - 1) / S;   // items issued to stage s
            (void)__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_k_full[s]), (uses - 1u) & 1u));
        }
    } else if (warp == 1) {
        // ---------------- query tiles ----------------
        wait_previous();
        const int H = p.heads;
        // the tile of the qi-th query with items (query q) into slot qi mod 3: row r =
        // head r (rows past num_heads repeat head 0), lane (r, half) the dims
        // 64 half .. 64 half + 63
        int qi = 0;
        for (int q = q_lo; q <= q_hi; ++q) {
            if (s_pre[q + 1] == s_pre[q])
                continue;   // no items (an empty history)
            const int x = qi % QS;
            if (qi >= QS) {   // the query that last used the slot has left the MMA and epilogue warps
                const uint32_t par = (uint32_t)((qi / QS - 1) & 1);
                if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                    !__all_sync(0xffffffffu, mbar_wait_fast(smem_u32(&bar_q_free[x]), par))) {
                    if (lane == 0)
                        *abort_flag = 1;
                    break;
                }
            }
            const int r = lane >> 1, half = lane & 1;
            const int h = r < H ? r : 0;
            const uint16_t *src = p.idx_q + ((int64_t)q * H + h) * 128 + half * 64;
            uint4 v[8];
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                v[c] = ldg16(src + 8 * c);
                const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[j] << 16)),
                                             fabsf(__uint_as_float(w[j] & 0xFFFF0000u))));
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            int e = 0;
            if (amax > 0.0f) {
                e = 7 - ((int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127);   // 7 - floor(log2 amax)
                e = e > 126 ? 126 : e;
            }
            const float sc = __int_as_float((e + 127) << 23);   // 2^e, e in [-120, 126]
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int c = 0; c < 8; ++c) {   // 8 dims -> 2 words of hi, 2 of lo
                const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
                for (int j = 0; j < 4; j += 2) {
                    const float x0 = __uint_as_float(w[j] << 16) * sc, x1 = __uint_as_float(w[j] & 0xFFFF0000u) * sc;
                    const float x2 = __uint_as_float(w[j + 1] << 16) * sc,
                                x3 = __uint_as_float(w[j + 1] & 0xFFFF0000u) * sc;
                    const uint32_t h01 = e4m3x2_from_f32(x0, x1), h23 = e4m3x2_from_f32(x2, x3);
                    const float2 d01 = f16x2_to_f2(e4m3x2_to_f16x2(h01)), d23 = f16x2_to_f2(e4m3x2_to_f16x2(h23));
                    hw[2 * c + j / 2] = h01 | (h23 << 16);
                    lw[2 * c + j / 2] = e4m3x2_from_f32(x0 - d01.x, x1 - d01.y) |
                                        (e4m3x2_from_f32(x2 - d23.x, x3 - d23.y) << 16);
                }
            }
            const uint32_t tile = qbase + (uint32_t)x * (uint32_t)kDecQBytes;
#pragma unroll
            for (int m = 0; m < 4; ++m) {   // chunks 4 half + m of row r (128-byte swizzle)
                const uint32_t off = (uint32_t)r * 128u + ((uint32_t)((4 * half + m) ^ (r & 7)) << 4);
                sts128(tile + off, hw[4 * m], hw[4 * m + 1], hw[4 * m + 2], hw[4 * m + 3]);
                sts128(tile + 2048u + off, lw[4 * m], lw[4 * m + 1], lw[4 * m + 2], lw[4 * m + 3]);
            }
            if (lane == 0)
                s_qinv[x] = __int_as_float((127 - e) << 23);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0)
                mbar_arrive_local(smem_u32(&bar_q_ready[x]));
            ++qi;
        }
    } else if (warp <= 3) {
        // ---------------- MMAs: warp 2 the even items, warp 3 the odd ones ----------------
        wait_previous();
        const uint32_t g = (uint32_t)(warp - 2);
        bool ok = true;
        int qi = 0;
        for (int q = q_lo; q <= q_hi && ok; ++q) {
            if (s_pre[q + 1] == s_pre[q])
                continue;   // no items (an empty history)
            const int x = qi % QS;
            // the query's tile (every query in order, so that no phase is skipped)
            if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                !__all_sync(0xffffffffu, mbar_wait_fast(smem_u32(&bar_q_ready[x]), (uint32_t)((qi / QS) & 1)))) {
                ok = false;
                break;
            }
            const uint32_t tile = qbase + (uint32_t)x * (uint32_t)kDecQBytes;
            const int64_t a0 = s_pre[q] > i0 ? s_pre[q] : i0;
            const int64_t a1 = s_pre[q + 1] < i1 ? s_pre[q + 1] : i1;
            for (int64_t it = a0 + ((uint32_t)((a0 - i0) & 1) != g ? 1 : 0); it < a1 && ok; it += 2) {
                const uint32_t k = (uint32_t)(it - i0);
                const uint32_t s = k % S, ph = (k / S) & 1u, a = k % NA, pa = (k / NA) & 1u;
                if (!__all_sync(0xffffffffu, mbar_try(smem_u32(&bar_k_full[s]), ph) &&
                                                 mbar_try(smem_u32(&bar_acc_empty[a]), pa ^ 1)) &&
                    (__any_sync(0xffffffffu, *abort_flag != 0) ||
                     !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_k_full[s]), ph) &&
                                                  mbar_wait(smem_u32(&bar_acc_empty[a]), pa ^ 1)))) {
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t d = tmem + a * 16u;
#ifndef MSA_STARVE
                const uint64_t kd = sw128_desc(kbase + s * (uint32_t)kRunsStageBytes);
                const uint64_t qd = sw128_desc(tile);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)   // K steps 0-3: keys x hi, 4-7: keys x lo (32 bytes each)
                    asm volatile(
                        "{\n\t.reg .pred pp, pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
                        "setp.ne.b32 pp, %4, 0;\n\t"
                        "@pe tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, pp;\n\t}" ::"r"(d),
                        "l"(kd + (uint64_t)((ks & 3) * 2)), "l"(qd + (uint64_t)((ks >> 2) * 128 + (ks & 3) * 2)),
                        "r"(kIdesc), "r"((uint32_t)ks)
                        : "memory");
                asm volatile(
                    "{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
                    "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t"
                    "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%1];\n\t}" ::"r"(
                        smem_u32(&bar_k_empty[s])),
                    "r"(smem_u32(&bar_acc_full[a]))
                    : "memory");
#else
                (void)d;
                (void)tile;
#endif
            }
            __syncwarp();
            if (ok && lane == 0)   // this warp is done with the query's tile (its MMAs may still run)
                mbar_arrive_local(smem_u32(&bar_q_free[x]));
            ++qi;
        }
        if (!ok && lane == 0)
            *abort_flag = 1;
        // every MMA of both warps has completed before tensor memory is released
        asm volatile(
            "{\n\t.reg .pred pe;\n\telect.sync _|pe, 0xffffffff;\n\t"
            "@pe tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                smem_u32(&bar_drain))
            : "memory");
        (void)mbar_wait_fast(smem_u32(&bar_drain), 0);
        __syncwarp();
    } else {
        // ---------------- epilogue: group g takes the items k with k mod 4 == g ----------------
        wait_previous();
        const int grp = (warp - 4) >> 2, quarter = warp & 3;
        const int key = quarter * 32 + lane;        // tensor-memory lane = key of the block
        const uint32_t d_lane = (uint32_t)(quarter * 32) << 16;
        const float kscale = __ldg(p.k_scale);
        auto group_sync = [&]() {
            if (grp == 0)
                asm volatile("bar.sync 2, 128;" ::: "memory");
            else if (grp == 1)
                asm volatile("bar.sync 3, 128;" ::: "memory");
            else if (grp == 2)
                asm volatile("bar.sync 4, 128;" ::: "memory");
            else
                asm volatile("bar.sync 5, 128;" ::: "memory");
        };
        bool aborted = false;
        int qi = 0;
        for (int q = q_lo; q <= q_hi; ++q) {
            if (s_pre[q + 1] == s_pre[q])
                continue;   // no items (an empty history)
            const int x = qi % QS;
            bool qok = false;
            if (!aborted) {
                const uint32_t par = (uint32_t)((qi / QS) & 1);
                qok = __all_sync(0xffffffffu, mbar_try(smem_u32(&bar_q_ready[x]), par));
                if (!qok && !__any_sync(0xffffffffu, *abort_flag != 0))
                    qok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_q_ready[x]), par));
                if (!qok) {
                    aborted = true;
                    *abort_flag = 1;
                }
            }
            const float qscale = qok ? kscale * s_qinv[x] : 0.0f;
            const int32_t len = s_len[q];
            const int64_t toff = s_toff[q];
            const int64_t a0 = s_pre[q] > i0 ? s_pre[q] : i0;
            const int64_t a1 = s_pre[q + 1] < i1 ? s_pre[q + 1] : i1;
            // this key's page entry in item itx of the query (-1: none), one item ahead
            auto page_of = [&](int64_t itx) -> int32_t {
                if (itx >= a1)
                    return -1;
                const int64_t j = (itx - s_pre[q]) * kTileKeys + key;
                if (j >= len)
                    return -1;
                const int64_t blk = p.page_shift >= 0 ? (j >> p.page_shift) : j / p.page_size;
                const int64_t ti2 = toff + blk;
                return (ti2 >= 0 && ti2 < p.page_table_len) ? __ldg(p.page_table + ti2) : -1;
            };
            int64_t it = a0 + (int64_t)(((uint32_t)grp - (uint32_t)(a0 - i0)) & 3u);
            int32_t pgc = page_of(it);
            for (; it < a1; it += 4) {
                const uint32_t k = (uint32_t)(it - i0);
                const uint32_t a = k % NA, pa = (k / NA) & 1u;
                const int b = (int)(it - s_pre[q]);
                const int32_t pgn = page_of(it + 4);   // in flight meanwhile
                bool got = false;
                if (!aborted) {
                    got = __all_sync(0xffffffffu, mbar_try(smem_u32(&bar_acc_full[a]), pa));
                    if (!got && !__any_sync(0xffffffffu, *abort_flag != 0))
                        got = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bar_acc_full[a]), pa));
                    if (!got) {
                        aborted = true;
                        *abort_flag = 1;
                    }
                }
                float m = -INFINITY;
                if (got) {
                    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                    uint32_t v[16];
                    tmem_ld16_nowait(tmem + d_lane + a * 16u, v);
                    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    float m2[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                    for (int c = 0; c < 16; ++c)   // the max over the heads (rows past them repeat head 0)
                        m2[c & 3] = fmaxf(m2[c & 3], __uint_as_float(v[c]));
                    const bool kvalid = pgc >= 0 && (int64_t)pgc < p.num_pages;
                    m = kvalid ? fmaxf(fmaxf(m2[0], m2[1]), fmaxf(m2[2], m2[3])) : -INFINITY;
                }
                asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_local(smem_u32(&bar_acc_empty[a]));
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                const int buf = (int)((k >> 2) & 1u);
                if (lane == 0)
                    s_part[grp][buf][quarter] = got ? m : __int_as_float(0x7fc00000);
                group_sync();
                if (quarter == 0 && lane == 0) {
                    const float *pp = s_part[grp][buf];
                    const bool bad = isnan(pp[0]) || isnan(pp[1]) || isnan(pp[2]) || isnan(pp[3]);
                    const float vmax = fmaxf(fmaxf(pp[0], pp[1]), fmaxf(pp[2], pp[3]));
                    p.block_scores[(int64_t)q * n + b] =
                        bad ? __int_as_float(0x7fc00000) : (vmax > -INFINITY ? vmax * qscale : -INFINITY);
                }
                pgc = pgn;
            }
            __syncwarp();
            if (lane == 0)   // this warp is done with the query's tile
                mbar_arrive_local(smem_u32(&bar_q_free[x]));
            ++qi;
        }
    }

    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 2) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kDecTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// top-k block ids
// ---------------------------------------------------------------------------
// One CTA per query, after a score kernel; under programmatic dependent launch it
// waits for the score kernel before reading its output.
__global__ void __launch_bounds__(kTopkThreads) msa_index_topk_kernel(const __grid_constant__ IndexerParams p)
{
    __shared__ __align__(16) float s_row[kRankMaxBlocks];
    __shared__ int s_nfin;
    const int64_t t = blockIdx.x;
    const int n = p.max_blocks;
    // blocks from nb on hold no visible token: the per-query score kernel does not
    // write them (its CTAs past the history leave at once), this kernel does
    const int32_t len_raw = __ldg(p.kv_len + t);
    const int64_t L = len_raw > 0 ? (int64_t)len_raw : 0;
    const int64_t nb64 = (L + p.block_tokens - 1) / p.block_tokens;
    const int nb = nb64 < n ? (int)nb64 : n;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // The next kernel may start its prologue once this grid has waited: every kernel
    // before this one has completed by then (see the producer's kernel for why the
    // signal comes after the wait).
    asm volatile("griddepcontrol.launch_dependents;" :::);
    float *row = p.block_scores + t * n;
    for (int b = nb + (int)threadIdx.x; b < n; b += kTopkThreads)
        row[b] = -INFINITY;
    if (n <= kRankMaxBlocks) {   // stage the row, with -inf past the history
        for (int b = threadIdx.x; b < n; b += kTopkThreads)
            s_row[b] = b < nb ? row[b] : -INFINITY;
    } else {
        __syncthreads();   // the -inf above is in place before warp 0 reads the row
    }
    topk_row(row, s_row, &s_nfin, n <= kRankMaxBlocks, n, p.topk, p.topk_ids + t * p.topk);
}

constexpr int kTopkRowsMax = 16;            // queries per CTA of the several-rows kernel
constexpr int64_t kTopkRowsMinQueries = 2048;  // batches that take it (each CTA then does more)

// The top-k of topk_rows consecutive queries per CTA, for large batches of short
// rows (topk_rows x max_blocks <= kRankMaxBlocks): the CTA writes -inf past each
// query's history, stages the rows (contiguous in block_scores) together, and every
// finite entry counts the entries of its row ranked before it, all rows at once --
// the rule of topk_row; ranks past a row's finite entries take -1.  One CTA per
// query would leave each of them mostly waiting on its loads, in dozens of waves.
__global__ void __launch_bounds__(kTopkThreads) msa_index_topk_rows_kernel(const __grid_constant__ IndexerParams p)
{
    __shared__ __align__(16) float s_row[kRankMaxBlocks];
    __shared__ int s_nb[kTopkRowsMax], s_nfin[kTopkRowsMax];
    const int n = p.max_blocks, topk = p.topk, tid = threadIdx.x;
    const int64_t q0 = (int64_t)blockIdx.x * p.topk_rows;
    const int64_t left = p.num_queries - q0;
    const int nq = left < p.topk_rows ? (int)left : p.topk_rows;
    if (tid < nq) {
        const int32_t len_raw = __ldg(p.kv_len + q0 + tid);
        const int64_t L = len_raw > 0 ? (int64_t)len_raw : 0;
        const int64_t nb64 = (L + p.block_tokens - 1) / p.block_tokens;
        s_nb[tid] = nb64 < n ? (int)nb64 : n;
        s_nfin[tid] = 0;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" :::);
    __syncthreads();
    float *rows = p.block_scores + q0 * n;
    for (int idx = tid; idx < nq * n; idx += kTopkThreads) {
        const int r = idx / n, b = idx - r * n;
        float v = -INFINITY;
        if (b < s_nb[r])
            v = rows[idx];
        else
            rows[idx] = -INFINITY;
        s_row[idx] = v;
    }
    __syncthreads();
    for (int idx = tid; idx < nq * n; idx += kTopkThreads) {
        const float v = s_row[idx];
        if (!(v > -INFINITY))   // NaN and -inf are not candidates
            continue;
        const int r = idx / n, b = idx - r * n;
        atomicAdd(&s_nfin[r], 1);
        const float *row = s_row + r * n;
        int rank = 0;
        // entries past the row's history are -inf and never rank before a candidate
        const int nb = s_nb[r];
        if ((n & 3) == 0) {   // rows start on 16-byte boundaries: four entries a load
            const float4 *r4 = reinterpret_cast<const float4 *>(row);
            for (int u4 = 0; u4 < (nb + 3) / 4; ++u4) {
                const float4 w = r4[u4];
                const int u = 4 * u4;
                rank += (w.x > v || (w.x == v && u < b)) ? 1 : 0;
                rank += (w.y > v || (w.y == v && u + 1 < b)) ? 1 : 0;
                rank += (w.z > v || (w.z == v && u + 2 < b)) ? 1 : 0;
                rank += (w.w > v || (w.w == v && u + 3 < b)) ? 1 : 0;
            }
        } else {
            for (int u = 0; u < nb; ++u) {
                const float w = row[u];
                rank += (w > v || (w == v && u < b)) ? 1 : 0;
            }
        }
        if (rank < topk)
            p.topk_ids[(q0 + r) * topk + rank] = b;
    }
    __syncthreads();
    for (int idx = tid; idx < nq * topk; idx += kTopkThreads) {
        const int r = idx / topk, k = idx - r * topk;
        if (k >= s_nfin[r])
            p.topk_ids[(q0 + r) * topk + k] = -1;
    }
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
                    int32_t *topk_ids, int32_t flags)
{
    msa_internal_set_detail("");
    if (!cfg)
        return fail(MSA_ERR_INVALID_ARGUMENT, "cfg is NULL");
    if (flags & ~(MSA_LAUNCH_PDL | MSA_LAUNCH_QUERY_RUNS))
        return fail(MSA_ERR_INVALID_ARGUMENT,
                    "launch flags 0x%x (MSA_LAUNCH_PDL, MSA_LAUNCH_QUERY_RUNS)", flags);
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

// The launches of both entry points; counters != nullptr: the per-query kernel takes
// the top-k itself (the query-run path keeps its top-k kernel).
msa_status indexer_launch(const msa_indexer_cfg *cfg, int64_t num_queries, const void *idx_q,
                          const int32_t *kv_len, const int64_t *table_offset,
                          const int32_t *page_table, int64_t page_table_len,
                          const msa_cache_desc *idx_k_cache, const float *k_scale,
                          float *block_scores, int32_t *topk_ids, int32_t *counters,
                          int32_t launch_flags, cudaStream_t stream)
{
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
    p.pdl = (launch_flags & MSA_LAUNCH_PDL) ? 1 : 0;

    const bool tiled = (launch_flags & MSA_LAUNCH_QUERY_RUNS) && cfg->block_tokens == kTileKeys;
    const int64_t cpq = (cfg->max_blocks + kScoreWarps - 1) / kScoreWarps;
    const void *score_fn =
        cfg->head_dim == 128
            ? (p.fp8 ? reinterpret_cast<const void *>(&msa_index_score_kernel<128, true>)
                     : reinterpret_cast<const void *>(&msa_index_score_kernel<128, false>))
            : (p.fp8 ? reinterpret_cast<const void *>(&msa_index_score_kernel<64, true>)
                     : reinterpret_cast<const void *>(&msa_index_score_kernel<64, false>));
    alignas(64) CUtensorMap kmap;   // the key rows, for E4M3 keys of 128 dims copied by TMA
    memset(&kmap, 0, sizeof kmap);
    // E4M3 keys of 128 dims whose rows lie on one grid (each page a whole number of
    // token strides, 16-byte aligned): encode the map, whole pages per box where a page
    // is a box (at most 16 boxes a block), else one row per box
    auto encode_key_rows = [&]() -> bool {
        if (!(p.fp8 && cfg->head_dim == 128 && p.num_pages >= 1 && p.stride_token > 0 &&
              p.stride_page % p.stride_token == 0 && (reinterpret_cast<uintptr_t>(p.kdata) & 15u) == 0))
            return false;
        const int64_t rpp = p.stride_page / p.stride_token;
        const int64_t rows = (p.num_pages - 1) * rpp + cfg->page_size;
        const int P = cfg->page_size;
        const int br = (kTileKeys % P == 0 && P >= 8) ? P : (P % kTileKeys == 0 ? kTileKeys : 1);
        if (rpp < P || rows >= ((int64_t)1 << 31) ||
            !msa_internal_encode_byte_rows(&kmap, p.kdata, rows, p.stride_token, br))
            return false;
        p.rows_per_page = rpp;
        p.box_rows = br;
        return true;
    };
    cudaLaunchConfig_t sc;
    memset(&sc, 0, sizeof sc);
    sc.gridDim = dim3((unsigned)(num_queries * cpq));
    sc.blockDim = dim3(kScoreWarps * 32);
    sc.stream = stream;
    if (tiled) {
        const int D = cfg->head_dim;
        const bool hp8 = cfg->num_heads <= 8;
        const int qt = hp8 ? 16 : 8;
        int major = 0, dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(MSA_ERR_CUDA, "device query failed");
        if (major != 10)
            return fail(MSA_ERR_UNSUPPORTED, "query runs need tcgen05 tensor cores (compute capability 10.x)");
        const int64_t tiles = (num_queries + qt - 1) / qt;
        // E4M3 keys of 128 dims on one row grid: the key rows are copied by TMA
        const bool tma = D == 128 && encode_key_rows();
        const int smem = tma ? kRunsDynSmemTma : kRunsDynSmem;
        const void *fns[10] = {
            reinterpret_cast<const void *>(&msa_index_runs_kernel<64, false, 8>),
            reinterpret_cast<const void *>(&msa_index_runs_kernel<64, false, 16>),
            reinterpret_cast<const void *>(&msa_index_runs_kernel<64, true, 8>),
            reinterpret_cast<const void *>(&msa_index_runs_kernel<64, true, 16>),
            reinterpret_cast<const void *>(&msa_index_runs_kernel<128, false, 8>),
            reinterpret_cast<const void *>(&msa_index_runs_kernel<128, false, 16>),
            reinterpret_cast<const void *>(&msa_index_runs_kernel<128, true, 8>),
            reinterpret_cast<const void *>(&msa_index_runs_kernel<128, true, 16>),
            reinterpret_cast<const void *>(&msa_index_runs_tma_kernel<8>),
            reinterpret_cast<const void *>(&msa_index_runs_tma_kernel<16>)};
        score_fn = tma ? fns[8 + (hp8 ? 0 : 1)] : fns[(D == 128 ? 4 : 0) + (p.fp8 ? 2 : 0) + (hp8 ? 0 : 1)];
        sc.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));   // persistent, one CTA per SM
        sc.blockDim = dim3(tma ? kRunsTmaThreads : kRunsThreads);
        if (cudaFuncSetAttribute(score_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
            return fail(MSA_ERR_CUDA, "cudaFuncSetAttribute failed");
        sc.dynamicSmemBytes = (size_t)smem;
    } else if (!counters && cfg->block_tokens == kTileKeys && cfg->num_heads <= 16 && num_queries <= kDecMaxQueries &&
               encode_key_rows() && p.box_rows > 1) {
        // decode batches of E4M3 keys in whole-page boxes: the flat item list on the
        // tcgen05 tensor cores
        int major = 0, dev = 0, sms = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(MSA_ERR_CUDA, "device query failed");
        if (major == 10) {
            score_fn = reinterpret_cast<const void *>(&msa_index_decode_tc_kernel);
            sc.gridDim = dim3((unsigned)sms);   // persistent, one CTA per SM
            sc.blockDim = dim3(kDecThreads);
            if (cudaFuncSetAttribute(score_fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDecDynSmem) !=
                cudaSuccess)
                return fail(MSA_ERR_CUDA, "cudaFuncSetAttribute failed");
            sc.dynamicSmemBytes = (size_t)kDecDynSmem;
        }
    }
    cudaLaunchAttribute sattr[1];
    if (p.pdl) {
        sattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        sattr[0].val.programmaticStreamSerializationAllowed = 1;
        sc.attrs = sattr;
        sc.numAttrs = 1;
    }
    if (!tiled)
        p.counters = counters;
    void *sargs[] = {&p, &kmap};   // the kernels without the map take p alone
    cudaError_t e = cudaLaunchKernelExC(&sc, score_fn, sargs);
    if (e != cudaSuccess)
        return fail(MSA_ERR_CUDA, "score kernel launch failed: %s", cudaGetErrorString(e));
    if (p.counters)
        return MSA_OK;
    // top-k: one CTA per query (several short rows per CTA in large batches),
    // launched programmatically dependent on the scores
    int rows = 1;
    if (num_queries >= kTopkRowsMinQueries && 2 * cfg->max_blocks <= kRankMaxBlocks) {
        rows = kRankMaxBlocks / cfg->max_blocks;
        rows = rows > kTopkRowsMax ? kTopkRowsMax : rows;
    }
    p.topk_rows = rows;
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3((unsigned)((num_queries + rows - 1) / rows));
    lc.blockDim = dim3(kTopkThreads);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    void *args[] = {&p};
    e = cudaLaunchKernelExC(&lc, rows > 1 ? reinterpret_cast<const void *>(&msa_index_topk_rows_kernel)
                                          : reinterpret_cast<const void *>(&msa_index_topk_kernel),
                            args);
    if (e != cudaSuccess)
        return fail(MSA_ERR_CUDA, "top-k kernel launch failed: %s", cudaGetErrorString(e));
    return MSA_OK;
}

}  // namespace

extern "C" msa_status msa_indexer_forward(const msa_indexer_cfg *cfg, int64_t num_queries,
                                          const void *idx_q, const int32_t *kv_len,
                                          const int64_t *table_offset, const int32_t *page_table,
                                          int64_t page_table_len, const msa_cache_desc *idx_k_cache,
                                          const float *k_scale, float *block_scores,
                                          int32_t *topk_ids, int32_t launch_flags,
                                          cudaStream_t stream)
{
    msa_status s = validate(cfg, num_queries, idx_q, kv_len, table_offset, page_table,
                            page_table_len, idx_k_cache, k_scale, block_scores, topk_ids,
                            launch_flags);
    if (s != MSA_OK || num_queries == 0)
        return s;
    return indexer_launch(cfg, num_queries, idx_q, kv_len, table_offset, page_table, page_table_len,
                          idx_k_cache, k_scale, block_scores, topk_ids, nullptr, launch_flags, stream);
}

extern "C" msa_status msa_indexer_forward_fused(const msa_indexer_cfg *cfg, int64_t num_queries,
                                                const void *idx_q, const int32_t *kv_len,
                                                const int64_t *table_offset,
                                                const int32_t *page_table, int64_t page_table_len,
                                                const msa_cache_desc *idx_k_cache,
                                                const float *k_scale, float *block_scores,
                                                int32_t *topk_ids, int32_t *counters,
                                                int32_t launch_flags, cudaStream_t stream)
{
    msa_status s = validate(cfg, num_queries, idx_q, kv_len, table_offset, page_table,
                            page_table_len, idx_k_cache, k_scale, block_scores, topk_ids,
                            launch_flags);
    if (s != MSA_OK)
        return s;
    if (!counters)
        return fail(MSA_ERR_INVALID_ARGUMENT, "counters is NULL");
    if (reinterpret_cast<uintptr_t>(counters) % 4)
        return fail(MSA_ERR_MISALIGNED, "counters is misaligned");
    if (num_queries == 0)
        return MSA_OK;
    return indexer_launch(cfg, num_queries, idx_q, kv_len, table_offset, page_table, page_table_len,
                          idx_k_cache, k_scale, block_scores, topk_ids, counters, launch_flags, stream);
}

// ---------------------------------------------------------------------------
// msa_indexer_forward_fused_noalloc: the single-launch indexer on counters this
// library owns (a file-scope device array), for callers that cannot allocate
// ---------------------------------------------------------------------------
namespace {

constexpr int64_t kNoAllocQueries = 65536;   // counters in the library's array

// one counter per query; all zero between launches (each launch that runs to
// completion leaves them zero)
static __device__ __align__(256) int32_t g_noalloc_counters[kNoAllocQueries];

std::mutex g_noalloc_mu;
int32_t *g_noalloc_ptr[64];   // the array's address on each device, once looked up and cleared

}  // namespace

extern "C" msa_status msa_indexer_forward_fused_noalloc(const msa_indexer_cfg *cfg,
                                                        int64_t num_queries, const void *idx_q,
                                                        const int32_t *kv_len,
                                                        const int64_t *table_offset,
                                                        const int32_t *page_table,
                                                        int64_t page_table_len,
                                                        const msa_cache_desc *idx_k_cache,
                                                        const float *k_scale, float *block_scores,
                                                        int32_t *topk_ids, int32_t launch_flags,
                                                        cudaStream_t stream)
{
    msa_status s = validate(cfg, num_queries, idx_q, kv_len, table_offset, page_table,
                            page_table_len, idx_k_cache, k_scale, block_scores, topk_ids,
                            launch_flags);
    if (s != MSA_OK)
        return s;
    if (num_queries > kNoAllocQueries)
        return fail(MSA_ERR_UNSUPPORTED, "num_queries %lld is above the %lld counters of the library",
                    (long long)num_queries, (long long)kNoAllocQueries);
    if (num_queries == 0)
        return MSA_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return fail(MSA_ERR_CUDA, "cudaGetDevice failed");
    int32_t *counters = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            // first use on this device: the array's address, and every counter zeroed
            // (stream-ordered before this call's launch)
            void *a = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&a, g_noalloc_counters);
            if (e != cudaSuccess)
                return fail(MSA_ERR_CUDA, "cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
            e = cudaMemsetAsync(a, 0, sizeof(g_noalloc_counters), stream);
            if (e != cudaSuccess)
                return fail(MSA_ERR_CUDA, "clearing the counters failed: %s", cudaGetErrorString(e));
            g_noalloc_ptr[dev] = static_cast<int32_t *>(a);
        }
        counters = g_noalloc_ptr[dev];
    }
    return indexer_launch(cfg, num_queries, idx_q, kv_len, table_offset, page_table, page_table_len,
                          idx_k_cache, k_scale, block_scores, topk_ids, counters, launch_flags, stream);
}
