// MiniMax-M3 MSA per-layer fused producer and paged-cache write for sm_103a.
//
// What it computes is stated in include/msa_producer.h, after "[None][perf] Fuse
// MiniMax-M3 QKV and index projection" (TensorRT-LLM PR 18205, Description) and
// "[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into one kernel"
// (PR 18614, "The problem" / "The fix").
//
// Design (GB300).  The path is streaming work bound by HBM bandwidth (about two
// flops per byte, no dense contraction), so it runs on the CUDA cores; there is
// nothing here for the tensor cores.  What keeps such a kernel off the bandwidth
// roofline is instruction issue, latency stalls and memory-level parallelism, and
// the design spends all three carefully:
//   * A CTA owns one token at a time and strides over the tokens (a persistent
//     grid of SMs x resident CTAs, or one CTA per token).
//   * Rows are staged into shared memory with cp.async, the next token's while
//     the current one is computed, so every CTA always has a row in flight
//     without holding it in registers.  Each thread copies exactly the pieces it
//     later reads, so no barrier guards the ring; cp.async.wait_group waits on the
//     thread's own copies only and cannot spin.
//   * A head row of D elements is L = D/16 lanes; every lane holds two 8-element
//     pieces chosen so that the NeoX rotate-half partners (dims k and k + rd/2)
//     sit in the same lane: RoPE needs no shuffle, and the RMS reduction is
//     log2(L) xor shuffles.  Pieces are 16 bytes, so loads and stores stay fully
//     coalesced (L lanes x 16 bytes = one contiguous segment per piece set).
//   * Arithmetic is fp32 with Blackwell's paired f32x2 FMA/MUL, halving the FP
//     instruction count; conversion uses cvt.rn.bf16x2.f32 and
//     cvt.rn.satfinite.e4m3x2.f32.
//   * Per-token work shared by every head -- the slot -> (page, offset)
//     derivation with its dependent page-table load, and the rotary cos/sin table
//     -- is computed for a group of kGroup tokens at a time by all threads into a
//     double-buffered shared table, with its loads issued one or two groups
//     ahead.  One barrier per group publishes it; between barriers the warps run
//     decoupled, so their memory and shuffle latencies overlap.
//   * No wait on another CTA, flag or mbarrier exists, so nothing can spin.
//     With programmatic dependent launch the kernel reads its constants and the
//     first group's metadata before waiting for the previous kernel, and lets the
//     next kernel start at once (its prologue overlaps this kernel's body).

#include "msa_producer.h"
#include "msa_internal.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

// Resident 256-thread CTAs per SM the register budget is sized for (3: 80 registers).
#ifndef MSA_MIN_CTAS_PER_SM
#define MSA_MIN_CTAS_PER_SM 3
#endif
// Rows in flight per CTA: the current token's and kStages - 1 ahead.
#ifndef MSA_STAGES
#define MSA_STAGES 2
#endif

// 1: under programmatic dependent launch the next kernel may start as soon as this
// one begins; 0: only once this one has waited for its own predecessor.  Measured on
// the 60-layer decode step (tiny shapes, batch 256): 2.6 us per layer with 1, 3.4
// with 0.  With 1, a chain of launches with programmatic dependent launch may run
// ahead of its kernels' completion, hence the contract on MSA_LAUNCH_PDL.
#ifndef MSA_PDL_EARLY_TRIGGER
#define MSA_PDL_EARLY_TRIGGER 1
#endif
// Tokens per CTA from which the caches' reciprocal scales are computed once per CTA
// into shared memory (measured: 1% faster at 143 tokens per CTA, 0.4 us per launch
// slower at one token per CTA in the decode step, where the load sits on the
// critical path).
#ifndef MSA_INV_TABLE_TOKENS
#define MSA_INV_TABLE_TOKENS 16
#endif
// Unroll factor of the loop over a token's head-row passes (1: not unrolled).
#ifndef MSA_PASS_UNROLL
#define MSA_PASS_UNROLL 2
#endif

// Tokens whose placement and rotary table are prepared together (one barrier each).
#ifndef MSA_GROUP
#define MSA_GROUP 8
#endif

namespace {

constexpr int kMaxRotaryHalf = 64;       // rotary_dim / 2 <= head_dim / 2 <= 64
constexpr int kMaxHeadScales = 256;      // per-head scale mode: 2*Hkv + Hik <= 256
constexpr int kStages = MSA_STAGES;
constexpr int kGroup = MSA_GROUP;        // tokens per metadata group (one barrier each)
constexpr int kPassUnroll = MSA_PASS_UNROLL;
constexpr int kInvTableTokens = MSA_INV_TABLE_TOKENS;
constexpr int kMaxRowBytes = 96 * 1024;  // widest token row the shared-memory ring takes

struct CacheArgs {
    uint8_t *data;          // nullptr: this cache is not written
    int64_t num_pages;
    int64_t stride_page;    // elements
    int64_t stride_head;
    int64_t stride_token;
    int32_t fp8;            // 1: E4M3, 0: bf16
    int32_t pad;
};

struct Params {
    const uint16_t *qkv;
    int64_t row_stride;             // elements
    const int32_t *positions;
    const int64_t *slots;
    const int32_t *page_table;      // nullptr: physical slots
    int64_t page_table_len;
    const uint16_t *norm_w[4];      // q, k, idx_q, idx_k (nullptr: unit weight, unused)
    uint16_t *q_out;
    uint16_t *idx_q_out;
    CacheArgs cache[3];             // k, v, idx_k
    const float *scales;
    int64_t num_tokens;
    int32_t hq, hkv, hiq, hik;
    int32_t htot;                   // head rows per token
    int32_t row_bytes;              // htot * D * 2: bytes staged per token
    int32_t rotary_dim;
    int32_t rope_style;
    int32_t page_size;
    int32_t page_shift;             // log2(page_size) when a power of two, else -1
    int32_t scale_mode;
    int32_t pdl;                    // launched with programmatic dependent launch
    float rms_eps;
    float inv_freq[kMaxRotaryHalf];
#ifdef MSA_CHECKED
    const uint8_t *out_hi[2];       // first byte past q_out, idx_q_out
    const uint8_t *cache_hi[3];     // first byte past each cache's reachable extent
#endif
};

#ifdef MSA_CHECKED
// Checked build: a global store whose bytes leave its destination's extent is
// skipped and counted here (read by msa_checked_violations).
__device__ unsigned long long g_msa_violations;

__device__ __forceinline__ bool msa_in_range(const void *ptr, int n, const void *lo, const void *hi)
{
    const uint8_t *b = static_cast<const uint8_t *>(ptr);
    if (b >= static_cast<const uint8_t *>(lo) && b + n <= static_cast<const uint8_t *>(hi))
        return true;
    atomicAdd(&g_msa_violations, 1ull);
    return false;
}
#define MSA_GUARD(ptr, n, lo, hi) if (!msa_in_range((ptr), (n), (lo), (hi))) {} else
#else
#define MSA_GUARD(ptr, n, lo, hi)
#endif

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;" ::"r"(dst), "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// a bf16 pair -> (element 0, element 1) in fp32
__device__ __forceinline__ float2 unpack2(uint32_t v)
{
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// (element 0, element 1) -> a bf16 pair, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float2 v)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(v.y), "f"(v.x));
    return d;
}

// two pairs -> four E4M3 bytes in element order; RNE, saturating to +-448
__device__ __forceinline__ uint32_t pack_e4m3x4(float2 a, float2 b)
{
    unsigned short lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a.y), "f"(a.x));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(b.y), "f"(b.x));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h)
{
    return __uint_as_float(((uint32_t)h) << 16);
}

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

__device__ __forceinline__ uint4 pack_bf16x8(const float2 *y)
{
    return make_uint4(pack_bf16x2(y[0]), pack_bf16x2(y[1]), pack_bf16x2(y[2]), pack_bf16x2(y[3]));
}

// ---------------------------------------------------------------------------
// per-token placement
// ---------------------------------------------------------------------------

struct TokenMeta {
    long long page;  // -1: no cache takes the token
    int off;
    int valid;       // bit c: cache c (k, v, idx_k) takes the token
};

// The page a slot points at before the page-count check: the table entry of its
// logical block (-1 past the table), or the block itself without a table; -1 for
// a padded slot.
__device__ __forceinline__ long long table_entry(const Params &p, long long ls)
{
    if (ls < 0)
        return -1;
    const long long blk = p.page_shift >= 0 ? (ls >> p.page_shift) : ls / p.page_size;
    if (!p.page_table)
        return blk;
    return blk < p.page_table_len ? (long long)__ldg(p.page_table + blk) : -1;
}

__device__ __forceinline__ TokenMeta place(const Params &p, long long ls, long long page)
{
    TokenMeta m;
    m.page = page;
    m.off = 0;
    m.valid = 0;
    if (ls < 0 || page < 0)
        return m;
    m.off = p.page_shift >= 0 ? (int)(ls & (long long)(p.page_size - 1))
                              : (int)(ls - (ls / p.page_size) * p.page_size);
#pragma unroll
    for (int ci = 0; ci < 3; ++ci)
        if (p.cache[ci].data && page < p.cache[ci].num_pages)
            m.valid |= 1 << ci;
    return m;
}

// ---------------------------------------------------------------------------
// the per-token compute (shared by both kernels)
// ---------------------------------------------------------------------------
//
// D   head_dim (64 or 128): a head row is L = D/16 lanes of 2 x 8 elements
// NT  compute threads per CTA (a multiple of 32)

// Which 2 x 8 elements of a head row a lane holds, and its first head row.
struct LaneGeom {
    int q;           // lane position inside its head rows
    int row0;        // first head row of this thread
    int npass;       // passes over the token's head rows (uniform across the warp)
    int aoff, boff;  // element offsets of piece A and piece B in the head row
    bool pair;       // NeoX: piece B holds the rotate-half partners of piece A
    bool rot_a, rot_b;  // GPT-J: piece A / B lies inside the rotary dims
};

template <int D, int NT>
__device__ __forceinline__ LaneGeom lane_geom(const Params &p, int tid)
{
    constexpr int L = D / 16;
    constexpr int RPP = NT / L;
    LaneGeom g;
    const int warp = tid >> 5;
    g.q = tid % L;
    g.row0 = tid / L;
    const int warp_row0 = (warp * 32) / L;
    g.npass = p.htot > warp_row0 ? (p.htot - warp_row0 + RPP - 1) / RPP : 0;
    const int rd = p.rotary_dim;
    const int half = rd / 2;
    g.pair = g.rot_a = g.rot_b = false;
    if (p.rope_style == MSA_ROPE_NEOX) {
        if (16 * g.q < rd) {          // rotated: dims k and k + rd/2 (k = 8q .. 8q+7)
            g.aoff = 8 * g.q;
            g.boff = 8 * g.q + half;
            g.pair = true;
        } else {                      // pass-through dims [rd, D)
            g.aoff = rd + 16 * (g.q - rd / 16);
            g.boff = g.aoff + 8;
        }
    } else {                          // GPT-J: pairs (2k, 2k+1) inside each piece
        g.aoff = 16 * g.q;
        g.boff = g.aoff + 8;
        g.rot_a = g.aoff < rd;
        g.rot_b = g.boff < rd;
    }
    return g;
}

// Every head row of token t that this thread takes part in: load its two pieces
// from the staged row at shared address srow, RMSNorm (all but V), RoPE, then the
// compact Q / index-Q store or the cache encode and scatter.
template <int D, int NT>
__device__ __forceinline__ void token_rows(const Params &p, const LaneGeom &g, uint32_t srow,
                                           const TokenMeta &meta, const float *cos_row,
                                           const float *sin_row, const float (*s_w)[D],
                                           const float *s_inv, int64_t t)
{
    constexpr int L = D / 16;
    constexpr int RPP = NT / L;
    const int htot = p.htot;
    const int e_k = p.hq, e_v = p.hq + p.hkv, e_iq = p.hq + 2 * p.hkv;
    const int e_ik = e_iq + p.hiq;
    const int aoff = g.aoff, boff = g.boff;
    uint16_t *q_tok = p.q_out + (int64_t)t * p.hq * D;
    uint16_t *iq_tok = p.idx_q_out + (int64_t)t * p.hiq * D;

#pragma unroll kPassUnroll
    for (int pass = 0; pass < g.npass; ++pass) {
        const int hr = g.row0 + pass * RPP;
        const bool active = hr < htot;

        // y holds piece A in y[0..3] and piece B in y[4..7], as element pairs
        float2 y[8];
        if (active) {
            const uint4 ra = lds128(srow + 2u * (uint32_t)(hr * D + aoff));
            const uint4 rb = lds128(srow + 2u * (uint32_t)(hr * D + boff));
            y[0] = unpack2(ra.x); y[1] = unpack2(ra.y);
            y[2] = unpack2(ra.z); y[3] = unpack2(ra.w);
            y[4] = unpack2(rb.x); y[5] = unpack2(rb.y);
            y[6] = unpack2(rb.z); y[7] = unpack2(rb.w);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
                y[j] = f2(0.0f);
        }

        float2 ss2 = __fmul2_rn(y[0], y[0]);
#pragma unroll
        for (int j = 1; j < 8; ++j)
            ss2 = __ffma2_rn(y[j], y[j], ss2);
        float ss = ss2.x + ss2.y;
#pragma unroll
        for (int o = 1; o < L; o <<= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o, L);
        if (!active)
            continue;

        // section of this head row: 0 Q, 1 K, 2 V, 3 idx-Q, 4 idx-K
        int sec, h;
        if (hr < e_k) { sec = 0; h = hr; }
        else if (hr < e_v) { sec = 1; h = hr - e_k; }
        else if (hr < e_iq) { sec = 2; h = hr - e_v; }
        else if (hr < e_ik) { sec = 3; h = hr - e_iq; }
        else { sec = 4; h = hr - e_ik; }

        if (sec != 2) {
            const int widx = sec == 0 ? 0 : sec == 1 ? 1 : sec == 3 ? 2 : 3;
            const float2 r2 = f2(rsqrtf(fmaf(ss, 1.0f / (float)D, p.rms_eps)));
            {
                const float4 w0 = *reinterpret_cast<const float4 *>(&s_w[widx][aoff]);
                const float4 w1 = *reinterpret_cast<const float4 *>(&s_w[widx][aoff + 4]);
                y[0] = __fmul2_rn(__fmul2_rn(y[0], r2), make_float2(w0.x, w0.y));
                y[1] = __fmul2_rn(__fmul2_rn(y[1], r2), make_float2(w0.z, w0.w));
                y[2] = __fmul2_rn(__fmul2_rn(y[2], r2), make_float2(w1.x, w1.y));
                y[3] = __fmul2_rn(__fmul2_rn(y[3], r2), make_float2(w1.z, w1.w));
            }
            {
                const float4 w0 = *reinterpret_cast<const float4 *>(&s_w[widx][boff]);
                const float4 w1 = *reinterpret_cast<const float4 *>(&s_w[widx][boff + 4]);
                y[4] = __fmul2_rn(__fmul2_rn(y[4], r2), make_float2(w0.x, w0.y));
                y[5] = __fmul2_rn(__fmul2_rn(y[5], r2), make_float2(w0.z, w0.w));
                y[6] = __fmul2_rn(__fmul2_rn(y[6], r2), make_float2(w1.x, w1.y));
                y[7] = __fmul2_rn(__fmul2_rn(y[7], r2), make_float2(w1.z, w1.w));
            }
            if (g.pair) {
                // u' = u c - v s, v' = v c + u s, with u in piece A and v in piece B;
                // pair j of each piece is at frequencies 8q + 2j, 8q + 2j + 1
                const float4 c0 = *reinterpret_cast<const float4 *>(cos_row);
                const float4 c1 = *reinterpret_cast<const float4 *>(cos_row + 4);
                const float4 s0 = *reinterpret_cast<const float4 *>(sin_row);
                const float4 s1 = *reinterpret_cast<const float4 *>(sin_row + 4);
                const float2 cs[4] = {make_float2(c0.x, c0.y), make_float2(c0.z, c0.w),
                                      make_float2(c1.x, c1.y), make_float2(c1.z, c1.w)};
                const float2 sn[4] = {make_float2(s0.x, s0.y), make_float2(s0.z, s0.w),
                                      make_float2(s1.x, s1.y), make_float2(s1.z, s1.w)};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 u = y[j], v = y[4 + j];
                    y[j] = __ffma2_rn(v, make_float2(-sn[j].x, -sn[j].y), __fmul2_rn(u, cs[j]));
                    y[4 + j] = __ffma2_rn(u, sn[j], __fmul2_rn(v, cs[j]));
                }
            } else if (g.rot_a || g.rot_b) {
                // GPT-J: (y[2m], y[2m+1]) at frequency 8q + m (piece A), 8q + 4 + m (B)
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    if (m < 4 ? g.rot_a : g.rot_b) {
                        const float c = cos_row[m], sn = sin_row[m];
                        const float u = y[m].x, v = y[m].y;
                        y[m] = make_float2(u * c - v * sn, v * c + u * sn);
                    }
                }
            }
        }

        if (sec == 0 || sec == 3) {
            uint16_t *dst = sec == 0 ? q_tok + h * D : iq_tok + h * D;
#ifdef MSA_CHECKED
            const void *lo = sec == 0 ? (const void *)p.q_out : (const void *)p.idx_q_out;
            const void *hi = p.out_hi[sec == 0 ? 0 : 1];
#endif
            MSA_GUARD(dst + aoff, 16, lo, hi) st_v4(dst + aoff, pack_bf16x8(y));
            MSA_GUARD(dst + boff, 16, lo, hi) st_v4(dst + boff, pack_bf16x8(y + 4));
        } else {
            const int ci = sec == 1 ? 0 : sec == 2 ? 1 : 2;
            if (!((meta.valid >> ci) & 1))
                continue;
            const CacheArgs &cc = p.cache[ci];
            const int64_t e = meta.page * cc.stride_page + (int64_t)h * cc.stride_head +
                              (int64_t)meta.off * cc.stride_token;
            if (cc.fp8) {
                const int si = p.scale_mode == MSA_SCALE_PER_HEAD
                                   ? (ci == 0 ? h : ci == 1 ? p.hkv + h : 2 * p.hkv + h)
                                   : ci;
                // the CTA's table of reciprocal scales when it has one (many tokens per
                // CTA), else the scale itself (a decode CTA's single token)
                const float2 inv = f2(s_inv ? s_inv[si] : __frcp_rn(__ldg(p.scales + si)));
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    y[j] = __fmul2_rn(y[j], inv);
                uint8_t *dst = cc.data + e;
                MSA_GUARD(dst + aoff, 8, cc.data, p.cache_hi[ci])
                st_v2(dst + aoff, pack_e4m3x4(y[0], y[1]), pack_e4m3x4(y[2], y[3]));
                MSA_GUARD(dst + boff, 8, cc.data, p.cache_hi[ci])
                st_v2(dst + boff, pack_e4m3x4(y[4], y[5]), pack_e4m3x4(y[6], y[7]));
            } else {
                uint16_t *dst = reinterpret_cast<uint16_t *>(cc.data) + e;
                MSA_GUARD(dst + aoff, 16, cc.data, p.cache_hi[ci])
                st_v4(dst + aoff, pack_bf16x8(y));
                MSA_GUARD(dst + boff, 16, cc.data, p.cache_hi[ci])
                st_v4(dst + boff, pack_bf16x8(y + 4));
            }
        }
    }
}

// The per-token metadata pipeline, shared by both kernels.  Tokens are taken in
// groups of kGroup; the placement and rotary table of group g + 1 are computed at
// the end of group g into the other half of a double-buffered shared table.
// Thread j < kGroup owns token j of every group: the slot and page-table entry of
// the group whose metadata is computed next (loaded a group earlier), and the slot
// of the group after that.  Table entry e = tid + m*NT is (token e / half,
// frequency e % half); its position is loaded a group early.
template <int NT>
struct MetaPipe {
    static constexpr int ME = kGroup * kMaxRotaryHalf / NT;  // table entries per thread
    long long ls_n = -1, pte_n = -1, ls_nn = -1;
    int pos_n[ME];

    __device__ __forceinline__ long long load_slot(const Params &p, int64_t t0, int64_t G,
                                                   int64_t ntok, int64_t i) const
    {
        return i < ntok ? __ldg(p.slots + t0 + i * G) : -1;
    }
    __device__ __forceinline__ void load_positions(const Params &p, int tid, int64_t t0, int64_t G,
                                                   int64_t ntok, int64_t gbase)
    {
        const int half = p.rotary_dim / 2;
#pragma unroll
        for (int m = 0; m < ME; ++m) {
            const int e = tid + m * NT;
            const int64_t i = gbase + (half > 0 ? e / half : 0);
            pos_n[m] = (half > 0 && e < kGroup * half && i < ntok) ? __ldg(p.positions + t0 + i * G) : 0;
        }
    }
    __device__ __forceinline__ void start(const Params &p, int tid, int64_t t0, int64_t G, int64_t ntok)
    {
        if (tid < kGroup) {
            ls_n = load_slot(p, t0, G, ntok, tid);
            pte_n = table_entry(p, ls_n);
            ls_nn = load_slot(p, t0, G, ntok, kGroup + tid);
        }
        load_positions(p, tid, t0, G, ntok, 0);
    }
    __device__ __forceinline__ void compute(const Params &p, int tid, int64_t ntok, int64_t gbase,
                                            TokenMeta (*s_meta)[kGroup],
                                            float (*s_cs)[kGroup][2][kMaxRotaryHalf], int b)
    {
        const int half = p.rotary_dim / 2;
        if (tid < kGroup)
            s_meta[b][tid] = place(p, ls_n, pte_n);
#pragma unroll
        for (int m = 0; m < ME; ++m) {
            const int e = tid + m * NT;
            if (half > 0 && e < kGroup * half && gbase + e / half < ntok) {
                const int j = e / half, k = e % half;
                float sn, c;
                sincosf((float)pos_n[m] * p.inv_freq[k], &sn, &c);
                s_cs[b][j][0][k] = c;
                s_cs[b][j][1][k] = sn;
            }
        }
    }
    __device__ __forceinline__ void prefetch(const Params &p, int tid, int64_t t0, int64_t G,
                                             int64_t ntok, int64_t gbase)
    {
        if (tid < kGroup) {
            ls_n = ls_nn;
            pte_n = table_entry(p, ls_n);
            ls_nn = load_slot(p, t0, G, ntok, gbase + kGroup + tid);
        }
        load_positions(p, tid, t0, G, ntok, gbase);
    }
};

// ---------------------------------------------------------------------------
// the producer kernel, rows staged by the compute threads (cp.async)
// ---------------------------------------------------------------------------
//
// A CTA takes the tokens blockIdx.x + i * gridDim.x, i = 0, 1, ...  in groups of
// kGroup.  Each thread copies the 16-byte pieces of the rows that it later reads
// into a kStages-deep shared-memory ring, one token ahead.
template <int D, int NT>
__global__ void __launch_bounds__(NT, MSA_MIN_CTAS_PER_SM * 256 / NT)
msa_producer_kernel(const __grid_constant__ Params p)
{
    constexpr int L = D / 16;
    constexpr int RPP = NT / L;                       // head rows per pass
    static_assert(NT % 32 == 0 && 32 % L == 0, "a head row must sit inside one warp");
    static_assert(kGroup <= NT && MetaPipe<NT>::ME * NT == kGroup * kMaxRotaryHalf, "group geometry");

    extern __shared__ __align__(128) uint8_t s_rows[];  // kStages x row_bytes
    __shared__ __align__(16) float s_w[4][D];
    __shared__ __align__(16) float s_cs[2][kGroup][2][kMaxRotaryHalf];  // [buf][token][cos|sin][k]
    __shared__ __align__(16) TokenMeta s_meta[2][kGroup];
    __shared__ float s_inv[kMaxHeadScales];   // 1 / scale of every FP8 cache (per tensor or head)

#if MSA_PDL_EARLY_TRIGGER
    asm volatile("griddepcontrol.launch_dependents;" :::);
#endif
    const int tid = threadIdx.x;
    const LaneGeom g = lane_geom<D, NT>(p, tid);
    const int htot = p.htot;

    // constants (may be read before waiting on the previous kernel): loaded into
    // registers now, stored to shared memory once the other loads are in flight
    constexpr int NW = (4 * D + NT - 1) / NT;
    float wreg[NW];
#pragma unroll
    for (int m = 0; m < NW; ++m) {
        const int i = tid + m * NT;
        const uint16_t *w = i < 4 * D ? p.norm_w[i / D] : nullptr;
        wreg[m] = w ? bf16_to_f32(__ldg(w + i % D)) : 1.0f;
    }

    const int64_t T = p.num_tokens;
    const int64_t G = gridDim.x;
    const int64_t t0 = blockIdx.x;
    if (t0 >= T)
        return;
    const int64_t ntok = (T - t0 + G - 1) / G;  // tokens of this CTA
    auto token = [&](int64_t i) { return t0 + i * G; };

    const uint32_t rows_base = smem_addr(s_rows);
    auto stage_row = [&](int64_t tok, int stage) {
        const uint16_t *src = p.qkv + tok * p.row_stride;
        const uint32_t dst = rows_base + (uint32_t)stage * (uint32_t)p.row_bytes;
        for (int hr = g.row0; hr < htot; hr += RPP) {
            const int e = hr * D;
            cp_async16(dst + 2u * (uint32_t)(e + g.aoff), src + e + g.aoff);
            cp_async16(dst + 2u * (uint32_t)(e + g.boff), src + e + g.boff);
        }
    };
    auto stage_first_rows = [&]() {
#pragma unroll
        for (int s = 0; s < kStages - 1; ++s) {
            if (s < ntok)
                stage_row(token(s), s);
            cp_async_commit();
        }
    };

    MetaPipe<NT> meta;
    // ---- prologue ----
    // Under programmatic dependent launch the first group's metadata is computed
    // before waiting on the previous kernel and the rows are read after it.
    // Otherwise the rows are requested first, so that their latency overlaps the
    // metadata's dependent loads.
    if (!p.pdl)
        stage_first_rows();
    meta.start(p, tid, t0, G, ntok);
    meta.compute(p, tid, ntok, 0, s_meta, s_cs, 0);
    meta.prefetch(p, tid, t0, G, ntok, kGroup);
#pragma unroll
    for (int m = 0; m < NW; ++m) {
        const int i = tid + m * NT;
        if (i < 4 * D)
            s_w[i / D][i % D] = wreg[m];
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");
    // (With MSA_PDL_EARLY_TRIGGER 0 the next kernel may start only once every CTA has
    // passed this point: every kernel enqueued before this one has then completed.)
#if !MSA_PDL_EARLY_TRIGGER
    asm volatile("griddepcontrol.launch_dependents;" :::);
#endif
    if (p.pdl)
        stage_first_rows();
    // The caches' reciprocal scales, once per CTA (published by the first group
    // barrier), when the CTA has tokens enough to amortise the extra load on its
    // critical path; a CTA with few tokens computes them per head row instead.
    const bool inv_table = p.scales && ntok >= kInvTableTokens;
    if (inv_table) {
        const int ns = p.scale_mode == MSA_SCALE_PER_HEAD ? 2 * p.hkv + p.hik : 3;
        for (int i = tid; i < ns; i += NT)
            s_inv[i] = __frcp_rn(__ldg(p.scales + i));
    }

    for (int64_t g0 = 0; g0 < ntok; g0 += kGroup) {
        const int buf = (int)((g0 / kGroup) & 1);
        const int64_t gn = g0 + kGroup;
        __syncthreads();  // publishes this group's metadata (and, the first time, the weights)

        const int64_t gend = gn < ntok ? gn : ntok;
        for (int64_t i = g0; i < gend; ++i) {
            const int jt = (int)(i - g0);
            {   // rows of the token kStages-1 ahead
                const int64_t ip = i + kStages - 1;
                if (ip < ntok)
                    stage_row(token(ip), (int)(ip % kStages));
                cp_async_commit();
            }
            cp_async_wait<kStages - 1>();  // this thread's pieces of token i have landed
            const uint32_t srow = rows_base + (uint32_t)(i % kStages) * (uint32_t)p.row_bytes;
            token_rows<D, NT>(p, g, srow, s_meta[buf][jt], &s_cs[buf][jt][0][8 * g.q],
                              &s_cs[buf][jt][1][8 * g.q], s_w, inv_table ? s_inv : nullptr,
                              token(i));
        }
        if (gn < ntok) {  // the next group's metadata, into the other buffer
            meta.compute(p, tid, ntok, gn, s_meta, s_cs, buf ^ 1);
            meta.prefetch(p, tid, t0, G, ntok, gn + kGroup);
        }
    }
    cp_async_wait<0>();
}

// ---------------------------------------------------------------------------
// host side: checks
// ---------------------------------------------------------------------------

thread_local char g_detail[256] = "";

msa_status fail(msa_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
msa_status fail(msa_status s, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
    return s;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// a*b + c with overflow detection (all non-negative)
bool mul_add_ok(int64_t a, int64_t b, int64_t c, int64_t *out)
{
    int64_t m;
    if (__builtin_mul_overflow(a, b, &m))
        return false;
    return !__builtin_add_overflow(m, c, out);
}

msa_status check_cache(const char *name, const msa_cache_desc *c, int64_t heads, int32_t D,
                       int32_t P)
{
    if (!c->data)
        return fail(MSA_ERR_INVALID_ARGUMENT, "%s: data is NULL", name);
    if (c->dtype != MSA_DTYPE_BF16 && c->dtype != MSA_DTYPE_FP8_E4M3)
        return fail(MSA_ERR_UNSUPPORTED, "%s: dtype %d", name, c->dtype);
    if (c->reserved != 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "%s: reserved field must be 0", name);
    if (c->num_heads != heads)
        return fail(MSA_ERR_INVALID_ARGUMENT, "%s: num_heads %lld, expected %lld", name,
                    (long long)c->num_heads, (long long)heads);
    if (c->num_pages < 0 || c->stride_page < 0 || c->stride_head < 0 || c->stride_token < 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "%s: negative page count or stride", name);
    if (!aligned(c->data, 16))
        return fail(MSA_ERR_MISALIGNED, "%s: data not 16-byte aligned", name);
    if (c->stride_page % 8 || c->stride_head % 8 || c->stride_token % 8)
        return fail(MSA_ERR_MISALIGNED, "%s: strides must be multiples of 8 elements", name);
    if (c->num_pages == 0 || heads == 0)
        return MSA_OK;
    // furthest element a write can reach, then in bytes
    const int64_t es = c->dtype == MSA_DTYPE_FP8_E4M3 ? 1 : 2;
    int64_t last = D - 1;
    if (!mul_add_ok(c->num_pages - 1, c->stride_page, last, &last) ||
        !mul_add_ok(heads - 1, c->stride_head, last, &last) ||
        !mul_add_ok(P - 1, c->stride_token, last, &last))
        return fail(MSA_ERR_OFFSET_OVERFLOW, "%s: reachable element offset overflows int64", name);
    int64_t bytes;
    if (!mul_add_ok(last, es, es, &bytes))
        return fail(MSA_ERR_OFFSET_OVERFLOW, "%s: reachable byte offset overflows int64", name);
    if ((uint64_t)bytes > UINTPTR_MAX - reinterpret_cast<uintptr_t>(c->data))
        return fail(MSA_ERR_OFFSET_OVERFLOW, "%s: extent wraps the address space", name);
    // rows must not overlap: sorted by stride, each stride must clear the extent of
    // everything inside it (a sufficient condition for a one-to-one layout)
    struct Dim { int64_t stride, count; } dims[3] = {
        {c->stride_token, P}, {c->stride_head, heads}, {c->stride_page, c->num_pages}};
    for (int i = 1; i < 3; ++i)
        for (int j = i; j > 0 && dims[j].stride < dims[j - 1].stride; --j) {
            Dim tmp = dims[j];
            dims[j] = dims[j - 1];
            dims[j - 1] = tmp;
        }
    int64_t extent = D;
    for (int i = 0; i < 3; ++i) {
        if (dims[i].count <= 1)
            continue;
        if (dims[i].stride < extent)
            return fail(MSA_ERR_INVALID_ARGUMENT, "%s: strides make cache rows overlap", name);
        if (!mul_add_ok(dims[i].stride, dims[i].count - 1, extent, &extent))
            return fail(MSA_ERR_OFFSET_OVERFLOW, "%s: extent overflows int64", name);
    }
    return MSA_OK;
}

// rows == false: everything except the token rows (qkv, its stride and the
// shared-memory row limit), for callers that make the rows themselves.
msa_status validate(const msa_producer_cfg *cfg, int64_t T, const void *qkv, int64_t row_stride,
                    const int32_t *positions, const int64_t *slots, const int32_t *page_table,
                    int64_t page_table_len, const void *wq, const void *wk, const void *wiq,
                    const void *wik, void *q_out, void *iq_out, const msa_cache_desc *kc,
                    const msa_cache_desc *vc, const msa_cache_desc *ikc, const float *scales,
                    int32_t flags, bool rows = true)
{
    g_detail[0] = '\0';
    if (!cfg)
        return fail(MSA_ERR_INVALID_ARGUMENT, "cfg is NULL");
    const int32_t Hq = cfg->num_q_heads, Hkv = cfg->num_kv_heads;
    const int32_t Hiq = cfg->num_idx_q_heads, Hik = cfg->num_idx_k_heads;
    const int32_t D = cfg->head_dim, rd = cfg->rotary_dim, P = cfg->page_size;
    if (Hq < 0 || Hkv < 0 || Hiq < 0 || Hik < 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "negative head count");
    const int64_t Htot = (int64_t)Hq + 2 * (int64_t)Hkv + Hiq + Hik;
    if (Htot == 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "no heads");
    if (D <= 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "head_dim %d", D);
    if (D != 64 && D != 128)
        return fail(MSA_ERR_UNSUPPORTED, "head_dim %d (built: 64, 128)", D);
    if (rows && Htot * D * 2 > kMaxRowBytes)
        return fail(MSA_ERR_UNSUPPORTED, "a token row of %lld bytes is wider than %d",
                    (long long)(Htot * D * 2), kMaxRowBytes);
    if (cfg->rope_style != MSA_ROPE_NEOX && cfg->rope_style != MSA_ROPE_GPTJ)
        return fail(MSA_ERR_UNSUPPORTED, "rope_style %d", cfg->rope_style);
    if (rd < 0 || rd > D || (rd & 1))
        return fail(MSA_ERR_INVALID_ARGUMENT, "rotary_dim %d with head_dim %d", rd, D);
    if (cfg->rope_style == MSA_ROPE_NEOX && rd % 16)
        return fail(MSA_ERR_UNSUPPORTED, "NeoX rotary_dim %d is not a multiple of 16", rd);
    if (cfg->rope_style == MSA_ROPE_GPTJ && rd % 8)
        return fail(MSA_ERR_UNSUPPORTED, "GPT-J rotary_dim %d is not a multiple of 8", rd);
    if (rd > 0 && !(cfg->rope_theta > 0.0f && std::isfinite(cfg->rope_theta)))
        return fail(MSA_ERR_INVALID_ARGUMENT, "rope_theta must be positive and finite");
    if (!(cfg->rms_eps >= 0.0f && std::isfinite(cfg->rms_eps)))
        return fail(MSA_ERR_INVALID_ARGUMENT, "rms_eps must be non-negative and finite");
    if (P <= 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "page_size %d", P);
    if (cfg->scale_mode != MSA_SCALE_PER_TENSOR && cfg->scale_mode != MSA_SCALE_PER_HEAD)
        return fail(MSA_ERR_UNSUPPORTED, "scale_mode %d", cfg->scale_mode);
    if (cfg->scale_mode == MSA_SCALE_PER_HEAD && 2 * (int64_t)Hkv + Hik > kMaxHeadScales)
        return fail(MSA_ERR_UNSUPPORTED, "per-head scales for more than %d heads", kMaxHeadScales);
    if (cfg->reserved != 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "cfg reserved field must be 0");
    if (flags & ~(MSA_LAUNCH_PERSISTENT | MSA_LAUNCH_PDL))
        return fail(MSA_ERR_INVALID_ARGUMENT, "unknown launch flag bits 0x%x", flags);
    if (T < 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "num_tokens %lld", (long long)T);
    if (T == 0)
        return MSA_OK;

    const int64_t W = Htot * D;
    if (!positions || !slots)
        return fail(MSA_ERR_INVALID_ARGUMENT, "positions and slot_mapping are required");
    int64_t tmp;
    if (rows) {
        if (!qkv)
            return fail(MSA_ERR_INVALID_ARGUMENT, "qkv is required");
        if (row_stride < W)
            return fail(MSA_ERR_INVALID_ARGUMENT, "qkv_row_stride %lld < row width %lld",
                        (long long)row_stride, (long long)W);
        if (!aligned(qkv, 16) || row_stride % 8)
            return fail(MSA_ERR_MISALIGNED, "qkv must be 16-byte aligned with a row stride of 8k elements");
        if (!mul_add_ok(T - 1, row_stride, W, &tmp))
            return fail(MSA_ERR_OFFSET_OVERFLOW, "token count times row size overflows int64");
    }
    if (!aligned(positions, 4) || !aligned(slots, 8))
        return fail(MSA_ERR_MISALIGNED, "positions / slot_mapping misaligned");
    if (!mul_add_ok(T, (int64_t)(Hq > Hiq ? Hq : Hiq) * D, 0, &tmp))
        return fail(MSA_ERR_OFFSET_OVERFLOW, "token count times row size overflows int64");
    if (page_table) {
        if (page_table_len <= 0)
            return fail(MSA_ERR_INVALID_ARGUMENT, "page_table given with length %lld",
                        (long long)page_table_len);
        if (!aligned(page_table, 4))
            return fail(MSA_ERR_MISALIGNED, "page_table misaligned");
    } else if (page_table_len < 0) {
        return fail(MSA_ERR_INVALID_ARGUMENT, "negative page_table_len");
    }
    if (Hq > 0 && (!q_out || !wq))
        return fail(MSA_ERR_INVALID_ARGUMENT, "Q heads need q_out and q_norm_w");
    if (Hiq > 0 && (!iq_out || !wiq))
        return fail(MSA_ERR_INVALID_ARGUMENT, "index-Q heads need idx_q_out and idx_q_norm_w");
    if ((q_out && !aligned(q_out, 16)) || (iq_out && !aligned(iq_out, 16)))
        return fail(MSA_ERR_MISALIGNED, "q_out / idx_q_out must be 16-byte aligned");
    for (const void *w : {wq, wk, wiq, wik})
        if (w && !aligned(w, 2))
            return fail(MSA_ERR_MISALIGNED, "norm weight misaligned");
    if (Hkv > 0 && (!kc || !vc))
        return fail(MSA_ERR_INVALID_ARGUMENT, "K/V heads need k_cache and v_cache");
    if (Hkv > 0 && !wk)
        return fail(MSA_ERR_INVALID_ARGUMENT, "K heads need k_norm_w");
    if (ikc && Hik > 0 && !wik)
        return fail(MSA_ERR_INVALID_ARGUMENT, "index-K heads need idx_k_norm_w");
    bool any_fp8 = false;
    struct { const char *name; const msa_cache_desc *c; int64_t heads; } cs[3] = {
        {"k_cache", kc, Hkv}, {"v_cache", vc, Hkv}, {"idx_k_cache", ikc, Hik}};
    for (auto &e : cs) {
        if (!e.c)
            continue;
        msa_status s = check_cache(e.name, e.c, e.heads, D, P);
        if (s != MSA_OK)
            return s;
        any_fp8 |= e.c->dtype == MSA_DTYPE_FP8_E4M3;
    }
    if (any_fp8 && !scales)
        return fail(MSA_ERR_INVALID_ARGUMENT, "FP8 caches need scales");
    if (scales && !aligned(scales, 4))
        return fail(MSA_ERR_MISALIGNED, "scales misaligned");
    return MSA_OK;
}

// ---------------------------------------------------------------------------
// host side: launch
// ---------------------------------------------------------------------------

struct Variant {
    const void *fn;
    int threads;
    int id;
};

template <int D, int NT>
Variant variant_of(int id)
{
    return Variant{reinterpret_cast<const void *>(&msa_producer_kernel<D, NT>), NT, id};
}

constexpr int kNumVariants = 6;

int64_t htot_of(const msa_producer_cfg *cfg)
{
    return (int64_t)cfg->num_q_heads + 2 * (int64_t)cfg->num_kv_heads + cfg->num_idx_q_heads +
           cfg->num_idx_k_heads;
}

// Threads per CTA: enough lanes for one pass over a token's head rows, at most 256.
Variant pick_variant(const msa_producer_cfg *cfg)
{
    const int64_t lanes = htot_of(cfg) * (cfg->head_dim / 16);
    if (cfg->head_dim == 128) {
        if (lanes <= 64) return variant_of<128, 64>(0);
        if (lanes <= 128) return variant_of<128, 128>(1);
        return variant_of<128, 256>(2);
    }
    if (lanes <= 64) return variant_of<64, 64>(3);
    if (lanes <= 128) return variant_of<64, 128>(4);
    return variant_of<64, 256>(5);
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct DeviceInfo {
    int sms = 0;
    int max_dyn_smem[kNumVariants] = {};  // 0: not configured yet on this device
};
DeviceInfo g_dev[kMaxDevices];

// Configures the variant on the current device once (its dynamic shared-memory
// limit) and returns the launch shape.  Host-side queries only; nothing is
// enqueued, so this is safe while a stream is being captured.
msa_status launch_shape(const msa_producer_cfg *cfg, int64_t T, int32_t flags, Variant *v,
                        int *grid, int *smem)
{
    *v = pick_variant(cfg);
    const int64_t row_bytes = htot_of(cfg) * cfg->head_dim * 2;
    *smem = (int)(kStages * row_bytes);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(MSA_ERR_CUDA, "cudaGetDevice failed");
    DeviceInfo &di = g_dev[dev];
    int max_dyn, sms;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        max_dyn = di.max_dyn_smem[v->id];
        sms = di.sms;
    }
    if (max_dyn == 0 || sms == 0) {
        int optin = 0;
        cudaFuncAttributes fa;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaFuncGetAttributes(&fa, v->fn) != cudaSuccess)
            return fail(MSA_ERR_CUDA, "device query failed");
        max_dyn = optin - (int)fa.sharedSizeBytes;
        if (cudaFuncSetAttribute(v->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn) !=
            cudaSuccess)
            return fail(MSA_ERR_CUDA, "cudaFuncSetAttribute failed");
        std::lock_guard<std::mutex> lk(g_mu);
        di.max_dyn_smem[v->id] = max_dyn;
        di.sms = sms;
    }
    if (*smem > max_dyn)
        return fail(MSA_ERR_UNSUPPORTED, "a row of %lld bytes does not fit the shared-memory ring",
                    (long long)row_bytes);
    if (!(flags & MSA_LAUNCH_PERSISTENT)) {   // one token per CTA
        *grid = (int)(T < 0x7fffffff ? T : 0x7fffffff);
        return MSA_OK;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, v->fn, v->threads, *smem) !=
            cudaSuccess ||
        per_sm <= 0)
        return fail(MSA_ERR_CUDA, "occupancy query failed");
    const int64_t cap = (int64_t)sms * per_sm;
    *grid = (int)(T < cap ? T : cap);
    return MSA_OK;
}

void fill_cache(CacheArgs &a, const msa_cache_desc *c)
{
    if (!c) {
        memset(&a, 0, sizeof a);
        return;
    }
    a.data = static_cast<uint8_t *>(c->data);
    a.num_pages = c->num_pages;
    a.stride_page = c->stride_page;
    a.stride_head = c->stride_head;
    a.stride_token = c->stride_token;
    a.fp8 = c->dtype == MSA_DTYPE_FP8_E4M3;
    a.pad = 0;
}

}  // namespace

extern "C" {

msa_status msa_producer_validate(const msa_producer_cfg *cfg, int64_t num_tokens, const void *qkv,
                                 int64_t qkv_row_stride, const int32_t *positions,
                                 const int64_t *slot_mapping, const int32_t *page_table,
                                 int64_t page_table_len, const void *q_norm_w, const void *k_norm_w,
                                 const void *idx_q_norm_w, const void *idx_k_norm_w, void *q_out,
                                 void *idx_q_out, const msa_cache_desc *k_cache,
                                 const msa_cache_desc *v_cache, const msa_cache_desc *idx_k_cache,
                                 const float *scales, int32_t launch_flags)
{
    return validate(cfg, num_tokens, qkv, qkv_row_stride, positions, slot_mapping, page_table,
                    page_table_len, q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out,
                    idx_q_out, k_cache, v_cache, idx_k_cache, scales, launch_flags);
}

msa_status msa_producer_forward(const msa_producer_cfg *cfg, int64_t num_tokens, const void *qkv,
                                int64_t qkv_row_stride, const int32_t *positions,
                                const int64_t *slot_mapping, const int32_t *page_table,
                                int64_t page_table_len, const void *q_norm_w, const void *k_norm_w,
                                const void *idx_q_norm_w, const void *idx_k_norm_w, void *q_out,
                                void *idx_q_out, const msa_cache_desc *k_cache,
                                const msa_cache_desc *v_cache, const msa_cache_desc *idx_k_cache,
                                const float *scales, int32_t launch_flags, cudaStream_t stream)
{
    msa_status s = validate(cfg, num_tokens, qkv, qkv_row_stride, positions, slot_mapping,
                            page_table, page_table_len, q_norm_w, k_norm_w, idx_q_norm_w,
                            idx_k_norm_w, q_out, idx_q_out, k_cache, v_cache, idx_k_cache, scales,
                            launch_flags);
    if (s != MSA_OK || num_tokens == 0)
        return s;

    Params p;
    memset(&p, 0, sizeof p);
    p.qkv = static_cast<const uint16_t *>(qkv);
    p.row_stride = qkv_row_stride;
    p.positions = positions;
    p.slots = slot_mapping;
    p.page_table = page_table;
    p.page_table_len = page_table ? page_table_len : 0;
    p.norm_w[0] = static_cast<const uint16_t *>(q_norm_w);
    p.norm_w[1] = static_cast<const uint16_t *>(k_norm_w);
    p.norm_w[2] = static_cast<const uint16_t *>(idx_q_norm_w);
    p.norm_w[3] = static_cast<const uint16_t *>(idx_k_norm_w);
    p.q_out = static_cast<uint16_t *>(q_out);
    p.idx_q_out = static_cast<uint16_t *>(idx_q_out);
    fill_cache(p.cache[0], cfg->num_kv_heads > 0 ? k_cache : nullptr);
    fill_cache(p.cache[1], cfg->num_kv_heads > 0 ? v_cache : nullptr);
    fill_cache(p.cache[2], cfg->num_idx_k_heads > 0 ? idx_k_cache : nullptr);
    p.scales = scales;
    p.num_tokens = num_tokens;
    p.hq = cfg->num_q_heads;
    p.hkv = cfg->num_kv_heads;
    p.hiq = cfg->num_idx_q_heads;
    p.hik = cfg->num_idx_k_heads;
    p.htot = (int32_t)htot_of(cfg);
    p.row_bytes = p.htot * cfg->head_dim * 2;
    p.rotary_dim = cfg->rotary_dim;
    p.rope_style = cfg->rope_style;
    p.page_size = cfg->page_size;
    p.page_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == cfg->page_size)
            p.page_shift = sh;
    p.scale_mode = cfg->scale_mode;
    p.pdl = (launch_flags & MSA_LAUNCH_PDL) ? 1 : 0;
#ifdef MSA_CHECKED
    p.out_hi[0] = p.q_out ? reinterpret_cast<const uint8_t *>(p.q_out) +
                                num_tokens * (int64_t)cfg->num_q_heads * cfg->head_dim * 2
                          : nullptr;
    p.out_hi[1] = p.idx_q_out ? reinterpret_cast<const uint8_t *>(p.idx_q_out) +
                                    num_tokens * (int64_t)cfg->num_idx_q_heads * cfg->head_dim * 2
                              : nullptr;
    for (int ci = 0; ci < 3; ++ci)
        p.cache_hi[ci] = msa_internal_cache_end(&p.cache[ci].data, ci == 2 ? cfg->num_idx_k_heads
                                                                           : cfg->num_kv_heads,
                                                p.cache[ci].num_pages, p.cache[ci].stride_page,
                                                p.cache[ci].stride_head, p.cache[ci].stride_token,
                                                p.cache[ci].fp8 ? 1 : 2, cfg->head_dim,
                                                cfg->page_size);
#endif
    p.rms_eps = cfg->rms_eps;
    // RoPE frequencies theta^(-2k/rd), evaluated in double and rounded once
    for (int k = 0; k < cfg->rotary_dim / 2; ++k)
        p.inv_freq[k] = (float)(1.0 / std::pow((double)cfg->rope_theta,
                                               2.0 * (double)k / (double)cfg->rotary_dim));

    Variant v;
    int grid = 0, smem = 0;
    s = launch_shape(cfg, num_tokens, launch_flags, &v, &grid, &smem);
    if (s != MSA_OK)
        return s;

    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3((unsigned)v.threads);
    lc.dynamicSmemBytes = (size_t)smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    if (launch_flags & MSA_LAUNCH_PDL) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
    }
    void *args[] = {&p};
    cudaError_t e = cudaLaunchKernelExC(&lc, v.fn, args);
    if (e != cudaSuccess)
        return fail(MSA_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    return MSA_OK;
}

msa_status msa_producer_launch_shape(const msa_producer_cfg *cfg, int64_t num_tokens,
                                     int32_t launch_flags, int32_t *grid, int32_t *block,
                                     int32_t *smem_bytes)
{
    if (!cfg || !grid || !block || !smem_bytes || num_tokens < 0)
        return fail(MSA_ERR_INVALID_ARGUMENT, "launch_shape: bad arguments");
    if (cfg->head_dim != 64 && cfg->head_dim != 128)
        return fail(MSA_ERR_UNSUPPORTED, "head_dim %d", cfg->head_dim);
    if (htot_of(cfg) <= 0 || htot_of(cfg) * cfg->head_dim * 2 > kMaxRowBytes)
        return fail(MSA_ERR_UNSUPPORTED, "head counts");
    Variant v;
    int g = 0, sm = 0;
    msa_status s = launch_shape(cfg, num_tokens, launch_flags, &v, &g, &sm);
    if (s != MSA_OK)
        return s;
    *grid = g;
    *block = v.threads;
    *smem_bytes = sm;
    return MSA_OK;
}

msa_status msa_host_buffer_device_address(const void *host_ptr, void **device_ptr)
{
    g_detail[0] = '\0';
    if (!host_ptr || !device_ptr)
        return fail(MSA_ERR_INVALID_ARGUMENT, "host_buffer_device_address: NULL argument");
    cudaPointerAttributes a;
    memset(&a, 0, sizeof a);
    if (cudaPointerGetAttributes(&a, host_ptr) != cudaSuccess) {
        (void)cudaGetLastError();  // an unregistered pointer is not a sticky error
        return fail(MSA_ERR_INVALID_ARGUMENT, "pointer unknown to the CUDA runtime");
    }
    if (a.type != cudaMemoryTypeHost || !a.devicePointer)
        return fail(MSA_ERR_INVALID_ARGUMENT, "not pinned, device-mapped host memory (type %d)",
                    (int)a.type);
    *device_ptr = a.devicePointer;
    return MSA_OK;
}

const char *msa_status_string(msa_status status)
{
    switch (status) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARGUMENT: return "MSA_ERR_INVALID_ARGUMENT";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_MISALIGNED: return "MSA_ERR_MISALIGNED";
    case MSA_ERR_OFFSET_OVERFLOW: return "MSA_ERR_OFFSET_OVERFLOW";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    }
    return "MSA_ERR_UNKNOWN";
}

const char *msa_last_error_detail(void) { return g_detail; }

}  // extern "C"

// Shared with the indexer's translation unit (declared in msa_internal.h).
void msa_internal_set_detail(const char *msg)
{
    snprintf(g_detail, sizeof g_detail, "%s", msg);
}

msa_status msa_internal_validate_producer(const msa_producer_cfg *cfg, int64_t num_tokens,
                                          const int32_t *positions, const int64_t *slot_mapping,
                                          const int32_t *page_table, int64_t page_table_len,
                                          const void *q_norm_w, const void *k_norm_w,
                                          const void *idx_q_norm_w, const void *idx_k_norm_w,
                                          void *q_out, void *idx_q_out,
                                          const msa_cache_desc *k_cache,
                                          const msa_cache_desc *v_cache,
                                          const msa_cache_desc *idx_k_cache, const float *scales)
{
    return validate(cfg, num_tokens, nullptr, 0, positions, slot_mapping, page_table,
                    page_table_len, q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out,
                    idx_q_out, k_cache, v_cache, idx_k_cache, scales, 0, false);
}

msa_status msa_internal_check_cache(const char *name, const msa_cache_desc *c, int64_t heads,
                                    int32_t head_dim, int32_t page_size)
{
    return check_cache(name, c, heads, head_dim, page_size);
}

// First byte past the furthest element a write to a cache can reach (nullptr for
// an absent or empty cache); the checked build's upper bound for its stores.
const uint8_t *msa_internal_cache_end(uint8_t *const *data, int64_t heads, int64_t num_pages,
                                      int64_t stride_page, int64_t stride_head,
                                      int64_t stride_token, int64_t elem_size, int32_t head_dim,
                                      int32_t page_size)
{
    if (!*data || num_pages <= 0 || heads <= 0)
        return *data;
    const int64_t last = (num_pages - 1) * stride_page + (heads - 1) * stride_head +
                         (int64_t)(page_size - 1) * stride_token + head_dim;
    return *data + last * elem_size;
}

extern "C" msa_status msa_checked_violations(uint64_t *count, int32_t reset)
{
    if (!count)
        return fail(MSA_ERR_INVALID_ARGUMENT, "count is NULL");
    *count = 0;
#ifdef MSA_CHECKED
    unsigned long long v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpyFromSymbol(&v, g_msa_violations, sizeof v) != cudaSuccess)
        return fail(MSA_ERR_CUDA, "reading the violation counter failed");
    uint64_t w = 0;
    if (msa_internal_projection_violations(&w, reset) != MSA_OK)
        return fail(MSA_ERR_CUDA, "reading the projection's violation counter failed");
    if (reset) {
        const unsigned long long z = 0;
        if (cudaMemcpyToSymbol(g_msa_violations, &z, sizeof z) != cudaSuccess)
            return fail(MSA_ERR_CUDA, "resetting the violation counter failed");
    }
    *count = (uint64_t)v + w;
    return MSA_OK;
#else
    (void)reset;
    return fail(MSA_ERR_UNSUPPORTED, "not a checked build (compile with -DMSA_CHECKED)");
#endif
}
