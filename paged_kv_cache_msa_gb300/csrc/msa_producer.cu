// MiniMax-M3 MSA per-layer fused producer and paged-cache write for sm_103a.
//
// What it computes is stated in include/msa_producer.h, after "[None][perf] Fuse
// MiniMax-M3 QKV and index projection" (TensorRT-LLM PR 18205, Description) and
// "[None][perf] Fuse MiniMax-M3 MSA per-layer KV-cache writes into one kernel"
// (PR 18614, "The problem" / "The fix").
//
// Design (GB300): the path is HBM-bound streaming work (~2-3 flop per byte, no
// dense contraction), so it runs on the CUDA cores with wide coalesced memory
// operations; there is nothing here for the tensor cores.
//   * One CTA owns one token at a time.  Its threads cover the token's projection
//     row in 16-byte chunks (8 bf16): a head row of D elements is D/8 adjacent
//     lanes of one warp, so every load is a fully coalesced 128/256-byte segment
//     and every cache row store is one 64/128-byte segment.
//   * All of a thread's row loads are issued before any arithmetic, so a CTA has
//     the whole 22.8 KB row in flight at once.
//   * The per-token work that is the same for every head -- the slot -> (page,
//     offset) derivation and the rotary cos/sin table -- is done once per token
//     by a few threads into shared memory (double-buffered, one barrier per
//     token), instead of once per head row.
//   * RMSNorm's sum of squares is reduced with xor shuffles inside the head row's
//     lane group; the NeoX rotate-half partner of a lane's 8 elements sits in one
//     other lane of the same group (rotary_dim a multiple of 16), fetched with one
//     shuffle per element; GPT-J pairs lie inside a lane.
//   * FP8 E4M3 packing uses the cvt.rn.satfinite.e4m3x2.f32 instruction; bf16
//     packing uses cvt.rn.bf16x2.f32.
//   * One-shot grid (a CTA per token) or a persistent grid of at most
//     SMs x resident CTAs that strides over the tokens.  No kernel waits on
//     another CTA, a flag or a barrier other than __syncthreads, so nothing can
//     spin.  Optional programmatic dependent launch.

#include "msa_producer.h"

#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace {

constexpr int kMaxRotaryHalf = 64;   // rotary_dim / 2 <= head_dim / 2 <= 64
constexpr int kMaxHeadScales = 256;  // per-head scale mode: 2*Hkv + Hik <= 256

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
    int32_t rotary_dim;
    int32_t rope_style;
    int32_t page_size;
    int32_t page_shift;             // log2(page_size) when a power of two, else -1
    int32_t scale_mode;
    int32_t num_chunks;             // 8-element chunks in one token's row section
    float rms_eps;
    float inv_freq[kMaxRotaryHalf];
};

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_row_chunk(const uint16_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// bf16 pair -> two floats (element 0 is the low half)
__device__ __forceinline__ void unpack_bf16x2(uint32_t v, float &lo, float &hi)
{
    lo = __uint_as_float(v << 16);
    hi = __uint_as_float(v & 0xFFFF0000u);
}

// two floats -> bf16 pair, round to nearest even; `lo` lands at the lower address
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// four floats -> four E4M3 bytes, round to nearest even, saturating to +-448
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d)
{
    unsigned short lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ float bf16_to_f32(uint16_t h)
{
    return __uint_as_float(((uint32_t)h) << 16);
}

// ---------------------------------------------------------------------------
// the producer kernel
// ---------------------------------------------------------------------------
//
// D      head_dim (64 or 128); a head row is G = D/8 lanes of 8 elements
// NT     threads per CTA (a multiple of 32, hence of G)
// MAXCH  chunks a thread holds in registers at once; a row of more than
//        NT*MAXCH chunks is processed in several batches
template <int D, int NT, int MAXCH>
__global__ void __launch_bounds__(NT) msa_producer_kernel(const __grid_constant__ Params p)
{
    constexpr int G = D / 8;
    static_assert(NT % 32 == 0 && 32 % G == 0, "a head row must sit inside one warp");

    __shared__ __align__(16) float s_w[4][D];
    __shared__ float s_cos[2][kMaxRotaryHalf];
    __shared__ float s_sin[2][kMaxRotaryHalf];
    __shared__ float s_inv_scale[kMaxHeadScales];
    __shared__ long long s_page[2];
    __shared__ int s_off[2];
    __shared__ int s_valid[2];

    const int tid = threadIdx.x;
    const int g = tid % G;  // this thread's 8-element slot inside every head row it touches

    // Inputs may be produced by the previous kernel in the stream (programmatic
    // dependent launch): wait for it before reading them.  A no-op otherwise.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    for (int i = tid; i < 4 * D; i += NT) {
        const uint16_t *w = p.norm_w[i / D];
        s_w[i / D][i % D] = w ? bf16_to_f32(w[i % D]) : 1.0f;
    }
    {
        const int nscales = p.scale_mode == MSA_SCALE_PER_HEAD ? 2 * p.hkv + p.hik : 3;
        if (p.scales)
            for (int i = tid; i < nscales; i += NT)
                s_inv_scale[i] = 1.0f / p.scales[i];
    }
    // Let the next kernel in the stream start its own prologue.
    asm volatile("griddepcontrol.launch_dependents;" :::);

    // RoPE geometry of this lane (fixed for every head row and token)
    const int rd = p.rotary_dim;
    const bool neox = p.rope_style == MSA_ROPE_NEOX;
    const bool rot = 8 * g < rd;
    const bool first_half = 8 * g < rd / 2;
    const int partner = neox ? (first_half ? g + rd / 16 : g - rd / 16) : g;
    const int fbase = neox ? (first_half ? 8 * g : 8 * g - rd / 2) : 4 * g;

    const int hq = p.hq, hkv = p.hkv, hiq = p.hiq;
    const int e_k = hq, e_v = hq + hkv, e_iq = hq + 2 * hkv, e_ik = hq + 2 * hkv + hiq;

    int buf = 0;
    for (int64_t t = blockIdx.x; t < p.num_tokens; t += gridDim.x, buf ^= 1) {
        const uint16_t *row = p.qkv + t * p.row_stride;
        float cs[8], sn[8];

        for (int c0 = 0; c0 < p.num_chunks; c0 += NT * MAXCH) {
            // 1. issue every row load of this batch
            uint4 raw[MAXCH];
#pragma unroll
            for (int k = 0; k < MAXCH; ++k) {
                const int c = c0 + k * NT + tid;
                raw[k] = c < p.num_chunks ? ld_row_chunk(row + 8 * c) : make_uint4(0, 0, 0, 0);
            }

            if (c0 == 0) {
                // 2. per-token work shared by every head row
                if (tid < rd / 2) {
                    const float a = (float)__ldg(p.positions + t) * p.inv_freq[tid];
                    float s, c;
                    sincosf(a, &s, &c);
                    s_cos[buf][tid] = c;
                    s_sin[buf][tid] = s;
                }
                if (tid == NT - 1) {
                    const long long ls = __ldg(p.slots + t);
                    long long page = -1;
                    int off = 0;
                    if (ls >= 0) {
                        long long blk;
                        if (p.page_shift >= 0) {
                            blk = ls >> p.page_shift;
                            off = (int)(ls & (long long)(p.page_size - 1));
                        } else {
                            blk = ls / p.page_size;
                            off = (int)(ls - blk * p.page_size);
                        }
                        if (p.page_table)
                            page = blk < p.page_table_len ? (long long)__ldg(p.page_table + blk) : -1;
                        else
                            page = blk;
                    }
                    int valid = 0;
#pragma unroll
                    for (int ci = 0; ci < 3; ++ci)
                        if (p.cache[ci].data && page >= 0 && page < p.cache[ci].num_pages)
                            valid |= 1 << ci;
                    s_page[buf] = page;
                    s_off[buf] = off;
                    s_valid[buf] = valid;
                }
                __syncthreads();
                if (rot) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int f = neox ? fbase + j : fbase + (j >> 1);
                        cs[j] = s_cos[buf][f];
                        sn[j] = s_sin[buf][f];
                    }
                }
            }
            const long long page = s_page[buf];
            const int off = s_off[buf];
            const int valid = s_valid[buf];

            // 3. normalise, rotate, convert and store each chunk
#pragma unroll
            for (int k = 0; k < MAXCH; ++k) {
                const int c = c0 + k * NT + tid;
                const bool active = c < p.num_chunks;
                const int hr = c / G;  // head row inside the token's row

                float x[8];
                unpack_bf16x2(raw[k].x, x[0], x[1]);
                unpack_bf16x2(raw[k].y, x[2], x[3]);
                unpack_bf16x2(raw[k].z, x[4], x[5]);
                unpack_bf16x2(raw[k].w, x[6], x[7]);

                float ss = 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    ss += x[j] * x[j];
#pragma unroll
                for (int o = 1; o < G; o <<= 1)
                    ss += __shfl_xor_sync(0xffffffffu, ss, o, G);

                // section of this head row: 0 Q, 1 K, 2 V, 3 idx-Q, 4 idx-K
                int sec, h;
                if (hr < e_k) { sec = 0; h = hr; }
                else if (hr < e_v) { sec = 1; h = hr - e_k; }
                else if (hr < e_iq) { sec = 2; h = hr - e_v; }
                else if (hr < e_ik) { sec = 3; h = hr - e_iq; }
                else { sec = 4; h = hr - e_ik; }
                const bool normed = sec != 2;
                const int widx = sec == 0 ? 0 : sec == 1 ? 1 : sec == 3 ? 2 : 3;

                float y[8];
                if (normed) {
                    const float r = 1.0f / sqrtf(ss / (float)D + p.rms_eps);
                    const float4 w0 = *reinterpret_cast<const float4 *>(&s_w[widx][8 * g]);
                    const float4 w1 = *reinterpret_cast<const float4 *>(&s_w[widx][8 * g + 4]);
                    y[0] = (x[0] * r) * w0.x; y[1] = (x[1] * r) * w0.y;
                    y[2] = (x[2] * r) * w0.z; y[3] = (x[3] * r) * w0.w;
                    y[4] = (x[4] * r) * w1.x; y[5] = (x[5] * r) * w1.y;
                    y[6] = (x[6] * r) * w1.z; y[7] = (x[7] * r) * w1.w;
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        y[j] = x[j];
                }

                if (neox) {
                    // every lane takes part in the shuffles; only rotated lanes of
                    // normed sections use the result
                    float pv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        pv[j] = __shfl_sync(0xffffffffu, y[j], partner, G);
                    if (normed && rot) {
                        if (first_half) {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                y[j] = y[j] * cs[j] - pv[j] * sn[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                y[j] = y[j] * cs[j] + pv[j] * sn[j];
                        }
                    }
                } else if (normed && rot) {
#pragma unroll
                    for (int j = 0; j < 8; j += 2) {
                        const float u = y[j], v = y[j + 1];
                        y[j] = u * cs[j] - v * sn[j];
                        y[j + 1] = v * cs[j] + u * sn[j];
                    }
                }

                if (!active)
                    continue;
                if (sec == 0 || sec == 3) {
                    uint16_t *dst = sec == 0 ? p.q_out + ((int64_t)t * hq + h) * D + 8 * g
                                             : p.idx_q_out + ((int64_t)t * hiq + h) * D + 8 * g;
                    st_v4(dst, pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                          pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                } else {
                    const int ci = sec == 1 ? 0 : sec == 2 ? 1 : 2;
                    if (!((valid >> ci) & 1))
                        continue;
                    const CacheArgs &cc = p.cache[ci];
                    const int64_t e = page * cc.stride_page + (int64_t)h * cc.stride_head +
                                      (int64_t)off * cc.stride_token + 8 * g;
                    if (cc.fp8) {
                        const int si = p.scale_mode == MSA_SCALE_PER_HEAD
                                           ? (ci == 0 ? h : ci == 1 ? hkv + h : 2 * hkv + h)
                                           : ci;
                        const float inv = s_inv_scale[si];
                        st_v2(cc.data + e, pack_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv),
                              pack_e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv));
                    } else {
                        st_v4(cc.data + 2 * e, pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
                              pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
                    }
                }
            }
        }
    }
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

msa_status validate(const msa_producer_cfg *cfg, int64_t T, const void *qkv, int64_t row_stride,
                    const int32_t *positions, const int64_t *slots, const int32_t *page_table,
                    int64_t page_table_len, const void *wq, const void *wk, const void *wiq,
                    const void *wik, void *q_out, void *iq_out, const msa_cache_desc *kc,
                    const msa_cache_desc *vc, const msa_cache_desc *ikc, const float *scales,
                    int32_t flags)
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
    if (Htot * (D / 8) > (int64_t)1 << 30)
        return fail(MSA_ERR_UNSUPPORTED, "too many heads");
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
    if (!qkv || !positions || !slots)
        return fail(MSA_ERR_INVALID_ARGUMENT, "qkv, positions and slot_mapping are required");
    if (row_stride < W)
        return fail(MSA_ERR_INVALID_ARGUMENT, "qkv_row_stride %lld < row width %lld",
                    (long long)row_stride, (long long)W);
    if (!aligned(qkv, 16) || row_stride % 8)
        return fail(MSA_ERR_MISALIGNED, "qkv must be 16-byte aligned with a row stride of 8k elements");
    if (!aligned(positions, 4) || !aligned(slots, 8))
        return fail(MSA_ERR_MISALIGNED, "positions / slot_mapping misaligned");
    int64_t tmp;
    if (!mul_add_ok(T - 1, row_stride, W, &tmp) || !mul_add_ok(T, (int64_t)(Hq > Hiq ? Hq : Hiq) * D, 0, &tmp))
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
};

template <int D, int NT, int MAXCH>
Variant variant_of()
{
    return Variant{reinterpret_cast<const void *>(&msa_producer_kernel<D, NT, MAXCH>), NT};
}

Variant pick_variant(int32_t D)
{
    if (D == 128)
        return variant_of<128, 256, 6>();
    return variant_of<64, 128, 6>();
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];
int g_blocks_per_sm[kMaxDevices][2];

msa_status grid_for(const msa_producer_cfg *cfg, int64_t T, int32_t flags, int *grid, int *block)
{
    const Variant v = pick_variant(cfg->head_dim);
    *block = v.threads;
    if (!(flags & MSA_LAUNCH_PERSISTENT)) {
        *grid = (int)(T < 0x7fffffff ? T : 0x7fffffff);
        return MSA_OK;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(MSA_ERR_CUDA, "cudaGetDevice failed");
    const int vi = cfg->head_dim == 128 ? 0 : 1;
    int sms, per_sm;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        sms = g_sms[dev];
        per_sm = g_blocks_per_sm[dev][vi];
    }
    if (sms == 0 || per_sm == 0) {
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return fail(MSA_ERR_CUDA, "cudaDeviceGetAttribute failed");
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, v.fn, v.threads, 0) != cudaSuccess ||
            per_sm <= 0)
            return fail(MSA_ERR_CUDA, "occupancy query failed");
        std::lock_guard<std::mutex> lk(g_mu);
        g_sms[dev] = sms;
        g_blocks_per_sm[dev][vi] = per_sm;
    }
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
    p.rotary_dim = cfg->rotary_dim;
    p.rope_style = cfg->rope_style;
    p.page_size = cfg->page_size;
    p.page_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == cfg->page_size)
            p.page_shift = sh;
    p.scale_mode = cfg->scale_mode;
    const int64_t Htot = (int64_t)p.hq + 2 * p.hkv + p.hiq + p.hik;
    p.num_chunks = (int32_t)(Htot * (cfg->head_dim / 8));
    p.rms_eps = cfg->rms_eps;
    // RoPE frequencies theta^(-2k/rd), evaluated in double and rounded once
    for (int k = 0; k < cfg->rotary_dim / 2; ++k)
        p.inv_freq[k] = (float)(1.0 / std::pow((double)cfg->rope_theta,
                                               2.0 * (double)k / (double)cfg->rotary_dim));

    int grid = 0, block = 0;
    s = grid_for(cfg, num_tokens, launch_flags, &grid, &block);
    if (s != MSA_OK)
        return s;

    const Variant v = pick_variant(cfg->head_dim);
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.gridDim = dim3((unsigned)grid);
    lc.blockDim = dim3((unsigned)block);
    lc.dynamicSmemBytes = 0;
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
    int g = 0, b = 0;
    msa_status s = grid_for(cfg, num_tokens, launch_flags, &g, &b);
    if (s != MSA_OK)
        return s;
    *grid = g;
    *block = b;
    *smem_bytes = 0;
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
