// The wide [Q | K | V | index-Q | index-K] projection on the tcgen05 tensor cores,
// with the MSA producer in its epilogue ("[None][perf] Fuse MiniMax-M3 QKV and
// index projection", Description, AFTER diagram: one wider fused GEMM feeding one
// fused producer).  The producer's arithmetic is the one msa_producer_forward
// applies to a row; only where the row comes from differs: here it is the fp32
// accumulator of a 128-token x 256-output tile in tensor memory, rounded to bf16.
//
// Kernel structure: persistent clusters of two CTAs (one per SM), 320 threads
// each (kThreads = 64 + 32 x 8).  A cluster computes 256-token x 256-output tiles
// with the 2-SM MMA: CTA r of the pair holds tokens [128r, 128r + 128) of the tile
// and weight rows [128r, 128r + 128) of its outputs, and its tensor memory
// receives the accumulator of its own 128 tokens over all 256 outputs.  Per CTA:
//   warp 0      TMA producer: 128-byte K blocks (64 bf16 or 128 E4M3 elements) of
//               its hidden rows and weight rows into a 7-stage shared-memory ring
//               (128-byte swizzle, K-major); the copies of both CTAs complete on
//               the leader's barrier
//   warp 1      tensor-memory owner; in the leader CTA (rank 0) one thread issues
//               tcgen05.mma.cta_group::2 (kind::f16 for bf16, kind::f8f6f4 for
//               E4M3; M 256, N 256) into one of two accumulators (2 x 256 columns),
//               so that the epilogue of a tile overlaps the main loop of the next,
//               and commits to both CTAs
//   warps 2..9  epilogue: warp w reads tensor-memory lane quarter w & 3 (thread
//               r of it owns token row r of its CTA's half of the tile) and takes
//               the head group (w - 2) >> 2, so the two warps of a lane quarter
//               split the tile's heads between them; each runs the producer on
//               its heads
// Per SM a K block moves 32 KB through shared memory for 128 x 256 x 64 bf16 MACs
// (half of what a one-SM 128 x 256 tile needs), which is what lets 7 stages --
// about 2 us of loads -- be in flight.
//
// At most 128 tokens the K dimension is split over a cluster of up to 8 CTAs
// instead (msa_projection_splitk_kernel, section "small batches" below).
//
// Tiles are visited output-group-major: for each group of n_group 256-wide output
// tiles, every 256-token tile in order, so that the group's weight panels stay in
// L2 while the hidden rows stream through once per group.
//
// Every mbarrier wait is bounded by %globaltimer; a wait that runs out sets
// MSA_STATUS_WAIT_TIMEOUT in the caller's status word and the CTA winds down
// (waiting, again bounded, for its own copies and MMAs in flight) and releases
// its tensor memory.

#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched at run time
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "msa_internal.h"
#include "msa_producer.h"
#include "msa_projection.h"

// K blocks of weight prefetched into L2 ahead of the ring at small batches (a build-time
// knob; 0 = off).  Measured at decode 64 / 256 / 1,024 tokens: 8 and 16 blocks ahead were 0-5%
// slower than none (the weight stream got no faster), so it is off.
#ifndef MSA_PROJ_PREFETCH
#define MSA_PROJ_PREFETCH 0
#endif
#ifndef MSA_PROJ_PREFETCH_MTILES
#define MSA_PROJ_PREFETCH_MTILES 4   // up to this many 256-token tiles
#endif
#ifndef MSA_PROJ_NGROUP
#define MSA_PROJ_NGROUP 8
#endif
#ifndef MSA_PROJ_STAGES
#define MSA_PROJ_STAGES 7
#endif

namespace {

constexpr int kBM = 128;                  // tokens per CTA and tile half: tensor-memory lanes
constexpr int kPairM = 2 * kBM;           // tokens per cluster tile (the 2-SM MMA's M)
constexpr int kBN = 256;                  // projection outputs per tile: accumulator columns
constexpr int kHalfN = kBN / 2;           // weight rows each CTA stages
constexpr int kBKBytes = 128;             // K bytes per stage: one 128-byte swizzle row
constexpr int kStages = MSA_PROJ_STAGES;
constexpr int kEpilogueWarps = 8;     // two per tensor-memory lane quarter
constexpr int kThreads = 64 + 32 * kEpilogueWarps;
constexpr uint32_t kTileABytes = kBM * kBKBytes;
constexpr uint32_t kTileBBytes = kHalfN * kBKBytes;
constexpr uint32_t kStageBytes = kTileABytes + kTileBBytes;  // per CTA
constexpr int kDynSmem = kStages * kStageBytes + 1024;        // + alignment slack for the ring
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr int kMaxRotaryHalf = 64;
constexpr unsigned long long kWaitLimitNs = MSA_WAIT_LIMIT_NS;

// tcgen05 instruction descriptors: fp32 accumulator (bits 4-5 = 1), A and B formats
// at bits 7-9 and 10-12 (kind::f16: 1 = bf16; kind::f8f6f4: 0 = E4M3), both K-major
// (bits 15, 16 = 0), N >> 3 at bit 17, M >> 4 at bit 24 (M = 256: the pair's tile).
constexpr uint32_t kIdescShape = ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kPairM >> 4) << 24);
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) | kIdescShape;
constexpr uint32_t kIdescE4m3 = (1u << 4) | kIdescShape;

struct CacheArgs {
    uint8_t *data;  // nullptr: not written
    int64_t num_pages;
    int64_t stride_page;
    int64_t stride_head;
    int64_t stride_token;
    int32_t fp8;
    int32_t pad;
};

struct Params {
    const int32_t *positions;
    const int64_t *slots;
    const int32_t *page_table;
    int64_t page_table_len;
    const uint16_t *norm_w[4];  // q, k, idx_q, idx_k
    uint16_t *q_out;
    uint16_t *idx_q_out;
    CacheArgs cache[3];         // k, v, idx_k
    const float *scales;
    uint16_t *rows_out;
    int64_t rows_out_stride;
    const float *hidden_scales;  // per token (nullptr: 1)
    const float *weight_scales;  // per output (nullptr: 1)
    uint32_t *status;
    int64_t num_tokens;
    int32_t num_k_blocks;
    int32_t m_tiles, n_tiles, n_group;
    int32_t split;              // CTAs per cluster sharing an output tile's K (small batches)
    int32_t prefetch;           // K blocks the weight tile is fetched into L2 ahead (0: none)
    int32_t hq, hkv, hiq, hik, htot;
    int32_t rotary_dim;
    int32_t rope_style;
    int32_t page_size;
    int32_t page_shift;
    int32_t scale_mode;
    float rms_eps;
    float inv_freq[kMaxRotaryHalf];
#ifdef MSA_CHECKED
    const uint8_t *out_hi[2];   // first byte past q_out, idx_q_out
    const uint8_t *cache_hi[3]; // first byte past each cache's reachable extent
    const uint8_t *rows_hi;     // first byte past rows_out
#endif
};

#ifdef MSA_CHECKED
// Checked build: a global store whose bytes leave its destination's extent is
// skipped and counted here.
__device__ unsigned long long g_msa_projection_violations;

__device__ __forceinline__ bool msa_in_range(const void *ptr, int n, const void *lo, const void *hi)
{
    const uint8_t *b = static_cast<const uint8_t *>(ptr);
    if (b >= static_cast<const uint8_t *>(lo) && b + n <= static_cast<const uint8_t *>(hi))
        return true;
    atomicAdd(&g_msa_projection_violations, 1ull);
    return false;
}
#define MSA_GUARD(ptr, n, lo, hi) if (!msa_in_range((ptr), (n), (lo), (hi))) {} else
#else
#define MSA_GUARD(ptr, n, lo, hi)
#endif

// ---------------------------------------------------------------------------
// PTX wrappers
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

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
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
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try(bar, parity))
        return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try(bar, parity))
            return true;
        if ((n & 63) == 0 && globaltimer() - t0 > kWaitLimitNs)
            return false;
    }
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Arrive on an mbarrier of any CTA of the cluster (shared::cluster address), with
// no memory ordering: it only tells the MMA issuer that this warp's tensor-memory
// reads are complete (tcgen05.wait::ld and tcgen05.fence::before_thread_sync
// precede it).  A release here would make the warp wait for all of its global
// stores -- the compact outputs and cache rows -- to be acknowledged first.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
                 : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// the shared::cluster address of the same shared-memory location in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank)
{
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

// A tile of the pair's operands into this CTA's shared memory; the transferred
// bytes are counted on `bar`, which may be the leader CTA's barrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t cluster_bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(cluster_bar)
        : "memory");
}

// Bring a box of the tensor into L2 without waiting for it.  Weights read once per
// launch come from DRAM; a stage's load issued after this prefetch finds them in L2
// instead of waiting out a DRAM round trip with the ring's few loads in flight.
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x),
                 "r"(y)
                 : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, groups of 8 rows 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);  // start address
    d |= (uint64_t)1 << 16;                           // leading byte offset (unused here)
    d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

// The 2-SM MMA (32 bytes of K per row: 16 bf16 or 32 E4M3 elements): A and B
// descriptors address the leader's tiles; the peer's halves sit at the same
// shared-memory offsets in the peer CTA.
template <bool FP8>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc)
{
    if (FP8)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(kIdescE4m3), "r"(acc)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(kIdescBf16), "r"(acc)
            : "memory");
}

// The mbarrier at this offset in both CTAs of the pair arrives once every
// tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit_both(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"((unsigned short)3)
        : "memory");
}

// the same, on this CTA's barrier only
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 32 bit, N consecutive columns per thread
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
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

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }



// Where an epilogue thread's accumulator row lives: this CTA's tensor memory.
struct AccSrc {
    uint32_t taddr;       // this warp's lanes at the tile's first column
};

// 32 accumulator columns [col, col + 32) of this thread's row
__device__ __forceinline__ void acc_ld32(const AccSrc &a, int col, uint32_t (&r)[32])
{
    tmem_ld32(a.taddr + (uint32_t)col, r);
    tmem_wait_ld();
}

// ---------------------------------------------------------------------------
// number formats and stores
// ---------------------------------------------------------------------------

// (element 0, element 1) -> a bf16 pair, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// four values -> four E4M3 bytes in element order; RNE, saturating to +-448
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d)
{
    unsigned short lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ void st_v4(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_v2(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

// The dequantised accumulator of output `col`: (acc * hidden scale) * weight
// scale; the accumulator itself when the projection has no scales.
struct RowScale {
    float sx;             // this token's scale
    const float *sw;      // per-output scales, or nullptr
    bool any;
};

__device__ __forceinline__ float dequant(const RowScale &rs, uint32_t acc, int col)
{
    const float a = __uint_as_float(acc);
    if (!rs.any)
        return a;
    const float v = a * rs.sx;
    return rs.sw ? v * __ldg(rs.sw + col) : v;
}

// 8 accumulator words of outputs [col, col + 8) -> the bf16 row values (as bf16
// pairs) and their fp32 values
__device__ __forceinline__ void round_row8(const RowScale &rs, const uint32_t (&acc)[8], int col,
                                           uint32_t (&bits)[4], float (&x)[8])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        bits[j] = pack_bf16x2(dequant(rs, acc[2 * j], col + 2 * j),
                              dequant(rs, acc[2 * j + 1], col + 2 * j + 1));
        x[2 * j] = bf16_lo(bits[j]);
        x[2 * j + 1] = bf16_hi(bits[j]);
    }
}

// ---------------------------------------------------------------------------
// per-token placement (the rule of msa_producer_forward)
// ---------------------------------------------------------------------------

struct Place {
    long long page;
    int off;
    int valid;  // bit c: cache c (k, v, idx_k) takes the token
};

__device__ __forceinline__ Place place_token(const Params &p, long long ls)
{
    Place m;
    m.page = -1;
    m.off = 0;
    m.valid = 0;
    if (ls < 0)
        return m;
    const long long blk = p.page_shift >= 0 ? (ls >> p.page_shift) : ls / p.page_size;
    long long page = blk;
    if (p.page_table)
        page = blk < p.page_table_len ? (long long)__ldg(p.page_table + blk) : -1;
    if (page < 0)
        return m;
    m.page = page;
    m.off = p.page_shift >= 0 ? (int)(ls & (long long)(p.page_size - 1))
                              : (int)(ls - blk * p.page_size);
#pragma unroll
    for (int ci = 0; ci < 3; ++ci)
        if (p.cache[ci].data && page < p.cache[ci].num_pages)
            m.valid |= 1 << ci;
    return m;
}

// ---------------------------------------------------------------------------
// the epilogue: one token row of one 128 x 256 tile
// ---------------------------------------------------------------------------

struct Head {
    int sec;  // 0 Q, 1 K, 2 V, 3 idx-Q, 4 idx-K; -1 past the last head
    int h;    // head index inside its section
};

__device__ __forceinline__ Head head_of(const Params &p, int g)
{
    const int e_k = p.hq, e_v = e_k + p.hkv, e_iq = e_v + p.hkv, e_ik = e_iq + p.hiq;
    Head r;
    if (g >= p.htot) { r.sec = -1; r.h = 0; }
    else if (g < e_k) { r.sec = 0; r.h = g; }
    else if (g < e_v) { r.sec = 1; r.h = g - e_k; }
    else if (g < e_iq) { r.sec = 2; r.h = g - e_v; }
    else if (g < e_ik) { r.sec = 3; r.h = g - e_iq; }
    else { r.sec = 4; r.h = g - e_ik; }
    return r;
}

// Where one head row of one token goes: its first byte, how it is encoded, and the
// reciprocal of its cache scale; computed once per (token, head).
struct Dest {
    uint8_t *row;  // nullptr: nothing is written (padded token, or a cache not taken)
    int fp8;       // 1: E4M3 codes of x * inv; 0: bf16
    float inv;
#ifdef MSA_CHECKED
    const uint8_t *lo, *hi;   // the destination's extent
#endif
};

// the reciprocal of the cache scale of a K, V or index-K head
__device__ __forceinline__ float cache_inv_scale(const Params &p, const Head &hd)
{
    const int ci = hd.sec == 1 ? 0 : hd.sec == 2 ? 1 : 2;
    const int si = p.scale_mode == MSA_SCALE_PER_HEAD
                       ? (ci == 0 ? hd.h : ci == 1 ? p.hkv + hd.h : 2 * p.hkv + hd.h)
                       : ci;
    return __frcp_rn(__ldg(p.scales + si));
}

// inv_pre: that reciprocal when the caller has it already (negative: read it here)
template <int D>
__device__ __forceinline__ Dest make_dest(const Params &p, const Head &hd, int64_t t, bool live,
                                          const Place &pl, float inv_pre = -1.0f)
{
    Dest ds;
    ds.row = nullptr;
    ds.fp8 = 0;
    ds.inv = 1.0f;
    if (!live || hd.sec < 0)
        return ds;
    if (hd.sec == 0 || hd.sec == 3) {
        uint16_t *r = hd.sec == 0 ? p.q_out + ((int64_t)t * p.hq + hd.h) * D
                                  : p.idx_q_out + ((int64_t)t * p.hiq + hd.h) * D;
        ds.row = reinterpret_cast<uint8_t *>(r);
#ifdef MSA_CHECKED
        ds.lo = reinterpret_cast<const uint8_t *>(hd.sec == 0 ? p.q_out : p.idx_q_out);
        ds.hi = p.out_hi[hd.sec == 0 ? 0 : 1];
#endif
        return ds;
    }
    const int ci = hd.sec == 1 ? 0 : hd.sec == 2 ? 1 : 2;
    if (!((pl.valid >> ci) & 1))
        return ds;
    const CacheArgs &cc = p.cache[ci];
    const int64_t e = pl.page * cc.stride_page + (int64_t)hd.h * cc.stride_head +
                      (int64_t)pl.off * cc.stride_token;
#ifdef MSA_CHECKED
    ds.lo = cc.data;
    ds.hi = p.cache_hi[ci];
#endif
    if (cc.fp8) {
        ds.row = cc.data + e;
        ds.fp8 = 1;
        ds.inv = inv_pre >= 0.0f ? inv_pre : cache_inv_scale(p, hd);
    } else {
        ds.row = cc.data + 2 * e;
    }
    return ds;
}

// Stores 8 finished values of dims [d0, d0 + 8) of a head row.
__device__ __forceinline__ void emit8(const Dest &ds, int d0, const float (&y)[8])
{
    if (!ds.row)
        return;
    if (ds.fp8) {
        const float inv = ds.inv;
        MSA_GUARD(ds.row + d0, 8, ds.lo, ds.hi)
        st_v2(ds.row + d0, pack_e4m3x4(y[0] * inv, y[1] * inv, y[2] * inv, y[3] * inv),
              pack_e4m3x4(y[4] * inv, y[5] * inv, y[6] * inv, y[7] * inv));
    } else {
        MSA_GUARD(ds.row + 2 * d0, 16, ds.lo, ds.hi)
        st_v4(ds.row + 2 * d0, pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]),
              pack_bf16x2(y[4], y[5]), pack_bf16x2(y[6], y[7]));
    }
}

// norm weight element i of a tensor (unit weight when absent)
__device__ __forceinline__ float norm_weight(const uint16_t *w, int i)
{
    return w ? __uint_as_float((uint32_t)__ldg(w + i) << 16) : 1.0f;
}

// which of the four norm weights a section takes (Q, K, idx-Q, idx-K)
__device__ __forceinline__ int norm_index(int sec)
{
    return sec == 0 ? 0 : sec == 1 ? 1 : sec == 3 ? 2 : 3;
}

// Sine and cosine of a RoPE angle.  Below 2^16 the angle is reduced to [-pi, pi]
// by k = rint(a / 2pi), r = a - k * 2pi, with 2pi split into three floats whose
// first, 6.28125, has 8 significant bits so that k * 6.28125 is exact (Cody and
// Waite's additive range reduction), and the hardware approximations take r
// (absolute error about 2^-21 on [-pi, pi]); larger angles use sincosf, called
// out of line: the epilogue unrolls this at every rotated pair of a head, and
// sincosf's full-range reduction inlined at each of those sites multiplied the
// epilogue's code several times over.  The epilogue runs once per tile, so its
// instructions stream through the instruction cache: at small batches, where
// the epilogue is not hidden behind the next tile's main loop, the inlined copies
// (never executed) tripled its time.
__device__ __noinline__ float2 rope_sincos_wide(float a)
{
    float s, c;
    sincosf(a, &s, &c);
    return make_float2(s, c);
}

__device__ __forceinline__ void rope_sincos(float a, float *s, float *c)
{
    if (fabsf(a) < 65536.0f) {
        const float k = rintf(a * 0.15915494f);
        float r = fmaf(-k, 6.28125f, a);
        r = fmaf(-k, 1.9353071693331003e-3f, r);
        r = fmaf(-k, 1.0253131677018246e-11f, r);
        __sincosf(r, s, c);
    } else {
        const float2 v = rope_sincos_wide(a);
        *s = v.x;
        *c = v.y;
    }
}

// One head of one token row, for NeoX RoPE over the first ROT of D dims (ROT = D,
// D/2 or 0).  The accumulator is read from tensor memory once and the bf16 row
// is kept in registers; the head's norm weights and per-output scales are held by
// the lanes of the warp (lane l: dims l, l + 32, ...) and shuffled to every lane.
template <int D, int ROT>
__device__ __forceinline__ void head_fast(const Params &p, const Head &hd, const AccSrc &src,
                                          int tcol, int col,
                                          int64_t t, bool live, const Place &pl, int pos,
                                          const RowScale &rs, int lane)
{
    constexpr int NW = D / 32;
    const bool normed = hd.sec != 2;
    const Dest ds = make_dest<D>(p, hd, t, live, pl);
    const uint16_t *w = normed ? p.norm_w[norm_index(hd.sec)] : nullptr;
    float wr[NW], swr[NW];
#pragma unroll
    for (int m = 0; m < NW; ++m) {
        wr[m] = norm_weight(w, 32 * m + lane);
        swr[m] = rs.sw ? __ldg(rs.sw + col + 32 * m + lane) : 1.0f;
    }

    // pass 1: the bf16 row (dequantised accumulator, rounded) and its sum of squares
    uint32_t row[D / 2];
    float ss = 0.0f;
#pragma unroll
    for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        acc_ld32(src, tcol + c, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            float a = __uint_as_float(r[2 * j]), b = __uint_as_float(r[2 * j + 1]);
            if (rs.any) {
                a = (a * rs.sx) * __shfl_sync(0xffffffffu, swr[c / 32], 2 * j);
                b = (b * rs.sx) * __shfl_sync(0xffffffffu, swr[c / 32], 2 * j + 1);
            }
            row[c / 2 + j] = pack_bf16x2(a, b);
            const float ra = bf16_lo(row[c / 2 + j]), rb = bf16_hi(row[c / 2 + j]);
            ss = fmaf(ra, ra, ss);
            ss = fmaf(rb, rb, ss);
        }
    }
    if (p.rows_out && live) {
        uint16_t *dst = p.rows_out + (int64_t)t * p.rows_out_stride + col;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            MSA_GUARD(dst + 8 * i, 16, p.rows_out, p.rows_hi)
            st_v4(dst + 8 * i, row[4 * i], row[4 * i + 1], row[4 * i + 2], row[4 * i + 3]);
    }
    auto elt = [&](int i) { return (i & 1) ? bf16_hi(row[i >> 1]) : bf16_lo(row[i >> 1]); };
    if (!normed) {  // V: the row itself, into its cache
#pragma unroll
        for (int c = 0; c < D; c += 8) {
            float y[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                y[j] = elt(c + j);
            emit8(ds, c, y);
        }
        return;
    }

    // pass 2: norm, RoPE, store
    const float rn = rsqrtf(fmaf(ss, 1.0f / (float)D, p.rms_eps));
    auto wgt = [&](int i) { return __shfl_sync(0xffffffffu, wr[i >> 5], i & 31); };
    constexpr int H = ROT / 2;
#pragma unroll
    for (int k0 = 0; k0 < H; k0 += 8) {
        float yu[8], yv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float sn, cs;
            rope_sincos((float)pos * p.inv_freq[k0 + j], &sn, &cs);
            const float a = (elt(k0 + j) * rn) * wgt(k0 + j);
            const float b = (elt(k0 + H + j) * rn) * wgt(k0 + H + j);
            yu[j] = fmaf(-b, sn, a * cs);
            yv[j] = fmaf(a, sn, b * cs);
        }
        emit8(ds, k0, yu);
        emit8(ds, k0 + H, yv);
    }
#pragma unroll
    for (int c = ROT; c < D; c += 8) {
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            y[j] = (elt(c + j) * rn) * wgt(c + j);
        emit8(ds, c, y);
    }
}

// taddr: tensor-memory address of this warp's lanes at the tile's first column.
// The warp runs the producer on the tile's heads hh with hh % 2 == hgroup (the
// other epilogue warp of the same tensor-memory lanes takes the rest).
template <int D>
__device__ __forceinline__ void epilogue_tile(const Params &p, const AccSrc &src, int n_tile,
                                              int64_t t, bool live, int hgroup, int lane)
{
    // a warp whose 32 rows are all past the last token has nothing to read or write
    // (a partial last token tile; at decode sizes half the tile)
    if (!__any_sync(0xffffffffu, live))
        return;
    const uint32_t taddr = src.taddr;
    constexpr int HPT = kBN / D;  // heads per tile
    const int g0 = n_tile * HPT;

    // token metadata
    int pos = 0;
    Place pl;
    pl.page = -1;
    pl.off = 0;
    pl.valid = 0;
    if (live) {
        pos = __ldg(p.positions + t);
        pl = place_token(p, __ldg(p.slots + t));
    }
    RowScale rs;
    rs.sw = p.weight_scales;
    rs.sx = (p.hidden_scales && live) ? __ldg(p.hidden_scales + t) : 1.0f;
    rs.any = p.hidden_scales || p.weight_scales;
    const int col0 = n_tile * kBN;  // projection output of the tile's first column

    const int rd = p.rotary_dim;
    if (p.rope_style == MSA_ROPE_NEOX && (rd == D || rd == D / 2 || rd == 0)) {
#pragma unroll
        for (int hh = hgroup; hh < HPT; hh += 2) {
            const Head hd = head_of(p, g0 + hh);
            if (hd.sec < 0)
                continue;
            const int col = col0 + hh * D;
            if (rd == D)
                head_fast<D, D>(p, hd, src, hh * D, col, t, live, pl, pos, rs, lane);
            else if (rd == D / 2)
                head_fast<D, D / 2>(p, hd, src, hh * D, col, t, live, pl, pos, rs, lane);
            else
                head_fast<D, 0>(p, hd, src, hh * D, col, t, live, pl, pos, rs, lane);
        }
        return;
    }

    // any other RoPE: the accumulator is read twice (norm factor, then values);
    // reached only without a split over K (the host keeps those on the 2-SM kernel)

    // pass 1: bf16 row values, optional row store, and each head's norm factor
    float rn[HPT];
#pragma unroll
    for (int hh = 0; hh < HPT; ++hh) {
        rn[hh] = 0.0f;
        if (g0 + hh >= p.htot || (hh & 1) != hgroup)
            continue;
        float ss = 0.0f;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
            uint32_t r[32];
            tmem_ld32(taddr + (uint32_t)(hh * D + c), r);
            tmem_wait_ld();
            uint32_t bits[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int col = col0 + hh * D + c + 2 * j;
                bits[j] = pack_bf16x2(dequant(rs, r[2 * j], col), dequant(rs, r[2 * j + 1], col + 1));
                const float a = bf16_lo(bits[j]), b = bf16_hi(bits[j]);
                ss = fmaf(a, a, ss);
                ss = fmaf(b, b, ss);
            }
            if (p.rows_out && live) {
                uint16_t *dst = p.rows_out + (int64_t)t * p.rows_out_stride +
                                (int64_t)(g0 + hh) * D + c;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    MSA_GUARD(dst + 8 * j, 16, p.rows_out, p.rows_hi)
                    st_v4(dst + 8 * j, bits[4 * j], bits[4 * j + 1], bits[4 * j + 2], bits[4 * j + 3]);
            }
        }
        rn[hh] = rsqrtf(fmaf(ss, 1.0f / (float)D, p.rms_eps));
    }

    Head hd[HPT];
    Dest ds[HPT];
    bool normed_any = false;
#pragma unroll
    for (int hh = 0; hh < HPT; ++hh) {
        hd[hh] = head_of(p, g0 + hh);
        if ((hh & 1) != hgroup)
            hd[hh].sec = -1;  // the other warp's head
        ds[hh] = make_dest<D>(p, hd[hh], t, live, pl);
        normed_any |= hd[hh].sec >= 0 && hd[hh].sec != 2;
    }

    // pass 2a: normed heads (Q, K, idx-Q, idx-K)
    if (normed_any) {
        if (p.rope_style == MSA_ROPE_NEOX) {
            const int half = rd / 2;
            // rotated pairs (k, k + rd/2), 8 frequencies at a time
            for (int k0 = 0; k0 < half; k0 += 8) {
                float cs[8], sn[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    sincosf((float)pos * p.inv_freq[k0 + j], &sn[j], &cs[j]);
#pragma unroll
                for (int hh = 0; hh < HPT; ++hh) {
                    if (hd[hh].sec < 0 || hd[hh].sec == 2)
                        continue;
                    const uint16_t *w = p.norm_w[hd[hh].sec == 0 ? 0 : hd[hh].sec == 1 ? 1 : hd[hh].sec == 3 ? 2 : 3];
                    uint32_t ru[8], rv[8], bu[4], bv[4];
                    float u[8], v[8];
                    tmem_ld8(taddr + (uint32_t)(hh * D + k0), ru);
                    tmem_ld8(taddr + (uint32_t)(hh * D + k0 + half), rv);
                    tmem_wait_ld();
                    round_row8(rs, ru, col0 + hh * D + k0, bu, u);
                    round_row8(rs, rv, col0 + hh * D + k0 + half, bv, v);
                    float yu[8], yv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float a = (u[j] * rn[hh]) * norm_weight(w, k0 + j);
                        const float b = (v[j] * rn[hh]) * norm_weight(w, k0 + half + j);
                        yu[j] = fmaf(-b, sn[j], a * cs[j]);
                        yv[j] = fmaf(a, sn[j], b * cs[j]);
                    }
                    emit8(ds[hh], k0, yu);
                    emit8(ds[hh], k0 + half, yv);
                }
            }
            // pass-through dims [rd, D)
            for (int c = rd; c < D; c += 8) {
#pragma unroll
                for (int hh = 0; hh < HPT; ++hh) {
                    if (hd[hh].sec < 0 || hd[hh].sec == 2)
                        continue;
                    const uint16_t *w = p.norm_w[hd[hh].sec == 0 ? 0 : hd[hh].sec == 1 ? 1 : hd[hh].sec == 3 ? 2 : 3];
                    uint32_t ru[8], bu[4];
                    float u[8], y[8];
                    tmem_ld8(taddr + (uint32_t)(hh * D + c), ru);
                    tmem_wait_ld();
                    round_row8(rs, ru, col0 + hh * D + c, bu, u);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        y[j] = (u[j] * rn[hh]) * norm_weight(w, c + j);
                    emit8(ds[hh], c, y);
                }
            }
        } else {
            // GPT-J: pairs (2k, 2k + 1); a chunk of 8 dims is rotated whole or not at all
            for (int c = 0; c < D; c += 8) {
                const bool rot = c < rd;
                float cs[4], sn[4];
                if (rot) {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sincosf((float)pos * p.inv_freq[c / 2 + j], &sn[j], &cs[j]);
                }
#pragma unroll
                for (int hh = 0; hh < HPT; ++hh) {
                    if (hd[hh].sec < 0 || hd[hh].sec == 2)
                        continue;
                    const uint16_t *w = p.norm_w[hd[hh].sec == 0 ? 0 : hd[hh].sec == 1 ? 1 : hd[hh].sec == 3 ? 2 : 3];
                    uint32_t ru[8], bu[4];
                    float u[8], y[8];
                    tmem_ld8(taddr + (uint32_t)(hh * D + c), ru);
                    tmem_wait_ld();
                    round_row8(rs, ru, col0 + hh * D + c, bu, u);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        y[j] = (u[j] * rn[hh]) * norm_weight(w, c + j);
                    if (rot) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float a = y[2 * j], b = y[2 * j + 1];
                            y[2 * j] = fmaf(-b, sn[j], a * cs[j]);
                            y[2 * j + 1] = fmaf(a, sn[j], b * cs[j]);
                        }
                    }
                    emit8(ds[hh], c, y);
                }
            }
        }
    }

    // pass 2b: V heads (no norm, no RoPE)
#pragma unroll
    for (int hh = 0; hh < HPT; ++hh) {
        if (hd[hh].sec != 2)
            continue;
        for (int c = 0; c < D; c += 8) {
            uint32_t ru[8], bu[4];
            float u[8];
            tmem_ld8(taddr + (uint32_t)(hh * D + c), ru);
            tmem_wait_ld();
            round_row8(rs, ru, col0 + hh * D + c, bu, u);
            emit8(ds[hh], c, u);
        }
    }
}

__device__ __forceinline__ void tile_coords(const Params &p, int64_t tile, int &m, int &n)
{
    const int64_t per_group = (int64_t)p.n_group * p.m_tiles;
    const int64_t g = tile / per_group;
    const int64_t r = tile - g * per_group;
    const int n0 = (int)g * p.n_group;
    const int gn = min(p.n_group, p.n_tiles - n0);
    m = (int)(r / gn);
    n = n0 + (int)(r % gn);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
msa_projection_kernel(const __grid_constant__ CUtensorMap tmap_x,
                      const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kStages];   // leader: both CTAs' copies landed
    __shared__ __align__(8) uint64_t bar_empty[kStages];  // both: the MMAs have read the stage
    __shared__ __align__(8) uint64_t bar_tfull[2];        // both: accumulator b is complete
    __shared__ __align__(8) uint64_t bar_tempty[2];       // leader: both epilogues drained b
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t s_tmem;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;  // the swizzle pattern needs 1024-byte alignment

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bar_full[s]), 1);
            mbar_init(smem_u32(&bar_empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bar_tfull[b]), 1);
            mbar_init(smem_u32(&bar_tempty[b]), 2 * kEpilogueWarps);  // each epilogue warp of the pair
        }
        mbar_init(smem_u32(&bar_drain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_x) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmap_w) : "memory");
    }
    if (warp == 1) {
        // one warp of each CTA of the pair: the same columns in both tensor memories
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();  // barriers initialised and tensor memory allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    constexpr int kBKElems = FP8 ? kBKBytes : kBKBytes / 2;  // K elements per stage
    const int64_t num_tiles = (int64_t)p.m_tiles * p.n_tiles;
    const int64_t cluster_id = blockIdx.x / 2;
    const int64_t num_clusters = gridDim.x / 2;
    bool ok = true;

    if (warp == 0) {
        // ---------------- TMA producer (both CTAs) ----------------
#ifdef MSA_STARVE
        if (false) {   // the starved test build: no copy is ever issued
#else
        if (lane == 0) {
#endif
            uint32_t stage = 0, phase = 0;
            for (int64_t tile = cluster_id; tile < num_tiles && ok; tile += num_clusters) {
                int m, n;
                tile_coords(p, tile, m, n);
                const int row_x = m * kPairM + (int)rank * kBM;
                const int row_w = n * kBN + (int)rank * kHalfN;
                const int pf = row_w < p.htot * D ? p.prefetch : 0;  // rows past W: nothing to fetch
                for (int kb = 0; kb < pf && kb < p.num_k_blocks; ++kb)
                    tma_prefetch_l2(&tmap_w, kb * kBKElems, row_w);
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (pf && kb + pf < p.num_k_blocks)
                        tma_prefetch_l2(&tmap_w, (kb + pf) * kBKElems, row_w);
                    if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_u32(&bar_full[stage]);
                    if (rank == 0)  // the leader expects the bytes of both CTAs
                        mbar_expect_tx(full, 2 * kStageBytes);
                    const uint32_t full_leader = map_to_rank(full, 0);
                    const uint32_t a = ring + stage * kStageBytes;
                    tma_load_2d(a, &tmap_x, kb * kBKElems, row_x, full_leader);
                    tma_load_2d(a + kTileABytes, &tmap_w, kb * kBKElems, row_w, full_leader);
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                // let the copies in flight land before the CTA may exit
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------- MMA issuer (leader CTA) ----------------
        if (lane == 0 && rank == 0) {
            uint32_t stage = 0, phase = 0, acc_i = 0;
            for (int64_t tile = cluster_id; tile < num_tiles && ok; tile += num_clusters, ++acc_i) {
                const uint32_t b = acc_i & 1, use_par = (acc_i >> 1) & 1;
                if (!mbar_wait(smem_u32(&bar_tempty[b]), use_par ^ 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + b * kBN;
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!mbar_wait(smem_u32(&bar_full[stage]), phase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = ring + stage * kStageBytes;
                    const uint32_t bb = a + kTileABytes;
#pragma unroll
                    for (int k = 0; k < kBKBytes / 32; ++k)
                        tc_mma<FP8>(d_tmem, sw128_desc(a + 32u * k), sw128_desc(bb + 32u * k),
                                    (kb | k) != 0);
                    tc_commit_both(smem_u32(&bar_empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok)
                    break;
                tc_commit_both(smem_u32(&bar_tfull[b]));
            }
            // every MMA of the pair is complete before tensor memory is released
            tc_commit(smem_u32(&bar_drain));
            if (!mbar_wait(smem_u32(&bar_drain), 0))
                ok = false;
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (both CTAs) ----------------
        const int quarter = warp & 3;  // the tensor-memory lanes this warp may read
        const int hgroup = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        uint32_t acc_i = 0;
        for (int64_t tile = cluster_id; tile < num_tiles; tile += num_clusters, ++acc_i) {
            int m, n;
            tile_coords(p, tile, m, n);
            const uint32_t b = acc_i & 1, use_par = (acc_i >> 1) & 1;
            const bool got = mbar_wait(smem_u32(&bar_tfull[b]), use_par);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int64_t t = (int64_t)m * kPairM + (int64_t)rank * kBM + row;
            AccSrc src;
            src.taddr = tmem + lane_base + b * kBN;
            epilogue_tile<D>(p, src, n, t, t < p.num_tokens, hgroup, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0)  // this warp is done reading accumulator b
                mbar_arrive_remote(map_to_rank(smem_u32(&bar_tempty[b]), 0));
        }
    }

    if (!ok && p.status)
        atomicOr(p.status, MSA_STATUS_WAIT_TIMEOUT);
    tc_fence_before();
    cluster_sync();  // no MMA, copy or tensor-memory read of the pair is still running
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// small batches: the K dimension split over a cluster
// ---------------------------------------------------------------------------
// With a single 128-token tile (num_tokens <= 128) the 2-SM kernel keeps at most
// one cluster per 256-wide output tile busy, each walking all of K.  Here a
// cluster of S CTAs takes one output tile and CTA s of it a contiguous S-th of the
// K blocks, accumulating 128 tokens x 256 outputs in its own tensor memory with the
// one-SM MMA (tcgen05.mma.cta_group::1, M 128, N 256).  Every CTA then writes its
// partial sum into its shared memory (the ring is free by then), and the
// producer epilogue of the tile is spread over the epilogue warps of all S CTAs,
// each (token, head) row taken by a group of lanes that add the S partial sums in
// rank order over distributed shared memory (splitk_epilogue).  Used for NeoX RoPE
// over D, D/2 or no dims; other layouts take the 2-SM kernel.

constexpr int kSplitStages = 4;
constexpr uint32_t kSplitStageBytes = kTileABytes + 2 * kTileBBytes;  // 128 tokens + 256 weight rows
constexpr int kSplitDynSmem = kSplitStages * kSplitStageBytes + 1024;
// an exported partial sum: 128 rows of 256 fp32 columns, rows 16 bytes further apart
// than their length so that both the export (a thread per row) and the epilogue's
// reads (lanes along a row) hit distinct banks
constexpr uint32_t kPartRowBytes = kBN * 4u + 16u;
static_assert(kSplitStages * kSplitStageBytes >= 128u * kPartRowBytes, "partial sums fit the ring");
constexpr uint32_t kIdescShape1 = ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
constexpr uint32_t kSplitTmemCols = kBN;   // the accumulator

template <bool FP8>
__device__ __forceinline__ void tc_mma1(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc)
{
    if (FP8)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"((1u << 4) | kIdescShape1), "r"(acc)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"((1u << 4) | (1u << 7) | (1u << 10) | kIdescShape1), "r"(acc)
            : "memory");
}

__device__ __forceinline__ void tc_commit1(uint32_t bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_own(uint32_t dst, const CUtensorMap *map, int x, int y,
                                             uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// The epilogue of a tile whose K dimension was split over the cluster's S CTAs,
// spread over every epilogue warp of the cluster.  Item i = (token t, head hh of
// the tile) goes to a group of D / 8 lanes; lane u of the group holds dims
// [8u, 8u + 8) of the head row.  Its accumulator is the sum, in rank order, of the
// partial sums the S CTAs exported to their shared memory; the sum of squares of
// the rounded bf16 row is a shuffle reduction over the group, and the NeoX partner
// of a rotated dim (k and k + rd/2) sits rd/16 lanes away.  What the items read
// besides the partial sums was staged in this CTA's shared memory during the main
// loop: per token its position, placement and hidden scale; per tile column its
// norm weight and per-output scale; per head of the tile its cache scale's
// reciprocal.
struct SplitStage {
    int pos[kBM];
    Place place[kBM];
    float sx[kBM];
    float nw[kBN];     // norm weight of the column's head (1: V, or no weight)
    float sw[kBN];     // per-output scale (1: none, or past the outputs)
    float dinv[8];     // per head of the tile (negative: not an fp8 cache head)
    float freq[kMaxRotaryHalf];   // RoPE frequencies: the lanes of a warp index them apart, which
                       // the kernel-parameter bank would serve one address at a time
};

template <int D>
__device__ __forceinline__ void splitk_epilogue(const Params &p, uint32_t part, int S, int n_tile,
                                                const SplitStage &st, int worker, int nworkers, int lane)
{
    constexpr int LPI = D / 8;          // lanes per item
    constexpr int IPW = 32 / LPI;       // items per warp and pass
    constexpr int HPT = kBN / D;        // heads per tile
    const int c = 8 * (lane % LPI);     // this lane's first dim of the head row
    const int g0 = n_tile * HPT;
    const int col0 = n_tile * kBN;
    const int total = p.num_tokens * HPT;
    const int rd = p.rotary_dim, half = rd / 2;
    const bool any_scale = p.hidden_scales || p.weight_scales;
    // every lane runs every pass (the shuffles need the whole warp); a lane past the
    // last item computes on row 0 and stores nothing
    const int stride = nworkers * IPW;
    for (int base = worker * IPW; base < total; base += stride) {
        const int i = base + lane / LPI;
        const bool on = i < total;
        const int t = on ? i / HPT : 0, hh = on ? i % HPT : 0;
        Head hd = head_of(p, g0 + hh);
        if (!on)
            hd.sec = -1;
        const int tc = hh * D + c, col = col0 + tc;
        const bool normed = hd.sec >= 0 && hd.sec != 2;
        // the accumulator: the partial sums in rank order, four ranks' loads in flight
        float acc[8];
        const uint32_t off = (uint32_t)t * kPartRowBytes + (uint32_t)tc * 4u;
        for (int r0 = 0; r0 < S; r0 += 4) {
            float4 v[4][2];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (r0 + k < S) {
                    const uint32_t a = map_to_rank(part + off, (uint32_t)(r0 + k));
                    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(v[k][0].x), "=f"(v[k][0].y), "=f"(v[k][0].z), "=f"(v[k][0].w) : "r"(a));
                    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                                 : "=f"(v[k][1].x), "=f"(v[k][1].y), "=f"(v[k][1].z), "=f"(v[k][1].w) : "r"(a + 16u));
                }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (r0 + k < S) {
                    const float x[8] = {v[k][0].x, v[k][0].y, v[k][0].z, v[k][0].w,
                                        v[k][1].x, v[k][1].y, v[k][1].z, v[k][1].w};
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[j] = (r0 + k == 0) ? x[j] : acc[j] + x[j];
                }
            }
        }

        // the bf16 row (dequantised accumulator, rounded) and its sum of squares
        const float sx = st.sx[t];
        uint32_t bits[4];
        float e[8];
        float ss = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            float a = acc[j], b = acc[j + 1];
            if (any_scale) {
                a = (a * sx) * st.sw[tc + j];
                b = (b * sx) * st.sw[tc + j + 1];
            }
            bits[j / 2] = pack_bf16x2(a, b);
            e[j] = bf16_lo(bits[j / 2]);
            e[j + 1] = bf16_hi(bits[j / 2]);
            ss = fmaf(e[j], e[j], ss);
            ss = fmaf(e[j + 1], e[j + 1], ss);
        }
        if (p.rows_out && hd.sec >= 0) {
            uint16_t *dst = p.rows_out + (int64_t)t * p.rows_out_stride + col;
            MSA_GUARD(dst, 16, p.rows_out, p.rows_hi)
            st_v4(dst, bits[0], bits[1], bits[2], bits[3]);
        }
#pragma unroll
        for (int m = 1; m < LPI; m <<= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, m);
        const float rn = rsqrtf(fmaf(ss, 1.0f / (float)D, p.rms_eps));

        // norm (Q, K, idx-Q, idx-K), then NeoX RoPE over the first rd dims
        float y[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            y[j] = normed ? (e[j] * rn) * st.nw[tc + j] : e[j];
        if (rd > 0) {
            float px[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                px[j] = __shfl_xor_sync(0xffffffffu, y[j], half / 8);
            if (normed && c < rd) {
                const bool first = c < half;
                const int kb = first ? c : c - half;
                const int pos = st.pos[t];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    float sn, cs;
                    rope_sincos((float)pos * st.freq[kb + j], &sn, &cs);
                    y[j] = first ? fmaf(-px[j], sn, y[j] * cs) : fmaf(px[j], sn, y[j] * cs);
                }
            }
        }
        emit8(make_dest<D>(p, hd, t, on, st.place[t], st.dinv[hh]), c, y);
    }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
msa_projection_splitk_kernel(const __grid_constant__ CUtensorMap tmap_x,
                             const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ Params p)
{
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bar_full[kSplitStages];
    __shared__ __align__(8) uint64_t bar_empty[kSplitStages];
    __shared__ __align__(8) uint64_t bar_tfull;
    __shared__ __align__(8) uint64_t bar_drain;
    __shared__ uint32_t s_tmem;
    __shared__ uint32_t s_fail;   // a wait of this CTA ran out: its partial sum is not valid
    __shared__ SplitStage s_st;   // what the epilogue reads besides the partial sums

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int S = p.split;
    const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int n_tile = blockIdx.x / S;
    const int kb0 = (int)((int64_t)p.num_k_blocks * rank / S);
    const int kb1 = (int)((int64_t)p.num_k_blocks * (rank + 1) / S);
    constexpr int kBKElems = FP8 ? kBKBytes : kBKBytes / 2;

    if (threadIdx.x == 0) {
        for (int st = 0; st < kSplitStages; ++st) {
            mbar_init(smem_u32(&bar_full[st]), 1);
            mbar_init(smem_u32(&bar_empty[st]), 1);
        }
        mbar_init(smem_u32(&bar_tfull), 1);
        mbar_init(smem_u32(&bar_drain), 1);
        s_fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(kSplitTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    bool ok = true;

    if (warp == 0) {
#ifdef MSA_STARVE
        if (false) {   // the starved test build: no copy is ever issued
#else
        if (lane == 0) {   // TMA: this CTA's K blocks of the hidden tile and the weight tile
#endif
            uint32_t stage = 0, phase = 0;
            for (int kb = kb0; kb < kb0 + p.prefetch && kb < kb1; ++kb)
                tma_prefetch_l2(&tmap_w, kb * kBKElems, n_tile * kBN);
            for (int kb = kb0; kb < kb1; ++kb) {
                if (p.prefetch && kb + p.prefetch < kb1)
                    tma_prefetch_l2(&tmap_w, (kb + p.prefetch) * kBKElems, n_tile * kBN);
                if (!mbar_wait(smem_u32(&bar_empty[stage]), phase ^ 1)) {
                    ok = false;
                    break;
                }
                const uint32_t full = smem_u32(&bar_full[stage]);
                const uint32_t a = ring + stage * kSplitStageBytes;
                mbar_expect_tx(full, kSplitStageBytes);
                tma_load_own(a, &tmap_x, kb * kBKElems, 0, full);
                tma_load_own(a + kTileABytes, &tmap_w, kb * kBKElems, n_tile * kBN, full);
                if (++stage == kSplitStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) {   // let the copies in flight land before the CTA may exit
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 200000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {   // MMA: the partial sum over this CTA's K blocks
            uint32_t stage = 0, phase = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&bar_full[stage]), phase)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t a = ring + stage * kSplitStageBytes;
                const uint32_t bb = a + kTileABytes;
#pragma unroll
                for (int k = 0; k < kBKBytes / 32; ++k)
                    tc_mma1<FP8>(tmem, sw128_desc(a + 32u * k), sw128_desc(bb + 32u * k),
                                 (kb > kb0) || (k != 0));
                tc_commit1(smem_u32(&bar_empty[stage]));
                if (++stage == kSplitStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            tc_commit1(smem_u32(&bar_tfull));
            tc_commit1(smem_u32(&bar_drain));
            if (!mbar_wait(smem_u32(&bar_drain), 0))
                ok = false;
        }
        __syncwarp();
    } else {
        // Every CTA exports its partial sum into the ring (free once the accumulator
        // is complete), as [row][256 columns] fp32 rows kPartRowBytes apart.  Before
        // that, while the main loop runs, the epilogue warps stage what this CTA's
        // share of the epilogue reads: one warp per lane quarter the metadata of its
        // 32 tokens, the other four the tile's per-column and per-head values.
        const int quarter = warp & 3, hgroup = (warp - 2) >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        if (hgroup == 0) {
            Place pl;
            pl.page = -1;
            pl.off = 0;
            pl.valid = 0;
            int pos = 0;
            float sx = 1.0f;
            if (row < p.num_tokens) {
                pos = __ldg(p.positions + row);
                pl = place_token(p, __ldg(p.slots + row));
                if (p.hidden_scales)
                    sx = __ldg(p.hidden_scales + row);
            }
            s_st.pos[row] = pos;
            s_st.place[row] = pl;
            s_st.sx[row] = sx;
        } else {
            constexpr int HPT = kBN / D;
            for (int tc = row; tc < kBN; tc += kBM) {
                const int hh = tc / D;
                const Head hd = head_of(p, n_tile * HPT + hh);
                const bool normed = hd.sec >= 0 && hd.sec != 2;
                s_st.nw[tc] = normed ? norm_weight(p.norm_w[norm_index(hd.sec)], tc % D) : 1.0f;
                s_st.sw[tc] = (p.weight_scales && hd.sec >= 0) ? __ldg(p.weight_scales + n_tile * kBN + tc) : 1.0f;
            }
            if (row < p.rotary_dim / 2)
                s_st.freq[row] = p.inv_freq[row];
            if (row < HPT) {
                const Head hd = head_of(p, n_tile * HPT + row);
                const int ci = hd.sec == 1 ? 0 : hd.sec == 2 ? 1 : hd.sec == 4 ? 2 : -1;
                s_st.dinv[row] = (ci >= 0 && p.cache[ci].data && p.cache[ci].fp8) ? cache_inv_scale(p, hd) : -1.0f;
            }
        }
        const bool got = mbar_wait(smem_u32(&bar_tfull), 0);
        if (!__all_sync(0xffffffffu, got))
            ok = false;
        tc_fence_after();
        if (ok && __any_sync(0xffffffffu, row < p.num_tokens)) {
            // (rows past the last token are never read back)
#pragma unroll
            for (int c0 = hgroup * (kBN / 2); c0 < (hgroup + 1) * (kBN / 2); c0 += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + lane_base + (uint32_t)c0, r);
                tmem_wait_ld();
                const uint32_t dst = ring + (uint32_t)row * kPartRowBytes + (uint32_t)c0 * 4u;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + 16u * (uint32_t)j),
                                 "r"(r[4 * j]), "r"(r[4 * j + 1]), "r"(r[4 * j + 2]), "r"(r[4 * j + 3])
                                 : "memory");
            }
        }
    }
    // A wait that ran out anywhere in the cluster (a copy, an MMA or the accumulator
    // that never completed) leaves some partial sum invalid -- the MMA thread still
    // commits the accumulator barrier after a timeout, so the epilogue warps cannot
    // see it from their own wait -- and then no CTA may run the epilogue: each CTA
    // flags its failure before the cluster barrier, and CTA 0 reads every flag.
    if (!ok)
        *(volatile uint32_t *)&s_fail = 1u;
    tc_fence_before();
    cluster_sync();   // every CTA's partial sums (and failure flags) are in place
    if (warp >= 2) {
        // every epilogue warp reads every CTA's flag (the loads issued together), so
        // the cluster agrees, and takes a share of the epilogue
        uint32_t fails = ok ? 0u : 1u;
        for (int r = 0; r < S; ++r) {
            uint32_t f;
            asm volatile("ld.shared::cluster.u32 %0, [%1];"
                         : "=r"(f)
                         : "r"(map_to_rank(smem_u32(&s_fail), (uint32_t)r))
                         : "memory");
            fails |= f;
        }
        if (__all_sync(0xffffffffu, fails == 0u))
            splitk_epilogue<D>(p, ring, S, n_tile, s_st, (warp - 2) * S + (int)rank, 8 * S, lane);
    }
    if (!ok && p.status)
        atomicOr(p.status, MSA_STATUS_WAIT_TIMEOUT);
    tc_fence_before();
    cluster_sync();   // no CTA reads another's partial sums any more
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kSplitTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

// ---------------------------------------------------------------------------
// build units
// ---------------------------------------------------------------------------
// The eight kernel instantiations below take minutes to compile in one unit, so
// the build may compile this file several times with MSA_PROJ_UNIT set: unit 0
// holds the host code alone, unit k = 1..8 the k-th kernel alone (returned by
// msa_internal_projection_kernel_<k>), and the units compile in parallel.
// Without MSA_PROJ_UNIT everything is in one unit (the checked build, whose
// device-side violation counter must live in one module).
#if defined(MSA_PROJ_UNIT) && defined(MSA_CHECKED)
#error "the checked build compiles the projection as one unit"
#endif
#if !defined(MSA_PROJ_UNIT)
#define MSA_PROJ_HOST 1
#elif MSA_PROJ_UNIT == 0
#define MSA_PROJ_HOST 1
#else
#define MSA_PROJ_HOST 0
#endif

#if MSA_PROJ_HOST
#if defined(MSA_PROJ_UNIT)
}  // namespace
const void *msa_internal_projection_kernel_1();
const void *msa_internal_projection_kernel_2();
const void *msa_internal_projection_kernel_3();
const void *msa_internal_projection_kernel_4();
const void *msa_internal_projection_kernel_5();
const void *msa_internal_projection_kernel_6();
const void *msa_internal_projection_kernel_7();
const void *msa_internal_projection_kernel_8();
namespace {
#endif

// Host address of a kernel: split over K or not; variant v = (D == 128) + 2 * FP8.
const void *projection_kernel(bool splitk, int v)
{
#if defined(MSA_PROJ_UNIT)
    static const void *(*const get[8])() = {
        msa_internal_projection_kernel_1, msa_internal_projection_kernel_2,
        msa_internal_projection_kernel_3, msa_internal_projection_kernel_4,
        msa_internal_projection_kernel_5, msa_internal_projection_kernel_6,
        msa_internal_projection_kernel_7, msa_internal_projection_kernel_8};
    return get[(splitk ? 4 : 0) + v]();
#else
    const void *k[8] = {reinterpret_cast<const void *>(&msa_projection_kernel<64, false>),
                        reinterpret_cast<const void *>(&msa_projection_kernel<128, false>),
                        reinterpret_cast<const void *>(&msa_projection_kernel<64, true>),
                        reinterpret_cast<const void *>(&msa_projection_kernel<128, true>),
                        reinterpret_cast<const void *>(&msa_projection_splitk_kernel<64, false>),
                        reinterpret_cast<const void *>(&msa_projection_splitk_kernel<128, false>),
                        reinterpret_cast<const void *>(&msa_projection_splitk_kernel<64, true>),
                        reinterpret_cast<const void *>(&msa_projection_splitk_kernel<128, true>)};
    return k[(splitk ? 4 : 0) + v];
#endif
}
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

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mu;
EncodeTiledFn g_encode = nullptr;
constexpr int kMaxDevices = 64;
struct DeviceInfo {
    int clusters[4] = {0, 0, 0, 0};  // resident clusters of two CTAs, per kernel variant
    int split_clusters[4][9] = {};   // resident clusters of S one-SM CTAs (-1: none fits)
    int sms = 0;
};
DeviceInfo g_dev[kMaxDevices];

EncodeTiledFn encoder()
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return g_encode;
}

// A [rows, cols] matrix of bf16 (elem_size 2) or 8-bit codes (1) with a row stride
// of `stride` elements, read in boxes of box_rows x 128 bytes with the 128-byte
// swizzle; out-of-range elements read as zero.
bool encode_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t stride,
                int box_rows, int elem_size)
{
    EncodeTiledFn enc = encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)stride * (cuuint64_t)elem_size};
    cuuint32_t box[2] = {(cuuint32_t)(kBKBytes / elem_size), (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, elem_size == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
               const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

void fill_cache(CacheArgs &a, const msa_cache_desc *c)
{
    memset(&a, 0, sizeof a);
    if (!c)
        return;
    a.data = static_cast<uint8_t *>(c->data);
    a.num_pages = c->num_pages;
    a.stride_page = c->stride_page;
    a.stride_head = c->stride_head;
    a.stride_token = c->stride_token;
    a.fp8 = c->dtype == MSA_DTYPE_FP8_E4M3;
}

msa_status validate(const msa_producer_cfg *cfg, int64_t num_tokens, const void *hidden,
                    int64_t hidden_size, int64_t hidden_row_stride, const void *weight,
                    int64_t weight_row_stride, msa_dtype operand_dtype, const float *hidden_scales,
                    const float *weight_scales, const int32_t *positions,
                    const int64_t *slot_mapping, const int32_t *page_table,
                    int64_t page_table_len, const void *q_norm_w, const void *k_norm_w,
                    const void *idx_q_norm_w, const void *idx_k_norm_w, void *q_out,
                    void *idx_q_out, const msa_cache_desc *k_cache, const msa_cache_desc *v_cache,
                    const msa_cache_desc *idx_k_cache, const float *scales, void *rows_out,
                    int64_t rows_out_stride, uint32_t *status)
{
    msa_status s = msa_internal_validate_producer(
        cfg, num_tokens, positions, slot_mapping, page_table, page_table_len, q_norm_w, k_norm_w,
        idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out, k_cache, v_cache, idx_k_cache, scales);
    if (s != MSA_OK || num_tokens == 0)
        return s;
    const int64_t htot = (int64_t)cfg->num_q_heads + 2 * (int64_t)cfg->num_kv_heads +
                         cfg->num_idx_q_heads + cfg->num_idx_k_heads;
    const int64_t W = htot * cfg->head_dim;
    if (num_tokens >= (int64_t)0x7fffffff - kPairM)
        return fail(MSA_ERR_UNSUPPORTED, "num_tokens %lld (limit 2^31 - 257)", (long long)num_tokens);
    if (!hidden || !weight)
        return fail(MSA_ERR_INVALID_ARGUMENT, "hidden and weight are required");
    if (operand_dtype != MSA_DTYPE_BF16 && operand_dtype != MSA_DTYPE_FP8_E4M3)
        return fail(MSA_ERR_UNSUPPORTED, "operand_dtype %d", (int)operand_dtype);
    const int64_t align_elems = operand_dtype == MSA_DTYPE_BF16 ? 8 : 16;  // 16 bytes
    if (hidden_size < 1)
        return fail(MSA_ERR_INVALID_ARGUMENT, "hidden_size %lld", (long long)hidden_size);
    if (hidden_row_stride < hidden_size || weight_row_stride < hidden_size)
        return fail(MSA_ERR_INVALID_ARGUMENT, "row strides must be at least hidden_size");
    if (!aligned(hidden, 16) || !aligned(weight, 16) || hidden_row_stride % align_elems ||
        weight_row_stride % align_elems)
        return fail(MSA_ERR_MISALIGNED,
                    "hidden / weight must be 16-byte aligned with row strides of 16 bytes");
    if ((hidden_scales && !aligned(hidden_scales, 4)) || (weight_scales && !aligned(weight_scales, 4)))
        return fail(MSA_ERR_MISALIGNED, "scales misaligned");
    if (hidden_size > ((int64_t)1 << 31) || W > ((int64_t)1 << 31) ||
        hidden_row_stride > ((int64_t)1 << 36) || weight_row_stride > ((int64_t)1 << 36))
        return fail(MSA_ERR_UNSUPPORTED, "hidden_size, width or row stride out of range");
    if (rows_out) {
        if (rows_out_stride < W)
            return fail(MSA_ERR_INVALID_ARGUMENT, "rows_out_stride %lld < width %lld",
                        (long long)rows_out_stride, (long long)W);
        if (!aligned(rows_out, 16) || rows_out_stride % 8)
            return fail(MSA_ERR_MISALIGNED, "rows_out must be 16-byte aligned, stride 8k elements");
        int64_t tmp;
        if (__builtin_mul_overflow(num_tokens, rows_out_stride, &tmp))
            return fail(MSA_ERR_OFFSET_OVERFLOW, "rows_out extent overflows int64");
    }
    if (status && !aligned(status, 4))
        return fail(MSA_ERR_MISALIGNED, "status misaligned");
    return MSA_OK;
}

}  // namespace

bool msa_internal_encode_byte_rows(CUtensorMap *m, const void *base, int64_t rows, int64_t stride_bytes,
                                   int box_rows)
{
    return encode_map(m, base, rows, kBKBytes, stride_bytes, box_rows, 1);
}

extern "C" msa_status msa_projection_validate(
    const msa_producer_cfg *cfg, int64_t num_tokens, const void *hidden, int64_t hidden_size,
    int64_t hidden_row_stride, const void *weight, int64_t weight_row_stride,
    msa_dtype operand_dtype, const float *hidden_scales, const float *weight_scales,
    const int32_t *positions, const int64_t *slot_mapping, const int32_t *page_table,
    int64_t page_table_len, const void *q_norm_w, const void *k_norm_w, const void *idx_q_norm_w,
    const void *idx_k_norm_w, void *q_out, void *idx_q_out, const msa_cache_desc *k_cache,
    const msa_cache_desc *v_cache, const msa_cache_desc *idx_k_cache, const float *scales,
    void *rows_out, int64_t rows_out_stride, uint32_t *status)
{
    return validate(cfg, num_tokens, hidden, hidden_size, hidden_row_stride, weight,
                    weight_row_stride, operand_dtype, hidden_scales, weight_scales, positions,
                    slot_mapping, page_table, page_table_len,
                    q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out, k_cache,
                    v_cache, idx_k_cache, scales, rows_out, rows_out_stride, status);
}

extern "C" msa_status msa_projection_forward(
    const msa_producer_cfg *cfg, int64_t num_tokens, const void *hidden, int64_t hidden_size,
    int64_t hidden_row_stride, const void *weight, int64_t weight_row_stride,
    msa_dtype operand_dtype, const float *hidden_scales, const float *weight_scales,
    const int32_t *positions, const int64_t *slot_mapping, const int32_t *page_table,
    int64_t page_table_len, const void *q_norm_w, const void *k_norm_w, const void *idx_q_norm_w,
    const void *idx_k_norm_w, void *q_out, void *idx_q_out, const msa_cache_desc *k_cache,
    const msa_cache_desc *v_cache, const msa_cache_desc *idx_k_cache, const float *scales,
    void *rows_out, int64_t rows_out_stride, uint32_t *status, cudaStream_t stream)
{
    msa_status s = validate(cfg, num_tokens, hidden, hidden_size, hidden_row_stride, weight,
                            weight_row_stride, operand_dtype, hidden_scales, weight_scales,
                            positions, slot_mapping, page_table, page_table_len,
                            q_norm_w, k_norm_w, idx_q_norm_w, idx_k_norm_w, q_out, idx_q_out,
                            k_cache, v_cache, idx_k_cache, scales, rows_out, rows_out_stride, status);
    if (s != MSA_OK || num_tokens == 0)
        return s;
    const int32_t D = cfg->head_dim;
    const int64_t htot = (int64_t)cfg->num_q_heads + 2 * (int64_t)cfg->num_kv_heads +
                         cfg->num_idx_q_heads + cfg->num_idx_k_heads;
    const int64_t W = htot * D;

    Params p;
    memset(&p, 0, sizeof p);
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
#ifdef MSA_CHECKED
    for (int ci = 0; ci < 3; ++ci)
        p.cache_hi[ci] = msa_internal_cache_end(&p.cache[ci].data, ci == 2 ? cfg->num_idx_k_heads
                                                                           : cfg->num_kv_heads,
                                                p.cache[ci].num_pages, p.cache[ci].stride_page,
                                                p.cache[ci].stride_head, p.cache[ci].stride_token,
                                                p.cache[ci].fp8 ? 1 : 2, cfg->head_dim,
                                                cfg->page_size);
#endif
    p.scales = scales;
    p.rows_out = static_cast<uint16_t *>(rows_out);
    p.rows_out_stride = rows_out_stride;
    p.hidden_scales = hidden_scales;
    p.weight_scales = weight_scales;
    p.status = status;
#ifdef MSA_CHECKED
    p.out_hi[0] = q_out ? static_cast<const uint8_t *>(q_out) +
                              num_tokens * (int64_t)cfg->num_q_heads * cfg->head_dim * 2
                        : nullptr;
    p.out_hi[1] = idx_q_out ? static_cast<const uint8_t *>(idx_q_out) +
                                  num_tokens * (int64_t)cfg->num_idx_q_heads * cfg->head_dim * 2
                            : nullptr;
    p.rows_hi = rows_out ? static_cast<const uint8_t *>(rows_out) + num_tokens * rows_out_stride * 2
                         : nullptr;
#endif
    p.num_tokens = num_tokens;
    const bool fp8 = operand_dtype == MSA_DTYPE_FP8_E4M3;
    const int es = fp8 ? 1 : 2;
    const int64_t k_per_block = kBKBytes / es;
    p.num_k_blocks = (int32_t)((hidden_size + k_per_block - 1) / k_per_block);
    p.m_tiles = (int32_t)((num_tokens + kPairM - 1) / kPairM);
    p.n_tiles = (int32_t)((W + kBN - 1) / kBN);
    p.n_group = p.n_tiles < MSA_PROJ_NGROUP ? p.n_tiles : MSA_PROJ_NGROUP;
    p.hq = cfg->num_q_heads;
    p.hkv = cfg->num_kv_heads;
    p.hiq = cfg->num_idx_q_heads;
    p.hik = cfg->num_idx_k_heads;
    p.htot = (int32_t)htot;
    p.rotary_dim = cfg->rotary_dim;
    p.rope_style = cfg->rope_style;
    p.page_size = cfg->page_size;
    p.page_shift = -1;
    for (int sh = 0; sh < 31; ++sh)
        if ((1 << sh) == cfg->page_size)
            p.page_shift = sh;
    p.scale_mode = cfg->scale_mode;
    p.rms_eps = cfg->rms_eps;
    // RoPE frequencies theta^(-2k/rd), evaluated in double and rounded once
    for (int k = 0; k < cfg->rotary_dim / 2; ++k)
        p.inv_freq[k] = (float)(1.0 / std::pow((double)cfg->rope_theta,
                                               2.0 * (double)k / (double)cfg->rotary_dim));

    // small batches with the register-resident epilogue: the K dimension split over
    // a cluster (one CTA per SM), when that keeps more SMs busy
    const int rdim = cfg->rotary_dim;
    const bool fast_rope = cfg->rope_style == MSA_ROPE_NEOX && (rdim == D || rdim == D / 2 || rdim == 0);
    int split = 1;
    if (num_tokens <= kBM && fast_rope) {
        int dev0 = 0, sms0 = 0;
        if (cudaGetDevice(&dev0) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms0, cudaDevAttrMultiProcessorCount, dev0) != cudaSuccess)
            return fail(MSA_ERR_CUDA, "device query failed");
        split = sms0 / p.n_tiles;
        split = split > 8 ? 8 : split;
        split = split > p.num_k_blocks ? p.num_k_blocks : split;
        split = split < 1 ? 1 : split;
    }
    p.split = split;
    // weights that each launch reads from DRAM about once (few token tiles): fetched
    // into L2 a number of K blocks ahead of the ring
    p.prefetch = (split > 1 || p.m_tiles <= MSA_PROJ_PREFETCH_MTILES) ? MSA_PROJ_PREFETCH : 0;

    CUtensorMap mx, mw;
    if (!encode_map(&mx, hidden, num_tokens, hidden_size, hidden_row_stride, kBM, es) ||
        !encode_map(&mw, weight, W, hidden_size, weight_row_stride, split > 1 ? kBN : kHalfN, es))
        return fail(MSA_ERR_CUDA, "tensor map encoding failed");

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fail(MSA_ERR_CUDA, "cudaGetDevice failed");
    if (split > 1) {
        const void *sfns[4] = {projection_kernel(true, 0), projection_kernel(true, 1),
                               projection_kernel(true, 2), projection_kernel(true, 3)};
        const int si = (D == 128 ? 1 : 0) + (fp8 ? 2 : 0);
        cudaLaunchConfig_t lc;
        memset(&lc, 0, sizeof lc);
        lc.blockDim = dim3(kThreads);
        lc.dynamicSmemBytes = kSplitDynSmem;
        lc.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)split;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        int fits;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            fits = g_dev[dev].split_clusters[si][split];
            if (fits == 0) {
                int major = 0;
                if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
                    return fail(MSA_ERR_CUDA, "device query failed");
                if (major != 10)
                    return fail(MSA_ERR_UNSUPPORTED, "tcgen05 tensor cores need compute capability 10.x");
                if (cudaFuncSetAttribute(sfns[si], cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSplitDynSmem) != cudaSuccess)
                    return fail(MSA_ERR_CUDA, "cudaFuncSetAttribute failed");
                lc.gridDim = dim3((unsigned)split);
                if (cudaOccupancyMaxActiveClusters(&fits, sfns[si], &lc) != cudaSuccess || fits <= 0) {
                    (void)cudaGetLastError();
                    fits = -1;
                }
                g_dev[dev].split_clusters[si][split] = fits;
            }
        }
        if (fits < 0) {   // no cluster of this size fits: the 2-SM kernel below
            split = 1;
            p.split = 1;
            if (!encode_map(&mw, weight, W, hidden_size, weight_row_stride, kHalfN, es))
                return fail(MSA_ERR_CUDA, "tensor map encoding failed");
        }
    }
    if (split > 1) {
        const void *sfns[4] = {projection_kernel(true, 0), projection_kernel(true, 1),
                               projection_kernel(true, 2), projection_kernel(true, 3)};
        const int si = (D == 128 ? 1 : 0) + (fp8 ? 2 : 0);
        cudaLaunchConfig_t lc;
        memset(&lc, 0, sizeof lc);
        lc.gridDim = dim3((unsigned)(p.n_tiles * split));
        lc.blockDim = dim3(kThreads);
        lc.dynamicSmemBytes = kSplitDynSmem;
        lc.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)split;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        lc.attrs = attr;
        lc.numAttrs = 1;
        void *args[] = {&mx, &mw, &p};
        if (cudaLaunchKernelExC(&lc, sfns[si], args) != cudaSuccess) {
            const cudaError_t e = cudaGetLastError();
            return fail(MSA_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
        }
        msa_internal_set_detail("");
        return MSA_OK;
    }
    const void *fns[4] = {projection_kernel(false, 0), projection_kernel(false, 1),
                          projection_kernel(false, 2), projection_kernel(false, 3)};
    const int vi = (D == 128 ? 1 : 0) + (fp8 ? 2 : 0);
    const void *fn = fns[vi];
    cudaLaunchConfig_t lc;
    memset(&lc, 0, sizeof lc);
    lc.blockDim = dim3(kThreads);
    lc.dynamicSmemBytes = kDynSmem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int clusters;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        clusters = g_dev[dev].clusters[vi];
        if (clusters == 0) {
            int major = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
                return fail(MSA_ERR_CUDA, "device query failed");
            if (major != 10)
                return fail(MSA_ERR_UNSUPPORTED, "tcgen05 tensor cores need compute capability 10.x");
            if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem) !=
                cudaSuccess)
                return fail(MSA_ERR_CUDA, "cudaFuncSetAttribute failed");
            lc.gridDim = dim3(2);
            if (cudaOccupancyMaxActiveClusters(&clusters, fn, &lc) != cudaSuccess || clusters <= 0)
                return fail(MSA_ERR_CUDA, "no cluster of two CTAs fits on this device");
            g_dev[dev].clusters[vi] = clusters;
        }
    }
    const int64_t tiles = (int64_t)p.m_tiles * p.n_tiles;
    lc.gridDim = dim3((unsigned)(2 * (tiles < clusters ? tiles : clusters)));
    void *args[] = {&mx, &mw, &p};
    if (cudaLaunchKernelExC(&lc, fn, args) != cudaSuccess) {
        const cudaError_t e = cudaGetLastError();
        return fail(MSA_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(MSA_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    msa_internal_set_detail("");
    return MSA_OK;
}

msa_status msa_internal_projection_violations(uint64_t *count, int32_t reset)
{
    *count = 0;
#ifdef MSA_CHECKED
    unsigned long long v = 0;
    if (cudaMemcpyFromSymbol(&v, g_msa_projection_violations, sizeof v) != cudaSuccess)
        return MSA_ERR_CUDA;
    if (reset) {
        const unsigned long long z = 0;
        if (cudaMemcpyToSymbol(g_msa_projection_violations, &z, sizeof z) != cudaSuccess)
            return MSA_ERR_CUDA;
    }
    *count = v;
#else
    (void)reset;
#endif
    return MSA_OK;
}

#else
}  // namespace
#endif  // MSA_PROJ_HOST

#if defined(MSA_PROJ_UNIT) && MSA_PROJ_UNIT > 0
#if MSA_PROJ_UNIT == 1
const void *msa_internal_projection_kernel_1() { return reinterpret_cast<const void *>(&msa_projection_kernel<64, false>); }
#elif MSA_PROJ_UNIT == 2
const void *msa_internal_projection_kernel_2() { return reinterpret_cast<const void *>(&msa_projection_kernel<128, false>); }
#elif MSA_PROJ_UNIT == 3
const void *msa_internal_projection_kernel_3() { return reinterpret_cast<const void *>(&msa_projection_kernel<64, true>); }
#elif MSA_PROJ_UNIT == 4
const void *msa_internal_projection_kernel_4() { return reinterpret_cast<const void *>(&msa_projection_kernel<128, true>); }
#elif MSA_PROJ_UNIT == 5
const void *msa_internal_projection_kernel_5() { return reinterpret_cast<const void *>(&msa_projection_splitk_kernel<64, false>); }
#elif MSA_PROJ_UNIT == 6
const void *msa_internal_projection_kernel_6() { return reinterpret_cast<const void *>(&msa_projection_splitk_kernel<128, false>); }
#elif MSA_PROJ_UNIT == 7
const void *msa_internal_projection_kernel_7() { return reinterpret_cast<const void *>(&msa_projection_splitk_kernel<64, true>); }
#elif MSA_PROJ_UNIT == 8
const void *msa_internal_projection_kernel_8() { return reinterpret_cast<const void *>(&msa_projection_splitk_kernel<128, true>); }
#endif
#endif
