// k-means assign step on the 5th-generation tensor cores (sm_103a).
//
// Quant VideoGen explainer, Sommario tecnico sec. 2A item 1: every token is
// grouped with its nearest centroid (squared Euclidean distance, lowest index
// on ties).  Per head, the distances of a 128-token tile to all C centroids
// are ranked through the score ||c_j||^2 - 2<x, c_j>, whose dot products are
// one [128 x D] x [D x C] bf16 GEMM with fp32 accumulation in tensor memory.
//
// One persistent CTA per SM works through a contiguous range of one head's
// token tiles with warp-specialised roles:
//   warp 0     TMA producer: token tiles (128 rows x 64 channels per copy,
//              128-byte swizzle) into a ring of 2-4 shared-memory stages,
//              the first ring requested before the centroids are staged;
//   warp 1     MMA issuer: tcgen05.mma (M = 128, N = C rounded up to 64,
//              K = 16 per instruction) into one of two TMEM accumulators;
//              also owns the TMEM allocation;
//   warps 2-17 epilogue, two groups of eight: group g takes the tiles that
//              use accumulator g.  The two warps of a group that share a TMEM
//              lane quadrant split a row's columns (and the row's channels for
//              ||x||^2) in halves; a thread owns one tile row and one half,
//              and the pair trades its partial results through shared memory
//              at a 64-thread named barrier.  Groups never wait on one another.
// The GEMM computes the score  <x, c_j> - ||c_j||^2 / 2  directly: one more
// K = 16 block multiplies a constant ones column of the token side by
// -||c_j||^2 / 2 split into three bf16 parts on the centroid side.  The
// nearest centroid is the largest score.  The epilogue makes two passes:
//   A. the row's largest score,
//   B. the bitmask of centroids whose score is within 2E of it, E being a
//      bound on the screen's error that grows with ||x|| (a fit's first
//      assign stores ||x||^2 per token; its later ones, on the same x, read
//      it back).
// A row with one candidate is decided.  The pair splits its other rows (2-3%
// on k-means data) by parity and re-ranks each over the row's candidates with
// direct fp32 distances (relative error bound), then with exact squared
// distances in 128-bit integers, and for near-exact ties with the squared
// distance in fp64 summed in channel order, exactly as the plain definition.
// Centroids (K-major, 128-byte swizzle) stay in shared memory for the whole
// CTA.  Every wait is a bounded
// wait on an mbarrier: on expiry the kernel records an error code, lets the
// other roles drain and returns after freeing its tensor memory.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace qvg {

namespace {

constexpr int kTile = 128;                 // tokens per tile = UMMA M
constexpr int kMaxStages = 4;              // token tiles in flight (fewer when shared memory is short)
constexpr int kEpiWarps = 16;              // two groups of eight (four pairs each)
constexpr int kTcThreads = 64 + 32 * kEpiWarps;
constexpr int kAtomBytes = kTile * 128;    // one 64-channel slab of a tile
constexpr uint32_t kErrTimeout = 0x7E000000u;

// Screen error bound, relative to ||x|| ||c||max and ||c||max^2: the dot
// products are sums of exact bf16 x bf16 products accumulated in fp32 (a
// sequential sum of 128 terms rounded to nearest errs by at most 2^-17 of the
// sum of magnitudes); the bound allows 4x that, plus the fp32 rounding of the
// norms and of the score.
constexpr float kScreenXC = 0x1p-15f;
constexpr float kScreenCC = 0x1p-16f;
// Relative error bound of a direct fp32 sum of D <= 128 squared differences
// ((D + 2) * 2^-24 < 2^-16.9), with a 3.7x margin.
constexpr float kDirectRel = 0x1p-15f;
constexpr float kDirectAbs = 1e-35f;

struct TcArgs {
    const uint16_t* cent;    // [H][C][D]
    int C, Cpad, stages;
    uint8_t* ids;            // [H][cap]
    int64_t cap, tok_offset, n_tokens;
    int tiles_per_head, ctas_per_head;
    int head_inner;              // tensor map dims are (D, H, N) rather than (D, N, H)
    unsigned long long* stats;   // [4] or null
    uint32_t* err;               // or null
    float* xnorm;                // [H][n_tokens] ||x||^2, or null
    int xnorm_mode;              // kNormCompute / kNormStore / kNormLoad
    int* chg_tok;                // changed ids: tokens, (old | new << 8), (start, count) per CTA; or null
    uint16_t* chg_on;
    int2* chg_parts;
    int64_t chg_stride;
    unsigned long long limit;    // bounded waits give up after this many ns
    uint32_t dbg;                // bit 0: the producer withholds each CTA's first tile (tests)
};

// ----------------------------------------------------- shared memory map

struct Layout {
    uint32_t b_off, bx_off, ax_off, x_off, xch_off, bar_off, misc_off, total;
};

// Centroids (nA slabs of Cpad rows), the extra K = 16 block of the centroid
// side (Cpad rows) and of the token side (128 rows) -- 32 bytes a row, as
// unswizzled core matrices (kx_off) -- the
// token stages, the epilogue pairs' exchange words ([pair][half][word][lane],
// 8 words), then the barriers.
__host__ __device__ inline Layout make_layout(int D, int Cpad, int stages) {
    Layout L;
    const int nA = D / 64;
    uint32_t o = 0;
    L.b_off = o;    o += (uint32_t)nA * Cpad * 128;
    L.bx_off = o;   o += (uint32_t)Cpad * 32;
    L.ax_off = o;   o += (uint32_t)kTile * 32;
    L.x_off = o;    o += (uint32_t)stages * nA * kAtomBytes;
    L.xch_off = o;  o += (uint32_t)(kEpiWarps / 2) * 2 * 8 * 32 * 4;
    L.bar_off = o;  o += (uint32_t)(2 * kMaxStages + 4) * 8;
    L.misc_off = o; o += 32;
    L.total = o + 1024;            // slack for 1024-byte alignment of the base
    return L;
}

// Byte offset of 16-byte chunk k (channels 8k..8k+7, k = 0, 1) of row r in
// an extra K = 16 block: 8-row core matrices of 16-byte rows, the two chunks
// of a group 128 bytes apart, groups 256 bytes apart.
__device__ __forceinline__ uint32_t kx_off(int r, int k) {
    return (uint32_t)(r >> 3) * 256u + (uint32_t)k * 128u + (uint32_t)(r & 7) * 16u;
}

template <int D>
__device__ double canonical_dist_smem(const uint8_t* xs, int row, const uint8_t* cs, int j, uint32_t cslab) {
    double acc = 0.0;
    for (int i = 0; i < D; ++i) {
        const float xv = bf16f(*reinterpret_cast<const uint16_t*>(xs + sw_off(row, i, kAtomBytes)));
        const float cv = bf16f(*reinterpret_cast<const uint16_t*>(cs + sw_off(j, i, cslab)));
        const double df = __dsub_rn((double)xv, (double)cv);
        acc = __dadd_rn(acc, __dmul_rn(df, df));
    }
    return acc;
}

// Direct fp32 squared distance, 4 (D = 128) or 2 (D = 64) channels per lane.
template <int D>
__device__ __forceinline__ float warp_dist(const uint8_t* xs, int row, const uint8_t* cs, int j, uint32_t cslab,
                                           int lane) {
    constexpr int CPL = D / 32;
    const int i0 = lane * CPL;
    float acc = 0.0f;
    if (CPL == 4) {
        const uint2 xv = *reinterpret_cast<const uint2*>(xs + sw_off(row, i0, kAtomBytes));
        const uint2 cv = *reinterpret_cast<const uint2*>(cs + sw_off(j, i0, cslab));
        float d;
        d = __fsub_rn(bf16_lo(xv.x), bf16_lo(cv.x)); acc = __fmaf_rn(d, d, acc);
        d = __fsub_rn(bf16_hi(xv.x), bf16_hi(cv.x)); acc = __fmaf_rn(d, d, acc);
        d = __fsub_rn(bf16_lo(xv.y), bf16_lo(cv.y)); acc = __fmaf_rn(d, d, acc);
        d = __fsub_rn(bf16_hi(xv.y), bf16_hi(cv.y)); acc = __fmaf_rn(d, d, acc);
    } else {
        const uint32_t xv = *reinterpret_cast<const uint32_t*>(xs + sw_off(row, i0, kAtomBytes));
        const uint32_t cv = *reinterpret_cast<const uint32_t*>(cs + sw_off(j, i0, cslab));
        float d;
        d = __fsub_rn(bf16_lo(xv), bf16_lo(cv)); acc = __fmaf_rn(d, d, acc);
        d = __fsub_rn(bf16_hi(xv), bf16_hi(cv)); acc = __fmaf_rn(d, d, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

typedef __int128 i128;

// bf16 value in units of 2^-30, exact for 2^-23 <= |x| < 2^16 and for 0
// (|value| < 2^46, so a difference squared and summed over 128 channels stays
// below 2^101); `ok` is cleared for a value outside that range.
__device__ __forceinline__ int64_t bf16_fixed30(uint32_t b, bool& ok) {
    const int e = (int)((b >> 7) & 0xFFu);
    const int64_t m = (int64_t)((b & 0x7Fu) | 0x80u);
    if (e == 0 && (b & 0x7Fu) == 0) return 0;                  // +-0
    if (e < 104 || e > 142) { ok = false; return 0; }
    const int64_t v = m << (e - 104);                          // x = m * 2^(e-134)
    return (b & 0x8000u) ? -v : v;
}

// Exact squared distance in units of 2^-60, channels split over the warp;
// `ok` is false (on every lane) when a value lies outside the exact range.
template <int D>
__device__ __forceinline__ i128 warp_dist_exact(const uint8_t* xs, int row, const uint8_t* cs, int j, uint32_t cslab,
                                                int lane, bool& ok) {
    constexpr int CPL = D / 32;
    const int i0 = lane * CPL;
    bool good = true;
    i128 acc = 0;
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
        const uint32_t xb = *reinterpret_cast<const uint16_t*>(xs + sw_off(row, i0 + k, kAtomBytes));
        const uint32_t cb = *reinterpret_cast<const uint16_t*>(cs + sw_off(j, i0 + k, cslab));
        const int64_t df = bf16_fixed30(xb, good) - bf16_fixed30(cb, good);
        acc += (i128)df * (i128)df;
    }
    ok = __all_sync(0xffffffffu, good);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t lo = (uint64_t)acc, hi = (uint64_t)((unsigned __int128)acc >> 64);
        const uint64_t olo = __shfl_xor_sync(0xffffffffu, lo, o), ohi = __shfl_xor_sync(0xffffffffu, hi, o);
        acc += (i128)(((unsigned __int128)ohi << 64) | (unsigned __int128)olo);
    }
    return acc;
}

// bf16 bits of x, round to nearest even (x finite).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Rows whose fp32 re-rank left several survivors (a few per ten thousand):
// exact squared distances decide (ties -> lowest j); candidates within 2^-40
// of the best, or any value outside the exact range, are settled by the
// channel-order fp64 sum of the plain definition.  Survivor list: lanes of sb
// (lane k holds candidate myj), or -- more than 32 candidates -- every
// candidate of the mask m, re-filtered.  Kept out of line so that the
// epilogue's hot loop stays small.  All 32 lanes call it together.
template <int D, int CP>
__device__ __noinline__ int rerank_exact(const uint8_t* xs, int r, const uint8_t* Bs, uint32_t cslab, int lane,
                                         const uint32_t* m, unsigned sb, int myj, int ncand, float dmin, float emin,
                                         unsigned long long& n_seq) {
    int best = -1;
    const bool listed = ncand <= 32;
    const int nlist = listed ? 32 : CP;
    i128 dbest = 0;
    bool exact = true, near = false;
    for (int k = 0; k < nlist && exact; ++k) {
        int j;
        if (listed) {
            if (!((sb >> k) & 1u)) continue;
            j = __shfl_sync(0xffffffffu, myj, k);
        } else {
            j = k;
            if (!((m[j >> 5] >> (j & 31)) & 1u)) continue;
            const float d = warp_dist<D>(xs, r, Bs, j, cslab, lane);
            if (d - (kDirectRel * d + kDirectAbs) > dmin + emin) continue;
        }
        bool ok;
        const i128 de = warp_dist_exact<D>(xs, r, Bs, j, cslab, lane, ok);
        if (!ok) { exact = false; break; }
        if (best < 0 || de < dbest) {
            if (best >= 0 && dbest - de <= (dbest >> 40)) near = true;
            dbest = de;
            best = j;
        } else if (de - dbest <= (de >> 40)) {
            near = true;
        }
    }
    if (!exact || near) {
        best = -1;
        double cbest = INFINITY;
        for (int k = 0; k < nlist; ++k) {
            int j;
            if (listed) {
                if (!((sb >> k) & 1u)) continue;
                j = __shfl_sync(0xffffffffu, myj, k);
            } else {
                j = k;
                if (!((m[j >> 5] >> (j & 31)) & 1u)) continue;
                const float d = warp_dist<D>(xs, r, Bs, j, cslab, lane);
                if (d - (kDirectRel * d + kDirectAbs) > dmin + emin) continue;
            }
            double cd = 0.0;
            if (lane == 0) cd = canonical_dist_smem<D>(xs, r, Bs, j, cslab);
            cd = __shfl_sync(0xffffffffu, cd, 0);
            if (cd < cbest) { cbest = cd; best = j; }
        }
        ++n_seq;
    }
    return best;
}

template <int D, int CP>
__global__ void __launch_bounds__(kTcThreads, 1)
    kmeans_assign_tc_kernel(const __grid_constant__ CUtensorMap tmap, TcArgs a) {
    constexpr int nA = D / 64;
    constexpr int Cpad = CP;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, derived from the shared array so that accesses stay in
    // the shared window
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int C = a.C, NS = a.stages;
    const Layout L = make_layout(D, Cpad, NS);
    uint8_t* Bs = base + L.b_off;     // centroids c_j
    uint8_t* Bx = base + L.bx_off;    // -||c_j||^2 / 2 as three bf16 parts
    uint8_t* Ax = base + L.ax_off;    // ones column block of the token side
    uint8_t* Xs = base + L.x_off;
    const uint32_t bar0 = smem_u32(base + L.bar_off);
    const uint32_t full_bar = bar0, empty_bar = bar0 + 8 * kMaxStages, tfull_bar = bar0 + 16 * kMaxStages,
                   tempty_bar = tfull_bar + 16;
    // [0] tmem base, [1] abort (producer / MMA), [2] cmax2 bits, [3] abort (epilogue)
    uint32_t* misc = reinterpret_cast<uint32_t*>(base + L.misc_off);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x / a.ctas_per_head, part = blockIdx.x % a.ctas_per_head;
    const int t_begin = (int)((int64_t)part * a.tiles_per_head / a.ctas_per_head);
    const int t_end = (int)((int64_t)(part + 1) * a.tiles_per_head / a.ctas_per_head);
    const int n_tiles = t_end - t_begin;
    const uint32_t cslab = (uint32_t)Cpad * 128u;
    const uint32_t acc_cols = (uint32_t)Cpad;
    uint32_t alloc_cols = 32;
    while (alloc_cols < 2u * acc_cols) alloc_cols <<= 1;

    // ---- set-up: barriers, tensor memory, centroids and their norms
    if (tid == 0) {
        for (int st = 0; st < NS; ++st) {
            mbar_init(full_bar + 8 * st, 1);
            mbar_init(empty_bar + 8 * st, kEpiWarps / 2);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar + 8 * b, 1);
            mbar_init(tempty_bar + 8 * b, kEpiWarps / 2);
        }
        misc[1] = 0;
        misc[2] = 0;
        misc[3] = 0;
        misc[4] = 0;              // changed ids recorded
        fence_mbar_init();
    }
    __syncthreads();
    // the first ring of token tiles is requested now, so that its copies land
    // while the centroids are staged (a stage's first use needs no empty wait)
    const bool withhold = (a.dbg & 1u) != 0;      // test: tile 0 never arrives
    auto issue_tile = [&](int i) {
        const int st = i % NS;
        mbar_arrive_tx(full_bar + 8 * st, (uint32_t)(nA * kAtomBytes));
        const int tok0 = (t_begin + i) * kTile;
        for (int at = 0; at < nA; ++at) {
            const uint32_t dst = smem_u32(Xs + (size_t)(st * nA + at) * kAtomBytes);
            if (a.head_inner) tma_load_3d(dst, &tmap, full_bar + 8 * st, at * 64, h, tok0);
            else tma_load_3d(dst, &tmap, full_bar + 8 * st, at * 64, tok0, h);
        }
    };
    const int pre = n_tiles < NS ? n_tiles : NS;
    if (tid == 0)
        for (int i = 0; i < pre; ++i)
            if (!(withhold && i == 0)) issue_tile(i);
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(misc)),
                     "r"(alloc_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    const uint16_t* cg = a.cent + (int64_t)h * C * D;
    {
        // centroids -> swizzled shared memory, four independent 16-byte loads in flight per thread
        constexpr int kBatch = 4;
        const int total = Cpad * (D / 8);
        for (int v0 = tid; v0 < total; v0 += kTcThreads * kBatch) {
            uint4 val[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = v0 + u * kTcThreads;
                const int j = v / (D / 8), k = v % (D / 8);
                val[u] = make_uint4(0, 0, 0, 0);
                if (v < total && j < C) val[u] = __ldg(reinterpret_cast<const uint4*>(cg + (int64_t)j * D) + k);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = v0 + u * kTcThreads;
                if (v < total) *reinterpret_cast<uint4*>(Bs + sw_off(v / (D / 8), (v % (D / 8)) * 8, cslab)) = val[u];
            }
        }
        // the token side's extra block: 1 in channels 0..2, 0 elsewhere
        for (int v = tid; v < kTile * 2; v += kTcThreads) {
            const int r = v >> 1, k = v & 1;
            uint4 w = make_uint4(0, 0, 0, 0);
            if (k == 0) { w.x = 0x3F803F80u; w.y = 0x00003F80u; }
            *reinterpret_cast<uint4*>(Ax + kx_off(r, k)) = w;
        }
    }
    __syncthreads();
    // -||c_j||^2 / 2 into the centroid side's extra block, one thread per
    // centroid (two fp32 chains of exact bf16 squares; any order of the sum
    // obeys the screen's bound on the norm's rounding)
    for (int j = tid; j < Cpad; j += kTcThreads) {
        float s0 = 0.0f, s1 = 0.0f;
#pragma unroll 4
        for (int i = 0; i < D; i += 8) {
            const uint4 w = *reinterpret_cast<const uint4*>(Bs + sw_off(j, i, cslab));
            s0 = __fmaf_rn(bf16_lo(w.x), bf16_lo(w.x), s0);
            s1 = __fmaf_rn(bf16_hi(w.x), bf16_hi(w.x), s1);
            s0 = __fmaf_rn(bf16_lo(w.y), bf16_lo(w.y), s0);
            s1 = __fmaf_rn(bf16_hi(w.y), bf16_hi(w.y), s1);
            s0 = __fmaf_rn(bf16_lo(w.z), bf16_lo(w.z), s0);
            s1 = __fmaf_rn(bf16_hi(w.z), bf16_hi(w.z), s1);
            s0 = __fmaf_rn(bf16_lo(w.w), bf16_lo(w.w), s0);
            s1 = __fmaf_rn(bf16_hi(w.w), bf16_hi(w.w), s1);
        }
        const float sq = __fadd_rn(s0, s1);
        uint4 w0 = make_uint4(0, 0, 0, 0);
        if (j < C) {
            const float v = -0.5f * sq;              // exact scaling
            const uint16_t hi = f32_to_bf16_bits(v);
            const float r1 = __fsub_rn(v, bf16f(hi));
            const uint16_t mid = f32_to_bf16_bits(r1);
            const uint16_t lo = f32_to_bf16_bits(__fsub_rn(r1, bf16f(mid)));
            w0.x = (uint32_t)hi | ((uint32_t)mid << 16);
            w0.y = lo;
            atomicMax(misc + 2, __float_as_uint(sq));
        } else {
            w0.x = 0xFB80u;                           // -2^120: never the largest score
        }
        *reinterpret_cast<uint4*>(Bx + kx_off(j, 0)) = w0;
        *reinterpret_cast<uint4*>(Bx + kx_off(j, 1)) = make_uint4(0, 0, 0, 0);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const float cm2 = __uint_as_float(misc[2]);
    const float cm = sqrtf(cm2);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int armed = pre;
            for (int i = pre; i < n_tiles; ++i) {
                const int st = i % NS;
                const uint32_t ph = (uint32_t)(i / NS) & 1u;
                if (!mbar_wait(empty_bar + 8 * st, ph ^ 1u, a.limit)) { atomicExch(misc + 1, 1u); break; }
                if (*(volatile uint32_t*)(misc + 1)) break;
                issue_tile(i);
                armed = i + 1;
            }
            // drain: every copy this thread issued has landed before exit
            for (int i = armed - NS > 0 ? armed - NS : 0; i < armed; ++i)
                if (!(withhold && i == 0)) mbar_wait(full_bar + 8 * (i % NS), (uint32_t)(i / NS) & 1u, a.limit);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(Cpad >> 3) << 17) |
                                   ((uint32_t)(kTile >> 4) << 24);
            const uint64_t dax = kmajor_plain_desc(smem_u32(Ax), 128u, 256u),
                           dbx = kmajor_plain_desc(smem_u32(Bx), 128u, 256u);
            int issued = 0;
            for (int i = 0; i < n_tiles; ++i) {
                const int st = i % NS, acc = i & 1;
                const uint32_t ph = (uint32_t)(i / NS) & 1u, aph = (uint32_t)(i >> 1) & 1u;
                if (!mbar_wait(tempty_bar + 8 * acc, aph ^ 1u, a.limit)) { atomicExch(misc + 1, 1u); break; }
                if (!mbar_wait(full_bar + 8 * st, ph, a.limit)) { atomicExch(misc + 1, 1u); break; }
                if (*(volatile uint32_t*)(misc + 1)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)acc * acc_cols;
                umma_bf16(d_tmem, dax, dbx, idesc, 0u);      // -||c||^2 / 2 (overwrites)
                for (int at = 0; at < nA; ++at)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t da = sw128_desc(smem_u32(Xs + (size_t)(st * nA + at) * kAtomBytes) + 32u * k);
                        const uint64_t db = sw128_desc(smem_u32(Bs + (size_t)at * cslab) + 32u * k);
                        umma_bf16(d_tmem, da, db, idesc, 1u);
                    }
                umma_commit(tfull_bar + 8 * acc);
                issued = i + 1;
            }
            // drain: the last accumulators are complete before tensor memory is freed
            for (int i = issued - 2 > 0 ? issued - 2 : 0; i < issued; ++i)
                mbar_wait(tfull_bar + 8 * (i & 1), (uint32_t)(i >> 1) & 1u, a.limit);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue
        const int e = warp - 2;                 // 0..15
        const int g = e >> 3;                   // group = accumulator it drains
        const int hf = (e >> 2) & 1;            // half of the row's columns and channels
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;          // tile row = TMEM lane
        const int pair = g * 4 + q;             // the two warps (halves) on these rows
        constexpr int NW = CP / 32;             // 32-column chunks = mask words
        constexpr int NWH = NW / 2;             // chunks per half
        constexpr int NR = NWH;                 // 32-column tensor-memory reads per half
        constexpr int DH = D / 2;               // channels per half
        uint32_t* xw = reinterpret_cast<uint32_t*>(base + L.xch_off) + (size_t)pair * 2 * 8 * 32 + lane;
        auto xword = [&](int half, int w) -> uint32_t* { return xw + (half * 8 + w) * 32; };
        auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + pair) : "memory"); };
        unsigned long long n_flag = 0, n_exact = 0, n_seq = 0;
        for (int i = g; i < n_tiles; i += 2) {
            const int st = i % NS;
            const uint32_t ph = (uint32_t)(i / NS) & 1u, aph = (uint32_t)(i >> 1) & 1u;
            const int64_t tok = (int64_t)(t_begin + i) * kTile + row;
            const bool valid = tok < a.n_tokens;
            // a stored ||x||^2 is fetched before the waits
            const bool load_norm = a.xnorm_mode == kNormLoad;
            const float xnt_in = load_norm && valid ? __ldg(a.xnorm + (int64_t)h * a.n_tokens + tok) : 0.0f;
            // so is the row's previous id, when changes are recorded
            const uint32_t old_id = a.chg_parts && valid ? a.ids[(int64_t)h * a.cap + a.tok_offset + tok] : 0u;
            const bool ok = mbar_wait(tfull_bar + 8 * g, aph, a.limit) && mbar_wait(full_bar + 8 * st, ph, a.limit);
            const uint8_t* xs = Xs + (size_t)st * nA * kAtomBytes;
            const uint32_t taddr =
                tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)g * acc_cols + 32u * (uint32_t)(hf * NWH);
            uint32_t v[32];
            float pmax = -INFINITY, pxn = 0.0f;
            if (ok) {
                tc_fence_after();
                // Pass A reads the half's NR 32-column chunks one at a time
                // (tensor-memory latency, not arithmetic, sets the pace, so
                // fewer and wider reads beat overlapping narrower ones).
                if (!load_norm) {
                    float2 s2 = make_float2(0.0f, 0.0f), t2 = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int i8 = hf * (DH / 8); i8 < (hf + 1) * (DH / 8); ++i8) {
                        const uint4 w = *reinterpret_cast<const uint4*>(xs + sw_off(row, i8 * 8, kAtomBytes));
                        const float2 f0 = make_float2(bf16_lo(w.x), bf16_hi(w.x)), f1 = make_float2(bf16_lo(w.y), bf16_hi(w.y));
                        const float2 f2v = make_float2(bf16_lo(w.z), bf16_hi(w.z)), f3 = make_float2(bf16_lo(w.w), bf16_hi(w.w));
                        s2 = f2_fma(f0, f0, s2);
                        t2 = f2_fma(f1, f1, t2);
                        s2 = f2_fma(f2v, f2v, s2);
                        t2 = f2_fma(f3, f3, t2);
                    }
                    pxn = (s2.x + s2.y) + (t2.x + t2.y);
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int c = 0; c < NR; ++c) {
                    tmem_ld32(taddr + 32u * c, v);
                    tmem_wait_ld_regs(v);
#pragma unroll
                    for (int jj = 0; jj < 32; jj += 8) {
                        m4[0] = fmax3(m4[0], __uint_as_float(v[jj]), __uint_as_float(v[jj + 1]));
                        m4[1] = fmax3(m4[1], __uint_as_float(v[jj + 2]), __uint_as_float(v[jj + 3]));
                        m4[2] = fmax3(m4[2], __uint_as_float(v[jj + 4]), __uint_as_float(v[jj + 5]));
                        m4[3] = fmax3(m4[3], __uint_as_float(v[jj + 6]), __uint_as_float(v[jj + 7]));
                    }
                }
                pmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            }
            // trade the halves' maxima and norms; a failed wait on either side
            // stops both warps of the pair together
            *xword(hf, 0) = __float_as_uint(pmax);
            *xword(hf, 1) = __float_as_uint(pxn);
            *xword(hf, 2) = ok ? 1u : 0u;
            pair_sync();
            if (!ok || !*xword(hf ^ 1, 2)) {
                atomicExch(misc + 3, 1u);
                break;
            }
            const float b1 = fmaxf(pmax, __uint_as_float(*xword(hf ^ 1, 0)));
            const float xnt = load_norm ? xnt_in : __uint_as_float(*xword(0, 1)) + __uint_as_float(*xword(1, 1));
            if (a.xnorm_mode == kNormStore && hf == 0 && valid) a.xnorm[(int64_t)h * a.n_tokens + tok] = xnt;
            // bound on the error of a score (half the bound on ||c||^2 - 2<x, c>)
            const float E = 0.5f * (1.01f * (kScreenXC * sqrtf(xnt) * cm + kScreenCC * cm2) + 1e-30f);
            const float thr = b1 - 2.0f * E;
            // pass B: the half's candidates, the scores above thr.  E holds a
            // 1% margin over the error bound, so the nearest centroid's score
            // lies strictly above thr and the sign of the exactly rounded
            // thr - score decides.  A chunk's signs are shifted into a word in
            // column order (first column in the top bit), then bit-reversed.
            const float2 thr2 = make_float2(thr, thr);
            uint32_t mw[NWH];
#pragma unroll
            for (int c = 0; c < NR; ++c) {
                tmem_ld32(taddr + 32u * c, v);
                tmem_wait_ld_regs(v);
                uint32_t mrev = 0u;
#pragma unroll
                for (int jj = 0; jj < 32; jj += 2) {
                    const float2 d = f2_sub(thr2, make_float2(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])));
                    mrev = __funnelshift_l(__float_as_uint(d.x), mrev, 1);
                    mrev = __funnelshift_l(__float_as_uint(d.y), mrev, 1);
                }
                mw[c] = __brev(mrev);
            }
            // accumulator drained: hand it back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar + 8 * g);
            // the row's whole candidate mask, low half first
#pragma unroll
            for (int w = 0; w < NWH; ++w) *xword(hf, 4 + w) = mw[w];
            pair_sync();
            uint32_t m[NW];
#pragma unroll
            for (int w = 0; w < NWH; ++w) {
                m[hf * NWH + w] = mw[w];
                m[(hf ^ 1) * NWH + w] = *xword(hf ^ 1, 4 + w);
            }
            int cnt = 0, first = -1;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                if (m[w] && first < 0) first = 32 * w + __ffs(m[w]) - 1;
                cnt += __popc(m[w]);
            }
            uint8_t* idrow = a.ids + (int64_t)h * a.cap + a.tok_offset;
            if (a.chg_parts) {
                // record the decided rows whose id changes: slots of the CTA's
                // range, one run per warp from a shared counter
                const bool dec = valid && cnt == 1 && hf == 0;
                const uint32_t old = old_id;
                const bool chg = dec && old != (uint32_t)first;
                const unsigned bal = __ballot_sync(0xffffffffu, chg);
                if (bal) {
                    const int lead = __ffs(bal) - 1;
                    int base = 0;
                    if (lane == lead) base = (int)atomicAdd(misc + 4, (uint32_t)__popc(bal));
                    base = __shfl_sync(0xffffffffu, base, lead);
                    if (chg) {
                        const int64_t at = (int64_t)h * a.chg_stride + (int64_t)t_begin * kTile + base +
                                           __popc(bal & ((1u << lane) - 1u));
                        a.chg_tok[at] = (int)tok;
                        a.chg_on[at] = (uint16_t)(old | ((uint32_t)first << 8));
                    }
                }
            }
            if (valid && cnt == 1 && hf == 0) idrow[tok] = (uint8_t)first;
            // undecided rows of the pair, alternately to the two halves, one at
            // a time with all lanes on the row
            int k = 0;
            for (unsigned und = __ballot_sync(0xffffffffu, valid && cnt != 1); und; und &= und - 1, ++k) {
                if ((k & 1) != hf) continue;
                const int src = __ffs(und) - 1;
                const int r = q * 32 + src;
                const uint32_t old_r = __shfl_sync(0xffffffffu, old_id, src);
                uint32_t mr[NW];
#pragma unroll
                for (int w = 0; w < NW; ++w) mr[w] = __shfl_sync(0xffffffffu, m[w], src);
                // direct fp32 distances of every candidate; lane k keeps candidate k
                float dmin = INFINITY, myd = INFINITY;
                int ncand = 0, myj = -1;
#pragma unroll
                for (int w = 0; w < NW; ++w)
                    for (uint32_t mm = mr[w]; mm; mm &= mm - 1) {
                        const int j = 32 * w + __ffs(mm) - 1;
                        const float d = warp_dist<D>(xs, r, Bs, j, cslab, lane);
                        if (lane == (ncand & 31)) { myd = d; myj = j; }
                        ++ncand;
                        dmin = fminf(dmin, d);
                    }
                const float emin = kDirectRel * dmin + kDirectAbs;
                // survivors: candidates whose distance may still be the smallest
                unsigned sb = 0xffffffffu;
                int best = -1;
                if (ncand <= 32) {
                    sb = __ballot_sync(0xffffffffu, myj >= 0 && myd - (kDirectRel * myd + kDirectAbs) <= dmin + emin);
                    if (__popc(sb) == 1) best = __shfl_sync(0xffffffffu, myj, __ffs(sb) - 1);
                }
                if (best < 0) {
                    best = rerank_exact<D, CP>(xs, r, Bs, cslab, lane, mr, sb, myj, ncand, dmin, emin, n_seq);
                    ++n_exact;
                }
                if (lane == 0 && best >= 0) {
                    const int64_t rt = (int64_t)(t_begin + i) * kTile + r;
                    if (a.chg_parts) {
                        const uint32_t old = old_r;
                        if (old != (uint32_t)best) {
                            const int64_t at = (int64_t)h * a.chg_stride + (int64_t)t_begin * kTile + atomicAdd(misc + 4, 1u);
                            a.chg_tok[at] = (int)rt;
                            a.chg_on[at] = (uint16_t)(old | ((uint32_t)best << 8));
                        }
                    }
                    idrow[rt] = (uint8_t)best;
                }
                ++n_flag;
            }
            // the token tile is no longer read by this warp
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + 8 * st);
        }
        if (a.stats && lane == 0 && (n_flag | n_exact | n_seq)) {
            atomicAdd(a.stats, n_flag);
            atomicAdd(a.stats + 1, n_exact);
            atomicAdd(a.stats + 2, n_seq);
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && (misc[1] | misc[3]) && a.err) atomicExch(a.err, kErrTimeout);
    if (tid == 0 && a.chg_parts) a.chg_parts[(int64_t)h * kChgParts + part] = make_int2(t_begin * kTile, (int)misc[4]);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(alloc_cols) : "memory");
    }
}

// CTAs per head: balance the tiles of all heads over the SMs, counting about
// two tiles of set-up per CTA.
int ctas_per_head(int H, int tiles) {
    const int sms = sm_count();
    int best_k = 1;
    int64_t best = INT64_MAX;
    for (int k = 1; k <= tiles; ++k) {
        const int64_t waves = ((int64_t)H * k + sms - 1) / sms;
        const int64_t span = waves * ((tiles + k - 1) / k + 2);
        if (span < best) { best = span; best_k = k; }
        if ((int64_t)H * k > 8 * (int64_t)sms) break;
    }
    return best_k;
}

template <int D>
cudaError_t assign_tc_d(int H, const AssignArgs& a, bool* launched, cudaStream_t s) {
    *launched = false;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaSuccess;
    // dims innermost first; the token and head dimensions in stride order
    const bool head_inner = a.head_stride <= a.token_stride;
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3], estr[3] = {1, 1, 1};
    dims[0] = (cuuint64_t)D;
    if (head_inner) {
        dims[1] = (cuuint64_t)H; dims[2] = (cuuint64_t)a.n_tokens;
        strides[0] = (cuuint64_t)a.head_stride * 2; strides[1] = (cuuint64_t)a.token_stride * 2;
        box[0] = 64; box[1] = 1; box[2] = kTile;
    } else {
        dims[1] = (cuuint64_t)a.n_tokens; dims[2] = (cuuint64_t)H;
        strides[0] = (cuuint64_t)a.token_stride * 2; strides[1] = (cuuint64_t)a.head_stride * 2;
        box[0] = 64; box[1] = kTile; box[2] = 1;
    }
    if (H == 1) {
        // a single head: any head stride will do
        if (head_inner) strides[0] = (cuuint64_t)D * 2;
        else strides[1] = strides[0] * (cuuint64_t)a.n_tokens;
    }
    CUtensorMap map;
    const CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.x), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaSuccess;   // layout not expressible: caller falls back
    TcArgs t;
    t.cent = a.cent; t.C = a.C; t.Cpad = (a.C + 63) / 64 * 64;
    t.ids = a.ids; t.cap = a.cap; t.tok_offset = a.tok_offset; t.n_tokens = a.n_tokens;
    t.tiles_per_head = (int)((a.n_tokens + kTile - 1) / kTile);
    t.head_inner = head_inner ? 1 : 0;
    t.ctas_per_head = ctas_per_head(H, t.tiles_per_head);
    t.stats = a.stats;
    t.err = a.err;
    t.xnorm = a.xnorm;
    t.xnorm_mode = a.xnorm ? a.xnorm_mode : kNormCompute;
    t.chg_tok = a.chg_tok; t.chg_on = a.chg_on; t.chg_parts = a.chg_parts; t.chg_stride = a.chg_stride;
    CodecCtl ctl;
    if (!codec_ctl(&ctl)) return cudaSuccess;
    t.limit = ctl.limit;
    t.dbg = ctl.flags;
    if (a.chg_parts && t.ctas_per_head > kChgParts) t.ctas_per_head = kChgParts;   // one record range per CTA
    // as many token stages (up to four) as fit in shared memory, at least two
    t.stages = kMaxStages;
    Layout L = make_layout(D, t.Cpad, t.stages);
    while (L.total > 232448u && t.stages > 2) L = make_layout(D, t.Cpad, --t.stages);
    if (L.total > 232448u) return cudaSuccess;
    // at least 116 KB so that one CTA (and one TMEM allocation) lives per SM
    const size_t smem = L.total < 118784u ? 118784u : L.total;
    auto kern = kmeans_assign_tc_kernel<D, 256>;
    switch (t.Cpad) {
        case 64: kern = kmeans_assign_tc_kernel<D, 64>; break;
        case 128: kern = kmeans_assign_tc_kernel<D, 128>; break;
        case 192: kern = kmeans_assign_tc_kernel<D, 192>; break;
        default: break;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(H * t.ctas_per_head), kTcThreads, smem, s>>>(map, t);
    e = cudaGetLastError();
    if (e == cudaSuccess) *launched = true;
    return e;
}

}  // namespace

cudaError_t launch_assign_tc(int D, int H, const AssignArgs& a, bool* launched, cudaStream_t s) {
    *launched = false;
    if (a.n_tokens == 0 || a.C < 1) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(a.x) & 15u) || (a.head_stride % 8) || (a.token_stride % 8)) return cudaSuccess;
    if (a.n_tokens > (int64_t)INT32_MAX - kTile) return cudaSuccess;
    switch (D) {
        case 64: return assign_tc_d<64>(H, a, launched, s);
        case 128: return assign_tc_d<128>(H, a, launched, s);
        default: return cudaSuccess;
    }
}

}  // namespace qvg
