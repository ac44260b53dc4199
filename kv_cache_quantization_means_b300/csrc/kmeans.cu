// Semantic-aware smoothing: per-head k-means along the token axis.
//
// Quant VideoGen explainer, Sommario tecnico sec. 2A items 1-2: tokens are
// grouped by k-means over the sequence axis and each group's mean (its
// centroid) is computed; sec. 3: centroids are cached across steps.
//
// Assign.  The squared distance ||x - c_j||^2 is ranked through the score
// ||c_j||^2 - 2<x, c_j>, whose dot products are one [128 tokens x D] x
// [D x C] bf16 GEMM per CTA on the tensor cores (fp32 accumulation).  The
// screen has a bounded error E per token, so the result is exact by
// construction: a token whose best score beats the runner-up by more than 2E
// is decided; otherwise its candidates are re-ranked with a direct fp32
// distance (relative error bound) and, if still within that bound, with the
// squared distance in fp64 summed in channel order -- the same arithmetic the
// plain definition uses -- with ties going to the lowest index.
//
// Update.  The per-cluster sums are formed exactly with 64-bit integer
// fixed-point accumulators (two words: 2^-36 and 2^-75 units), so they do not
// depend on the order of accumulation: tokens are bucketed by cluster with a
// counting sort, each warp accumulates a run of one cluster's tokens and adds
// its partial sums with integer atomics.  The mean is the exact sum rounded
// to fp64, divided in fp64 and rounded once to bf16.  Exactness holds for
// |x| >= 2^-68 (smaller magnitudes contribute 0) and cluster sums below 2^27
// in magnitude.
#include "common.cuh"
#include "kernels.h"
#include "exact_mean.cuh"

namespace qvg {

namespace {

constexpr int kThreads = 256;
constexpr int kTile = 128;           // tokens per assign CTA, 16 per warp
constexpr int kPass = 64;            // centroids per accumulator pass

// Error bound of the tensor-core screen, relative to ||x|| ||c||max and
// ||c||max^2.  The dot products are sums of exact bf16 x bf16 products; the
// bound allows 2^-17 relative accumulation error per dot product (8x the
// worst case of a sequential fp32 sum of 128 terms rounded to nearest), plus
// the fp32 rounding of the norms and of the score itself.
constexpr float kScreenXC = 0x1p-15f;
constexpr float kScreenCC = 0x1p-16f;
// Relative error bound of a direct fp32 sum of D <= 128 squared differences
// ((D + 2) * 2^-24 < 2^-16.9), with a 3.7x margin.
constexpr float kDirectRel = 0x1p-15f;
constexpr float kDirectAbs = 1e-35f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct Top3 {
    float b1, b2, b3;
    int a1, a2;
};

__device__ __forceinline__ void top3_push(Top3& t, float v, int j) {
    if (v < t.b3) {
        if (v < t.b2) {
            t.b3 = t.b2;
            if (v < t.b1) {
                t.b2 = t.b1; t.a2 = t.a1; t.b1 = v; t.a1 = j;
            } else {
                t.b2 = v; t.a2 = j;
            }
        } else {
            t.b3 = v;
        }
    }
}

__device__ __forceinline__ void top3_merge_xor(Top3& t, int mask) {
    float o1 = __shfl_xor_sync(0xffffffffu, t.b1, mask);
    float o2 = __shfl_xor_sync(0xffffffffu, t.b2, mask);
    float o3 = __shfl_xor_sync(0xffffffffu, t.b3, mask);
    int p1 = __shfl_xor_sync(0xffffffffu, t.a1, mask);
    int p2 = __shfl_xor_sync(0xffffffffu, t.a2, mask);
    top3_push(t, o1, p1);
    top3_push(t, o2, p2);
    top3_push(t, o3, -1);
}

struct Flag {
    int row, a1, a2, wide;
};

// Squared distance in fp64 accumulated in channel order 0..D-1 (one thread).
template <int D>
__device__ double canonical_dist(const uint16_t* xr, const uint16_t* cr) {
    double acc = 0.0;
#pragma unroll 4
    for (int i = 0; i < D; ++i) {
        double df = __dsub_rn((double)bf16f(xr[i]), (double)bf16f(cr[i]));
        acc = __dadd_rn(acc, __dmul_rn(df, df));
    }
    return acc;
}

// Direct fp32 squared distance, channels split over the warp.
template <int D>
__device__ float warp_direct_dist(const uint16_t* xr, const uint16_t* cr, int lane) {
    float acc = 0.0f;
#pragma unroll
    for (int i = lane; i < D; i += 32) {
        float df = __fsub_rn(bf16f(xr[i]), bf16f(cr[i]));
        acc = __fmaf_rn(df, df, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    return acc;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) kmeans_assign_kernel(AssignArgs a) {
    constexpr int LD = D + 8;               // padded smem row (bank-conflict-free ldmatrix)
    constexpr int KSTEPS = D / 16;
    extern __shared__ __align__(16) unsigned char smem[];
    const int C = a.C;
    const int Cpad = (C + kPass - 1) / kPass * kPass;
    uint16_t* cs = reinterpret_cast<uint16_t*>(smem);                 // [Cpad][LD]
    uint16_t* xs = cs + (size_t)Cpad * LD;                            // [kTile][LD]
    float* cn = reinterpret_cast<float*>(xs + (size_t)kTile * LD);    // [Cpad]
    int* hist = reinterpret_cast<int*>(cn + Cpad);                    // [Cpad]
    Flag* flags = reinterpret_cast<Flag*>(hist + Cpad);               // [kTile]
    int* nflag = reinterpret_cast<int*>(flags + kTile);
    float* cmax2 = reinterpret_cast<float*>(nflag + 1);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y;
    const int64_t n0 = (int64_t)blockIdx.x * kTile;
    const uint16_t* cg = a.cent + (size_t)h * C * D;
    const uint16_t* xg = a.x + (int64_t)h * a.head_stride;

    // ---- stage centroids and the token tile in shared memory
    for (int v = tid; v < Cpad * (D / 8); v += kThreads) {
        int j = v / (D / 8), k = v % (D / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (j < C) val = __ldg(reinterpret_cast<const uint4*>(cg + (size_t)j * D) + k);
        *reinterpret_cast<uint4*>(cs + (size_t)j * LD + k * 8) = val;
    }
    for (int v = tid; v < kTile * (D / 8); v += kThreads) {
        int r = v / (D / 8), k = v % (D / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (n0 + r < a.n_tokens) val = ldg_nc_v4(xg + (n0 + r) * a.token_stride + k * 8);
        *reinterpret_cast<uint4*>(xs + (size_t)r * LD + k * 8) = val;
    }
    if (tid == 0) { *nflag = 0; *cmax2 = 0.0f; }
    for (int j = tid; j < Cpad; j += kThreads) hist[j] = 0;
    __syncthreads();
    for (int j = tid; j < Cpad; j += kThreads) {
        float acc = 0.0f;
        for (int i = 0; i < D; ++i) {
            float c = bf16f(cs[(size_t)j * LD + i]);
            acc = __fmaf_rn(c, c, acc);
        }
        cn[j] = j < C ? acc : INFINITY;
        if (j < C) atomicMax(reinterpret_cast<int*>(cmax2), __float_as_int(acc));
    }
    __syncthreads();

    // ---- per warp: 16 tokens x all centroids on the tensor cores
    const int g = lane >> 2, q = lane & 3;
    const int rbase = warp * 16;
    // ||x||^2 of rows g and g+8 (quad-split, then reduced)
    float xn2[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const uint16_t* xr = xs + (size_t)(rbase + g + 8 * s) * LD;
        float acc = 0.0f;
        for (int i = q * (D / 4); i < (q + 1) * (D / 4); ++i) {
            float v = bf16f(xr[i]);
            acc = __fmaf_rn(v, v, acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        xn2[s] = acc;
    }
    uint32_t afrag[KSTEPS][4];
    {
        const int r = lane & 15, cofs = (lane >> 4) * 8;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk)
            ldsm_x4(smem_u32(xs + (size_t)(rbase + r) * LD + kk * 16 + cofs), afrag[kk][0], afrag[kk][1],
                    afrag[kk][2], afrag[kk][3]);
    }
    Top3 t[2];
#pragma unroll
    for (int s = 0; s < 2; ++s) { t[s].b1 = t[s].b2 = t[s].b3 = INFINITY; t[s].a1 = t[s].a2 = 0; }

    // ldmatrix.x4 address for B: lanes 0-7 -> n-tile A rows, k lo; 8-15 -> k hi;
    // 16-23 -> n-tile A+1 rows, k lo; 24-31 -> k hi.
    const int brow = (lane & 7) + ((lane >> 4) << 3), bk = ((lane >> 3) & 1) * 8;
    for (int p = 0; p < Cpad; p += kPass) {
        float acc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[nt][r] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
#pragma unroll
            for (int ntp = 0; ntp < 4; ++ntp) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(cs + (size_t)(p + ntp * 16 + brow) * LD + kk * 16 + bk), b0, b1, b2, b3);
                mma_bf16_16816(acc[2 * ntp], afrag[kk], b0, b1);
                mma_bf16_16816(acc[2 * ntp + 1], afrag[kk], b2, b3);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int j = p + nt * 8 + 2 * q + (r & 1);
                const float sc = __fsub_rn(cn[j], 2.0f * acc[nt][r]);
                top3_push(t[r >> 1], sc, j);
            }
        }
    }
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        top3_merge_xor(t[s], 1);
        top3_merge_xor(t[s], 2);
    }

    // ---- decide or flag
    const float cm2 = *cmax2;
    const float cm = sqrtf(cm2);
    if (q == 0) {
#pragma unroll
        for (int s = 0; s < 2; ++s) {
            const int row = rbase + g + 8 * s;
            const int64_t n = n0 + row;
            if (n >= a.n_tokens) continue;
            const float E = 1.01f * (kScreenXC * sqrtf(xn2[s]) * cm + kScreenCC * cm2) + 1e-30f;
            const float lim = t[s].b1 + 2.0f * E;
            if (t[s].b2 > lim) {
                a.ids[(int64_t)h * a.cap + a.tok_offset + n] = (uint8_t)t[s].a1;
                atomicAdd(&hist[t[s].a1], 1);
            } else {
                int e = atomicAdd(nflag, 1);
                flags[e] = Flag{row, t[s].a1, t[s].a2, t[s].b3 <= lim ? 1 : 0};
            }
        }
    }
    __syncthreads();

    // ---- refine flagged rows (one warp per row)
    const int nf = *nflag;
    for (int e = warp; e < nf; e += kThreads / 32) {
        const Flag f = flags[e];
        const uint16_t* xr = xs + (size_t)f.row * LD;
        int best;
        if (!f.wide) {
            const float d1 = warp_direct_dist<D>(xr, cs + (size_t)f.a1 * LD, lane);
            const float d2 = warp_direct_dist<D>(xr, cs + (size_t)f.a2 * LD, lane);
            const float e1 = kDirectRel * d1 + kDirectAbs, e2 = kDirectRel * d2 + kDirectAbs;
            if (d1 + e1 < d2 - e2) {
                best = f.a1;
            } else if (d2 + e2 < d1 - e1) {
                best = f.a2;
            } else {
                double c = 0.0;
                if (lane < 2) c = canonical_dist<D>(xr, cs + (size_t)(lane == 0 ? f.a1 : f.a2) * LD);
                const double c1 = __shfl_sync(0xffffffffu, c, 0), c2 = __shfl_sync(0xffffffffu, c, 1);
                if (c1 < c2) best = f.a1;
                else if (c2 < c1) best = f.a2;
                else best = min(f.a1, f.a2);
                if (a.stats && lane == 0) atomicAdd(a.stats + 1, 1ull);
            }
        } else {
            // every centroid: direct fp32 distances, then fp64 among the survivors
            constexpr int kPer = kMaxClusters / 32;
            float d[kPer];
            float dmin = INFINITY;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int j = lane + 32 * k;
                d[k] = INFINITY;
                if (j < C) {
                    const uint16_t* cr = cs + (size_t)j * LD;
                    float acc = 0.0f;
                    for (int i = 0; i < D; ++i) {
                        float df = __fsub_rn(bf16f(xr[i]), bf16f(cr[i]));
                        acc = __fmaf_rn(df, df, acc);
                    }
                    d[k] = acc;
                    dmin = fminf(dmin, acc);
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dmin = fminf(dmin, __shfl_xor_sync(0xffffffffu, dmin, o));
            const float emin = kDirectRel * dmin + kDirectAbs;
            double cbest = INFINITY;
            int jbest = 0x7fffffff;
            int ncand = 0;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int j = lane + 32 * k;
                const bool cand = j < C && d[k] - (kDirectRel * d[k] + kDirectAbs) <= dmin + emin;
                ncand += __popc(__ballot_sync(0xffffffffu, cand));
                if (cand) {
                    const double c = canonical_dist<D>(xr, cs + (size_t)j * LD);
                    if (c < cbest || (c == cbest && j < jbest)) { cbest = c; jbest = j; }
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const double oc = __shfl_xor_sync(0xffffffffu, cbest, o);
                const int oj = __shfl_xor_sync(0xffffffffu, jbest, o);
                if (oc < cbest || (oc == cbest && oj < jbest)) { cbest = oc; jbest = oj; }
            }
            best = jbest;
            if (a.stats && lane == 0) atomicAdd(a.stats + 2, 1ull);
            (void)ncand;
        }
        if (lane == 0) {
            a.ids[(int64_t)h * a.cap + a.tok_offset + n0 + f.row] = (uint8_t)best;
            atomicAdd(&hist[best], 1);
        }
    }
    if (a.stats && tid == 0 && nf) atomicAdd(a.stats, (unsigned long long)nf);
    if (a.counts) {
        __syncthreads();
        for (int j = tid; j < C; j += kThreads)
            if (hist[j]) atomicAdd(a.counts + (size_t)h * C + j, hist[j]);
    }
}

// c_j = x[floor(j*N/C)] (cold) or warm[j] for every head; one CTA per (j, h).
__global__ void kmeans_init_kernel(const uint16_t* x, int64_t head_stride, int64_t token_stride,
                                   int64_t n_tokens, const uint16_t* warm, int C, int D,
                                   uint16_t* cent) {
    const int j = blockIdx.x, h = blockIdx.y;
    const uint16_t* src;
    if (warm) src = warm + ((size_t)h * C + j) * D;
    else src = x + (int64_t)h * head_stride + (((int64_t)j * n_tokens) / C) * token_stride;
    uint16_t* dst = cent + ((size_t)h * C + j) * D;
    for (int k = threadIdx.x; k < D / 8; k += blockDim.x)
        reinterpret_cast<uint4*>(dst)[k] = __ldg(reinterpret_cast<const uint4*>(src) + k);
}

// ------------------------------------------------------------- update ---
//
// 1. sort: per block of kSortBlock tokens a histogram of ids, then a stable
//    counting sort of the tokens by cluster (perm), the cluster sizes and a
//    table of pieces: runs of at most kPieceTokens sorted positions of one
//    cluster.  Offsets come from the block histograms in a fixed order and
//    ranks from __match_any_sync, so neither the counts nor the order depend
//    on scheduling.
// 2. sum: one warp per piece gathers its rows and forms their exact sum
//    (fixed-point windows); the only piece of a cluster is turned into the
//    centroid directly, other pieces store their exact partial.
// 3. mean: clusters with several pieces add their partials in piece order
//    and round the mean.  Integer sums make the result independent of any
//    order; no atomic operation is used.

constexpr int kSortWarps = kThreads / 32;
constexpr int kSortPerWarp = kSortBlock / kSortWarps;

// Exclusive scan of v over threads 0..kMaxClusters-1 of a 256-thread block;
// returns the prefix, *total receives the sum.
__device__ __forceinline__ int block_scan256(int v, int* warp_tot, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int before = 0, all = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
        if (w < warp) before += warp_tot[w];
        all += warp_tot[w];
    }
    __syncthreads();
    *total = all;
    return before + inc - v;
}

// Histogram of the ids of one block of kSortBlock tokens.
__global__ void __launch_bounds__(kThreads) kmeans_hist_kernel(UpdateArgs a) {
    __shared__ int hist[kMaxClusters];
    const int h = blockIdx.y, b = blockIdx.x, C = a.C;
    for (int j = threadIdx.x; j < kMaxClusters; j += kThreads) hist[j] = 0;
    __syncthreads();
    const uint8_t* idh = a.ids + (int64_t)h * a.cap + a.tok_offset;
    const int64_t n0 = (int64_t)b * kSortBlock, n1 = min(n0 + kSortBlock, a.n_tokens);
    for (int64_t n = n0 + threadIdx.x; n < n1; n += kThreads) atomicAdd(&hist[min((int)idh[n], C - 1)], 1);
    __syncthreads();
    int* bh = a.blockhist + ((int64_t)h * a.n_blocks + b) * C;
    for (int j = threadIdx.x; j < C; j += kThreads) bh[j] = hist[j];
}

// Stable counting sort, one block of kSortBlock tokens per CTA: the block's
// first position for cluster j is (tokens of clusters < j) + (tokens of j in
// earlier blocks), both from the block histograms in a fixed order; inside the
// block, warp w's slice follows warps < w and a warp ranks equal ids with
// __match_any_sync.  Block 0 of each head also writes the counts and the
// table of pieces.
__global__ void __launch_bounds__(kThreads) kmeans_scatter_kernel(UpdateArgs a) {
    __shared__ int cur[kSortWarps][kMaxClusters];
    __shared__ int warp_tot[kThreads / 32];
    __shared__ __align__(16) uint8_t ids_s[kSortBlock];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y, b = blockIdx.x, C = a.C;
    const uint8_t* idh = a.ids + (int64_t)h * a.cap + a.tok_offset;
    const int64_t n0 = (int64_t)b * kSortBlock;
    const int nb = (int)min((int64_t)kSortBlock, a.n_tokens - n0);
    for (int i = tid; i < nb; i += kThreads) ids_s[i] = idh[n0 + i];
    for (int i = tid; i < kSortWarps * kMaxClusters; i += kThreads) (&cur[0][0])[i] = 0;
    // totals and the part before this block, per cluster (thread j)
    const int* bh = a.blockhist + (int64_t)h * a.n_blocks * C;
    int total = 0, before = 0;
    if (tid < C)
        for (int bb = 0; bb < a.n_blocks; ++bb) {
            const int v = bh[(int64_t)bb * C + tid];
            total += v;
            if (bb < b) before += v;
        }
    int all;
    const int off = block_scan256(tid < C ? total : 0, warp_tot, &all);   // also syncs ids_s / cur
    const int np = (total + kPieceTokens - 1) / kPieceTokens;
    int np_all;
    const int pfirst = block_scan256(tid < C ? np : 0, warp_tot, &np_all);
    if (b == 0 && tid < C) {
        a.counts[(int64_t)h * C + tid] = total;
        a.first_piece[(int64_t)h * C + tid] = pfirst;
        int4* ph = a.pieces + (int64_t)h * a.max_pieces;
        for (int p = 0; p < np; ++p)
            ph[pfirst + p] = make_int4(off + p * kPieceTokens, min(kPieceTokens, total - p * kPieceTokens), tid,
                                       np == 1 ? 1 : 0);
    }
    if (b == 0 && tid == 0) a.npieces[h] = np_all;
    // per-warp histograms of this block
    const int w0 = warp * kSortPerWarp, w1 = min(w0 + kSortPerWarp, nb);
    for (int bs = w0; bs < w1; bs += 32) {
        const int n = bs + lane;
        const int id = n < w1 ? min((int)ids_s[n], C - 1) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, id);
        if (id >= 0 && lane == __ffs(m) - 1) cur[warp][id] += __popc(m);
    }
    __syncthreads();
    if (tid < C) {
        int run = off + before;
        for (int w = 0; w < kSortWarps; ++w) {
            const int t = cur[w][tid];
            cur[w][tid] = run;
            run += t;
        }
    }
    __syncthreads();
    int* perm = a.perm + (int64_t)h * a.n_tokens;
    const unsigned lt = (1u << lane) - 1u;
    for (int bs = w0; bs < w1; bs += 32) {
        const int n = bs + lane;
        const int id = n < w1 ? min((int)ids_s[n], C - 1) : -1;
        const unsigned m = __match_any_sync(0xffffffffu, id);
        if (id >= 0) perm[cur[warp][id] + __popc(m & lt)] = (int)(n0 + n);
        __syncwarp();
        if (id >= 0 && lane == __ffs(m) - 1) cur[warp][id] += __popc(m);
        __syncwarp();
    }
}

__device__ __forceinline__ i128 shfl_xor_i128(i128 v, int mask) {
    const uint64_t lo = (uint64_t)v, hi = (uint64_t)((u128)v >> 64);
    const uint64_t olo = __shfl_xor_sync(0xffffffffu, lo, mask), ohi = __shfl_xor_sync(0xffffffffu, hi, mask);
    return (i128)(((u128)ohi << 64) | (u128)olo);
}

// One warp per piece.  The warp stages the piece's rows (at most
// kPieceTokens, gathered in sorted order) kSumRows at a time into its slice of
// shared memory with 16-byte asynchronous copies, all of a round in flight at
// once, then sums them from there.  A lane owns 8 consecutive channels of one
// row slot; D/8 lanes cover a row and 32/(D/8) rows go per instruction.  Row
// slots are reduced at the end (integer additions: exact, any order).
constexpr int kSumWarps = 4;
constexpr int kSumRows = 16;      // rows staged per round
static_assert(kPieceTokens <= 64, "a warp holds a piece's token indices in two registers per lane");

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

template <int D>
__global__ void __launch_bounds__(32 * kSumWarps, 8) kmeans_sum_kernel(UpdateArgs a) {
    constexpr int LPR = D / 8, RPI = 32 / LPR;
    extern __shared__ __align__(16) uint16_t sum_rows[];     // [warp][kSumRows][D]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % LPR, slot = lane / LPR;
    const int h = blockIdx.y;
    const int p = blockIdx.x * kSumWarps + warp;
    if (p >= a.npieces[h]) return;
    uint16_t* rows = sum_rows + (size_t)warp * kSumRows * D;
    const int4 pc = a.pieces[(int64_t)h * a.max_pieces + p];
    const int start = pc.x, len = pc.y, j = pc.z;
    const int* ph = a.perm + (int64_t)h * a.n_tokens + start;
    const uint16_t* xh = a.x + (int64_t)h * a.head_stride + sub * 8;
    // the piece's token indices (len <= kPieceTokens = 64): lane k holds
    // positions k and k + 32
    const int pa = lane < len ? ph[lane] : 0, pb = lane + 32 < len ? ph[lane + 32] : 0;
    // rows [r0, r0 + kSumRows) of the piece into the warp's slice
    auto stage = [&](int r0) {
        for (int k0 = 0; k0 < kSumRows; k0 += RPI) {
            const int k = r0 + k0 + slot;
            const int na = __shfl_sync(0xffffffffu, pa, k & 31), nb = __shfl_sync(0xffffffffu, pb, k & 31);
            if (k < len)
                cp_async16(smem_u32(rows + (k0 + slot) * D + sub * 8), xh + (int64_t)(k < 32 ? na : nb) * a.token_stride);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncwarp();
    };
    int w1[8], w2[8], w3[8];
#pragma unroll
    for (int d = 0; d < 8; ++d) w1[d] = w2[d] = w3[d] = 0;
    float amax = 0.0f;
    for (int r0 = 0; r0 < len; r0 += kSumRows) {
        stage(r0);
#pragma unroll 2
        for (int k = slot; k < kSumRows && r0 + k < len; k += RPI) {
            const uint4 v = *reinterpret_cast<const uint4*>(rows + k * D + sub * 8);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float lo = bf16_lo(wv[q]), hi = bf16_hi(wv[q]);
                amax = fmax3(amax, fabsf(lo), fabsf(hi));
                window_add2(make_float2(lo, hi), w1 + 2 * q, w2 + 2 * q, w3 + 2 * q);
            }
        }
        __syncwarp();                      // the slice is read before the next round overwrites it
    }
    i128 tot[8];
    if (__any_sync(0xffffffffu, !(amax < kWinMax))) {
        // a value outside the first window: redo the piece with 128-bit sums
#pragma unroll
        for (int d = 0; d < 8; ++d) tot[d] = 0;
        for (int k = slot; k < len; k += RPI) {
            const uint4 v = ldg_nc_v4(xh + (int64_t)ph[k] * a.token_stride);
            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                tot[2 * q] += bf16_to_i128_units(wv[q] & 0xFFFFu);
                tot[2 * q + 1] += bf16_to_i128_units(wv[q] >> 16);
            }
        }
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
            for (int d = 0; d < 8; ++d) tot[d] += shfl_xor_i128(tot[d], o);
    } else {
        // row slots first, in int32 (at most kPieceTokens terms of <= 2^22 each)
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                w1[d] += __shfl_xor_sync(0xffffffffu, w1[d], o);
                w2[d] += __shfl_xor_sync(0xffffffffu, w2[d], o);
                w3[d] += __shfl_xor_sync(0xffffffffu, w3[d], o);
            }
#pragma unroll
        for (int d = 0; d < 8; ++d) tot[d] = windows_to_i128(w1[d], w2[d], w3[d]);
    }
    if (slot != 0) return;
    if (pc.w) {
        uint16_t r[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) r[d] = mean_bf16_bits(tot[d], (uint32_t)len);
        uint4 o;
        o.x = r[0] | ((uint32_t)r[1] << 16); o.y = r[2] | ((uint32_t)r[3] << 16);
        o.z = r[4] | ((uint32_t)r[5] << 16); o.w = r[6] | ((uint32_t)r[7] << 16);
        *reinterpret_cast<uint4*>(a.cent + ((int64_t)h * a.C + j) * D + sub * 8) = o;
    } else {
        i128* pr = reinterpret_cast<i128*>(a.partials) + ((int64_t)h * a.max_pieces + p) * D + sub * 8;
#pragma unroll
        for (int d = 0; d < 8; ++d) pr[d] = tot[d];
    }
}

// Clusters made of several pieces: add the partials in piece order, round.
template <int D>
__global__ void kmeans_mean_kernel(UpdateArgs a) {
    const int j = blockIdx.x, h = blockIdx.y;
    const int cnt = a.counts[(int64_t)h * a.C + j];
    const int np = (cnt + kPieceTokens - 1) / kPieceTokens;
    if (np <= 1) return;
    const int first = a.first_piece[(int64_t)h * a.C + j];
    const i128* pr = reinterpret_cast<const i128*>(a.partials) + ((int64_t)h * a.max_pieces + first) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        i128 s = 0;
        for (int p = 0; p < np; ++p) s += pr[(int64_t)p * D + d];
        a.cent[((int64_t)h * a.C + j) * D + d] = mean_bf16_bits(s, (uint32_t)cnt);
    }
}

__global__ void set_chunk_kernel(int64_t* off, int32_t* ver, int idx, int64_t begin, int64_t end,
                                 int32_t version) {
    if (idx == 0) off[0] = begin;
    off[idx + 1] = end;
    ver[idx] = version;
}

size_t assign_smem(int D, int C) {
    const int Cpad = (C + kPass - 1) / kPass * kPass;
    const int LD = D + 8;
    return (size_t)Cpad * LD * 2 + (size_t)kTile * LD * 2 + (size_t)Cpad * 4 * 2 + sizeof(Flag) * kTile + 16;
}

template <int D>
cudaError_t assign_d(int H, const AssignArgs& a, cudaStream_t s) {
    if (a.n_tokens == 0) return cudaSuccess;
    const size_t smem = assign_smem(D, a.C);
    cudaError_t e = cudaFuncSetAttribute(kmeans_assign_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.n_tokens + kTile - 1) / kTile), (unsigned)H);
    kmeans_assign_kernel<D><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t update_d(const UpdateArgs& a, cudaStream_t s) {
    if (a.n_tokens == 0) return cudaSuccess;
    dim3 g1((unsigned)a.n_blocks, (unsigned)a.H);
    kmeans_hist_kernel<<<g1, kThreads, 0, s>>>(a);
    kmeans_scatter_kernel<<<g1, kThreads, 0, s>>>(a);
    dim3 g2((unsigned)((a.max_pieces + kSumWarps - 1) / kSumWarps), (unsigned)a.H);
    const size_t sum_smem = sizeof(uint16_t) * kSumWarps * kSumRows * D;
    cudaError_t e = cudaFuncSetAttribute(kmeans_sum_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sum_smem);
    if (e != cudaSuccess) return e;
    kmeans_sum_kernel<D><<<g2, 32 * kSumWarps, sum_smem, s>>>(a);
    kmeans_mean_kernel<D><<<dim3((unsigned)a.C, (unsigned)a.H), D, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_kmeans_init(int D, const uint16_t* x, int64_t head_stride, int64_t token_stride,
                               int64_t n_tokens, const uint16_t* warm, int H, int C, uint16_t* cent,
                               cudaStream_t s) {
    kmeans_init_kernel<<<dim3((unsigned)C, (unsigned)H), 32, 0, s>>>(x, head_stride, token_stride, n_tokens,
                                                                     warm, C, D, cent);
    return cudaGetLastError();
}

cudaError_t launch_assign(int D, int H, const AssignArgs& a, cudaStream_t s) {
    bool launched = false;
    const cudaError_t e = launch_assign_tc(D, H, a, &launched, s);
    if (e != cudaSuccess || launched) return e;
    switch (D) {
        case 32: return assign_d<32>(H, a, s);
        case 64: return assign_d<64>(H, a, s);
        case 128: return assign_d<128>(H, a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_update(int D, const UpdateArgs& a, cudaStream_t s) {
    switch (D) {
        case 32: return update_d<32>(a, s);
        case 64: return update_d<64>(a, s);
        case 128: return update_d<128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_set_chunk(int64_t* chunk_offset, int32_t* chunk_version, int idx, int64_t begin,
                             int64_t end, int32_t version, cudaStream_t s) {
    set_chunk_kernel<<<1, 1, 0, s>>>(chunk_offset, chunk_version, idx, begin, end, version);
    return cudaGetLastError();
}

}  // namespace qvg
