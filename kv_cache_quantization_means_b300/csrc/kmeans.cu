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

// Histogram of ids per head.
__global__ void kmeans_count_kernel(UpdateArgs a) {
    __shared__ int hist[kMaxClusters];
    const int h = blockIdx.y;
    for (int j = threadIdx.x; j < a.C; j += blockDim.x) hist[j] = 0;
    __syncthreads();
    const uint8_t* idh = a.ids + (int64_t)h * a.cap + a.tok_offset;
    for (int64_t n = (int64_t)blockIdx.x * blockDim.x * 8 + threadIdx.x;
         n < a.n_tokens && n < (int64_t)(blockIdx.x + 1) * blockDim.x * 8; n += blockDim.x)
        atomicAdd(&hist[min((int)idh[n], a.C - 1)], 1);
    __syncthreads();
    for (int j = threadIdx.x; j < a.C; j += blockDim.x)
        if (hist[j]) atomicAdd(a.counts + (size_t)h * a.C + j, hist[j]);
}

constexpr int kScatterTokens = 2048;

// Counting sort of token indices by cluster: perm[h][offset[j] + k] = the
// k-th token of cluster j (order inside a cluster is immaterial: the sums are
// exact integers).  Each CTA reserves one contiguous range per cluster.
__global__ void kmeans_scatter_kernel(UpdateArgs a) {
    __shared__ int offs[kMaxClusters];
    __shared__ int local[kMaxClusters];
    __shared__ int base[kMaxClusters];
    const int h = blockIdx.y, tid = threadIdx.x;
    const int C = a.C;
    // exclusive scan of counts[h][*] by warp 0
    if (tid < 32) {
        constexpr int kPerLane = kMaxClusters / 32;
        int v[kPerLane], tot = 0;
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
            const int j = tid * kPerLane + k;
            v[k] = j < C ? a.counts[(size_t)h * C + j] : 0;
            tot += v[k];
        }
        int inc = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int u = __shfl_up_sync(0xffffffffu, inc, o);
            if (tid >= o) inc += u;
        }
        int run = inc - tot;
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) {
            const int j = tid * kPerLane + k;
            if (j < kMaxClusters) offs[j] = run;
            run += v[k];
        }
    }
    for (int j = tid; j < kMaxClusters; j += blockDim.x) local[j] = 0;
    __syncthreads();
    const uint8_t* idh = a.ids + (int64_t)h * a.cap + a.tok_offset;
    const int64_t t0 = (int64_t)blockIdx.x * kScatterTokens;
    const int64_t t1 = min(t0 + kScatterTokens, a.n_tokens);
    for (int64_t n = t0 + tid; n < t1; n += blockDim.x) atomicAdd(&local[min((int)idh[n], C - 1)], 1);
    __syncthreads();
    for (int j = tid; j < C; j += blockDim.x) {
        base[j] = local[j] ? offs[j] + atomicAdd(a.cursors + (size_t)h * C + j, local[j]) : 0;
        local[j] = 0;
    }
    __syncthreads();
    int* ph = a.perm + (int64_t)h * a.n_tokens;
    for (int64_t n = t0 + tid; n < t1; n += blockDim.x) {
        const int j = min((int)idh[n], C - 1);
        ph[base[j] + atomicAdd(&local[j], 1)] = (int)n;
    }
}

// bf16 bits -> exact fixed-point parts (units 2^-36 and 2^-75).
__device__ __forceinline__ void fixed_add(uint32_t b, long long& hi, long long& lo) {
    uint32_t e = (b >> 7) & 0xFFu;
    long long m = (long long)((b & 0x7Fu) | (e ? 0x80u : 0u));
    if (e == 0) e = 1;
    if (b & 0x8000u) m = -m;
    if (e >= 98) hi += m * (1ll << min(e - 98u, 54u));   // |x| >= 2^26 is outside the exact range
    else if (e >= 59) lo += m * (1ll << (e - 59));
}

constexpr int kSumPositions = 64;    // sorted positions per warp

template <int DPL>
__device__ __forceinline__ void load_lane_channels(const uint16_t* p, uint32_t* v) {
    if constexpr (DPL == 4) {
        uint2 w = *reinterpret_cast<const uint2*>(p);
        v[0] = w.x & 0xFFFFu; v[1] = w.x >> 16; v[2] = w.y & 0xFFFFu; v[3] = w.y >> 16;
    } else if constexpr (DPL == 2) {
        uint32_t w = *reinterpret_cast<const uint32_t*>(p);
        v[0] = w & 0xFFFFu; v[1] = w >> 16;
    } else {
        v[0] = *p;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) kmeans_sum_kernel(UpdateArgs a) {
    constexpr int DPL = D / 32;          // channels per lane
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = blockIdx.y;
    const int64_t p0 = ((int64_t)blockIdx.x * (kThreads / 32) + warp) * kSumPositions;
    if (p0 >= a.n_tokens) return;
    const int64_t p1 = min(p0 + kSumPositions, a.n_tokens);
    const int* ph = a.perm + (int64_t)h * a.n_tokens;
    const uint8_t* idh = a.ids + (int64_t)h * a.cap + a.tok_offset;
    const uint16_t* xh = a.x + (int64_t)h * a.head_stride + lane * DPL;
    long long hi[DPL], lo[DPL];
#pragma unroll
    for (int k = 0; k < DPL; ++k) hi[k] = lo[k] = 0;
    int cur = -1;
    auto flush = [&](int j) {
        long long* sh = a.sum_hi + ((size_t)h * a.C + j) * D + lane * DPL;
        long long* sl = a.sum_lo + ((size_t)h * a.C + j) * D + lane * DPL;
#pragma unroll
        for (int k = 0; k < DPL; ++k) {
            if (hi[k]) atomicAdd(reinterpret_cast<unsigned long long*>(sh + k), (unsigned long long)hi[k]);
            if (lo[k]) atomicAdd(reinterpret_cast<unsigned long long*>(sl + k), (unsigned long long)lo[k]);
            hi[k] = lo[k] = 0;
        }
    };
    for (int64_t pb = p0; pb < p1; pb += 32) {
        const int cnt = (int)min((int64_t)32, p1 - pb);
        int myn = 0, myj = 0;
        if (lane < cnt) {
            myn = ph[pb + lane];
            myj = min((int)idh[myn], a.C - 1);
        }
        for (int k0 = 0; k0 < cnt; k0 += 8) {
            uint32_t v[8][DPL];
            int jj[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int k = k0 + u;
                const int n = __shfl_sync(0xffffffffu, myn, k & 31);
                jj[u] = __shfl_sync(0xffffffffu, myj, k & 31);
                if (k < cnt) load_lane_channels<DPL>(xh + (int64_t)n * a.token_stride, v[u]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (k0 + u >= cnt) break;
                if (jj[u] != cur) {
                    if (cur >= 0) flush(cur);
                    cur = jj[u];
                }
#pragma unroll
                for (int d = 0; d < DPL; ++d) fixed_add(v[u][d], hi[d], lo[d]);
            }
        }
    }
    if (cur >= 0) flush(cur);
}

// Exact sum -> fp64 -> mean -> bf16; empty clusters keep their centroid.
// Also clears the accumulators for the next iteration.
__global__ void kmeans_mean_kernel(UpdateArgs a, int D) {
    const int hj = blockIdx.x;                  // h * C + j
    const int cnt = a.counts[hj];
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const size_t i = (size_t)hj * D + d;
        const long long hi = a.sum_hi[i], lo = a.sum_lo[i];
        if (cnt > 0) {
            double s = __dadd_rn(__dmul_rn(__ll2double_rn(hi), 0x1p-36),
                                 __dmul_rn(__ll2double_rn(lo), 0x1p-75));
            a.cent[i] = f64_to_bf16_rn(__ddiv_rn(s, (double)cnt));
        }
        a.sum_hi[i] = 0;
        a.sum_lo[i] = 0;
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
    dim3 g1((unsigned)((a.n_tokens + kScatterTokens - 1) / kScatterTokens), (unsigned)a.H);
    kmeans_scatter_kernel<<<g1, kThreads, 0, s>>>(a);
    const int64_t per_cta = (int64_t)(kThreads / 32) * kSumPositions;
    dim3 g2((unsigned)((a.n_tokens + per_cta - 1) / per_cta), (unsigned)a.H);
    kmeans_sum_kernel<D><<<g2, kThreads, 0, s>>>(a);
    kmeans_mean_kernel<<<(unsigned)(a.H * a.C), D < 128 ? D : 128, 0, s>>>(a, D);
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
    switch (D) {
        case 32: return assign_d<32>(H, a, s);
        case 64: return assign_d<64>(H, a, s);
        case 128: return assign_d<128>(H, a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_count(const UpdateArgs& a, cudaStream_t s) {
    if (a.n_tokens == 0) return cudaSuccess;
    const int64_t per = 256 * 8;
    kmeans_count_kernel<<<dim3((unsigned)((a.n_tokens + per - 1) / per), (unsigned)a.H), 256, 0, s>>>(a);
    return cudaGetLastError();
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
