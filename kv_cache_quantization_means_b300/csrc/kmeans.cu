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
// One CTA per (head, group of 2^k consecutive clusters), one launch per
// update.  Cluster sums are exact integers (three fixed-point windows per
// value), so they do not depend on the order in which tokens are listed or
// added, and shared-memory atomics may place and add them in any order.
//
// Full update: the CTA finds its clusters' tokens in the id array itself --
// one scan counts them and lists their token indices in shared memory in
// arrival order, and a counting sort in shared memory groups that list by
// cluster.  Each unit of D/8 lanes takes a contiguous run of the sorted list,
// gathers those rows and adds them into per-lane windows, which it flushes
// into the cluster's shared sums when its run reaches the next cluster.  The
// sums and counts are stored for the next update, and the means rounded.  A
// group whose tokens overflow the list is taken in token segments (a
// counting scan and a placing scan each); a group holding a value of
// magnitude >= 2^14 is summed again with 128-bit integers and marked, so that
// its next update is a full one too.
//
// Incremental update: the stored sums already hold the members under the
// previous ids, and the assign in between recorded the ids it changed.  The
// CTA lists the changes that touch its clusters (a token leaving is
// subtracted from the old cluster, one arriving added to the new), sums those
// rows the same way, adds the result to the stored sums and counts, and
// rounds again the means of the clusters that changed; the others keep their
// centroid, which is already the mean of the same members.  A changed row
// with a value of magnitude >= 2^14 sends the group to a full update.

constexpr int kUpdThreads = 256;
constexpr int kListCap = 4096;                         // rows listed at once
constexpr int kMaxGroup = 16;                          // clusters per CTA
constexpr int kScanR = 2;                              // 16-byte chunks per lane and round of an id scan
constexpr int kSumRows = 4;                            // token rows a unit has in flight
constexpr int kSumAhead = 2 * kSumRows;                // rows ahead a unit asks into L2
constexpr int kFlushTerms = 255;                       // window terms a lane adds between flushes (|sum| < 2^30)
constexpr int64_t kPackLimit = (int64_t)1 << 26;       // token index packed above a 5-bit bucket
constexpr int kMaxGroupChannels = 1024;                // G * D: the group's int64 sums fit over the two lists
static_assert(3 * kMaxGroupChannels * 8 <= 2 * 4 * kListCap, "sums copy over the lists");
static_assert(kChgParts % 32 == 0, "change ranges are scanned 32 lanes wide");

// Calls f(i, byte) for the bytes i in [t0, t1) of p whose value v has
// (v & keep) == want: 16-byte loads in the aligned middle, four bytes per
// word tested at once (a byte of (w & mask) ^ want is zero exactly for a
// member).
template <class F>
__device__ __forceinline__ void for_matching_bytes(const uint8_t* p, int64_t t0, int64_t t1, uint32_t keep,
                                                   uint32_t want, F&& f) {
    const uint32_t mask4 = keep * 0x01010101u, want4 = want * 0x01010101u;
    auto one = [&](int64_t n, uint32_t v) {
        if ((v & keep) == want) f(n, v);
    };
    const uint8_t* p0 = p + t0;
    int64_t pre = (int64_t)((16u - ((uint32_t)(uintptr_t)p0 & 15u)) & 15u);
    if (pre > t1 - t0) pre = t1 - t0;
    const int64_t body = (t1 - t0 - pre) >> 4;
    for (int64_t i = threadIdx.x; i < pre; i += kUpdThreads) one(t0 + i, p0[i]);
    const uint4* pb = reinterpret_cast<const uint4*>(p0 + pre);
    for (int64_t i0 = threadIdx.x; i0 < body; i0 += 4 * kUpdThreads) {
        uint4 v[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
            if (i0 + r * kUpdThreads < body) v[r] = __ldg(pb + i0 + r * kUpdThreads);
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            if (i0 + r * kUpdThreads >= body) break;
            const uint32_t w[4] = {v[r].x, v[r].y, v[r].z, v[r].w};
            uint32_t hit[4], any = 0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t t = (w[q] & mask4) ^ want4;            // zero byte <=> member
                hit[q] = (t - 0x01010101u) & ~t & 0x80808080u;        // nonzero iff t has a zero byte
                any |= hit[q];
            }
            if (any) {
                const int64_t n = t0 + pre + 16 * (i0 + r * kUpdThreads);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (hit[q])
#pragma unroll
                        for (int j = 0; j < 4; ++j) one(n + 4 * q + j, (w[q] >> (8 * j)) & 0xFFu);
            }
        }
    }
    for (int64_t n = t0 + pre + 16 * body + threadIdx.x; n < t1; n += kUpdThreads) one(n, p[n]);
}

// 0x80 in every byte of t that is zero, nothing in the others (exact, unlike
// the borrow-based test, which can also mark a 0x01 byte above a zero one).
__device__ __forceinline__ uint32_t zero_bytes(uint32_t t) {
    return ~(((t & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | t | 0x7F7F7F7Fu);
}

// All 32 lanes: lane i reserves m_i consecutive slots of *counter; returns
// its first slot (one shared atomic per warp instead of one per entry).
__device__ __forceinline__ int warp_reserve(int m, int* counter, int lane) {
    int inc = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += u;
    }
    int base = 0;
    if (lane == 31 && inc) base = atomicAdd(counter, inc);
    base = __shfl_sync(0xffffffffu, base, 31);
    return base + inc - m;
}

// Shared memory: the sorted list and the arrival-order list (int[kListCap]
// each), then the window sums of the group split at bit 15 (int lo, hi
// [G][3][D], the layout of the stored sums), which the 128-bit sums reuse.
__host__ __device__ inline size_t update_smem(int D, int lg) {
    return 2 * sizeof(int) * kListCap + 2 * sizeof(int) * ((size_t)3 * D << lg);
}

template <int D>
__global__ void __launch_bounds__(kUpdThreads, 3) kmeans_update_kernel(UpdateArgs a) {
    constexpr int LPR = D / 8, RPW = 32 / LPR, UNITS = (kUpdThreads / 32) * RPW;
    extern __shared__ __align__(16) unsigned char upd_smem[];
    const int lg = a.group_log2, G = 1 << lg, GD3 = 3 * (D << lg);
    int* list = reinterpret_cast<int*>(upd_smem);
    int* raw = list + kListCap;
    int* lo = raw + kListCap;
    int* hi = lo + GD3;
    __shared__ int cnt[kMaxGroup], dcnt[kMaxGroup], bcnt[2 * kMaxGroup], off[2 * kMaxGroup + 1], cur[2 * kMaxGroup];
    __shared__ int touched[kMaxGroup];
    __shared__ int n_raw, big, ibig;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y, c0 = blockIdx.x << lg;
    const int ng = min(G, a.C - c0);
    const int64_t N = a.n_tokens;
    const uint8_t* idh = a.ids + (int64_t)h * a.cap + a.tok_offset;
    const uint16_t* xh = a.x + (int64_t)h * a.head_stride;
    long long* ks = a.ksum + ((int64_t)h * a.C + c0) * 3 * D;        // [k][w][d], k < ng
    int* kc = a.kcount + (int64_t)h * a.C + c0;
    int* kb = a.kbig + (int64_t)h * a.C + blockIdx.x;
    const uint32_t keep = (0xFFu << lg) & 0xFFu;

    // offsets of nb buckets from their counts c[] (cur becomes the cursors)
    auto set_offsets = [&](const int* c, int nb) {
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int b = 0; b < nb; ++b) {
                const int v = c[b];
                off[b] = run;
                cur[b] = run;
                run += v;
            }
            for (int b = nb; b <= 2 * kMaxGroup; ++b) off[b] = run;
        }
        __syncthreads();
    };
    // bucket counts of the arrival-order list of n_raw <= kListCap entries
    // (n << 5 | bucket) into c[nb]; lanes on the same bucket add together
    auto count_raw = [&](int* c, int nb) {
        if (tid < nb) c[tid] = 0;
        __syncthreads();
        const int n = n_raw;
        for (int i0 = warp * 32; i0 < n; i0 += kUpdThreads) {
            const int i = i0 + lane;
            const int b = i < n ? (raw[i] & 31) : -1;
            const unsigned mm = __match_any_sync(0xffffffffu, b);
            if (b >= 0 && lane == __ffs(mm) - 1) atomicAdd(&c[b], __popc(mm));
        }
        __syncthreads();
    };
    // that list, sorted by bucket (ranks within a warp from __match_any_sync)
    auto sort_raw = [&](const int* c, int nb) {
        set_offsets(c, nb);
        const int n = n_raw;
        const unsigned lt = (1u << lane) - 1u;
        for (int i0 = warp * 32; i0 < n; i0 += kUpdThreads) {
            const int i = i0 + lane;
            const int v = i < n ? raw[i] : -1;
            const int b = v >= 0 ? (v & 31) : -1;
            const unsigned mm = __match_any_sync(0xffffffffu, b);
            const int leader = __ffs(mm) - 1;
            int base = 0;
            if (b >= 0 && lane == leader) base = atomicAdd(&cur[b], __popc(mm));
            base = __shfl_sync(0xffffffffu, base, leader);
            if (b >= 0) list[base + __popc(mm & lt)] = v >> 5;
        }
        __syncthreads();
    };
    auto clear_sums = [&]() {
        for (int i = tid; i < GD3; i += kUpdThreads) lo[i] = hi[i] = 0;
    };

    // window sums of the listed rows into lo/hi: unit u takes the contiguous
    // run [u T / UNITS, (u + 1) T / UNITS) of the list.  In an incremental
    // list bucket 2k adds rows to cluster k and bucket 2k + 1 subtracts them.
    float amax = 0.0f;
    auto sum_list = [&](bool signed_buckets) {
        const int T = off[2 * kMaxGroup];
        const int unit = warp * RPW + lane / LPR, sub = lane % LPR;
        const int pb = (int)((int64_t)unit * T / UNITS), pe = (int)((int64_t)(unit + 1) * T / UNITS);
        if (pb >= pe) return;
        const uint16_t* xs = xh + sub * 8;
        int w1[8], w2[8], w3[8];
#pragma unroll
        for (int d = 0; d < 8; ++d) w1[d] = w2[d] = w3[d] = 0;
        int b = 0, terms = 0;
        while (pb >= off[b + 1]) ++b;
        auto flush = [&]() {
            const int k = signed_buckets ? b >> 1 : b;
            const bool neg = signed_buckets && (b & 1);
            int* l0 = lo + k * 3 * D + 8 * sub;
            int* h0 = hi + k * 3 * D + 8 * sub;
#pragma unroll
            for (int d = 0; d < 8; ++d) {
                const int v1 = neg ? -w1[d] : w1[d], v2 = neg ? -w2[d] : w2[d], v3 = neg ? -w3[d] : w3[d];
                atomicAdd(l0 + d, v1 & 0x7FFF);         atomicAdd(h0 + d, v1 >> 15);
                atomicAdd(l0 + D + d, v2 & 0x7FFF);     atomicAdd(h0 + D + d, v2 >> 15);
                atomicAdd(l0 + 2 * D + d, v3 & 0x7FFF); atomicAdd(h0 + 2 * D + d, v3 >> 15);
                w1[d] = w2[d] = w3[d] = 0;
            }
            terms = 0;
        };
        for (int p0 = pb; p0 < pe; p0 += kSumRows) {
            // rows two rounds ahead are asked into L2 now, so that their loads
            // there meet L2 latency rather than DRAM's (no registers held)
#pragma unroll
            for (int j = 0; j < kSumRows; ++j) {
                const int pf = p0 + kSumAhead + j;
                if (pf < pe)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(xs + (int64_t)list[pf] * a.token_stride));
            }
            uint4 v[kSumRows];
#pragma unroll
            for (int j = 0; j < kSumRows; ++j)
                if (p0 + j < pe) v[j] = ldg_nc_v4(xs + (int64_t)list[p0 + j] * a.token_stride);
#pragma unroll
            for (int j = 0; j < kSumRows; ++j) {
                const int p = p0 + j;
                if (p >= pe) break;
                if (p >= off[b + 1] || terms == kFlushTerms) {
                    if (terms) flush();
                    while (p >= off[b + 1]) ++b;
                }
                const uint32_t wv[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float l = bf16_lo(wv[q]), u = bf16_hi(wv[q]);
                    amax = fmax3(amax, fabsf(l), fabsf(u));
                    window_add2(make_float2(l, u), w1 + 2 * q, w2 + 2 * q, w3 + 2 * q);
                }
                ++terms;
            }
        }
        if (terms) flush();
    };
    // lo/hi into the stored sums (= when first, else +=), then cleared
    // ... and a copy in shared memory (ksm, over the lists) for the means;
    // the stored sums are read four at a time so that their loads overlap
    long long* ksm = reinterpret_cast<long long*>(list);
    constexpr int kFoldPer = 3 * kMaxGroupChannels / kUpdThreads;       // entries per thread, at most
    auto fold = [&](bool first) {
        __syncthreads();
        const int n3 = ng * 3 * D;
        long long old[kFoldPer];
#pragma unroll
        for (int r = 0; r < kFoldPer; ++r) {
            const int i = tid + r * kUpdThreads;
            old[r] = (!first && i < n3) ? ks[i] : 0;
        }
#pragma unroll
        for (int r = 0; r < kFoldPer; ++r) {
            const int i = tid + r * kUpdThreads;
            if (i < n3) {
                const long long v = old[r] + (long long)hi[i] * 32768 + lo[i];
                ks[i] = v;
                ksm[i] = v;
                lo[i] = hi[i] = 0;
            }
        }
        __syncthreads();
    };
    auto mean_of = [&](int k, int d, bool from_lohi, int count) -> uint16_t {
        long long w[3];
#pragma unroll
        for (int q = 0; q < 3; ++q) {
            const int j = (k * 3 + q) * D + d;
            w[q] = from_lohi ? (long long)hi[j] * 32768 + lo[j] : ksm[j];
        }
        return mean_bf16_bits_fast(((i128)w[0] << 44) + ((i128)w[1] << 22) + (i128)w[2], (uint32_t)count);
    };
    uint16_t* ch = a.cent + ((int64_t)h * a.C + c0) * D;

    if (a.mode == kUpdIncremental && *kb == 0 && N < kPackLimit) {
        // The changes lie in the ranges chg_parts[h][p] = (start, count) of
        // the head's chg_tok / chg_on rows (stride chg_stride, a multiple of
        // 8; every start a multiple of 128), bytes 2i and 2i + 1 of chg_on
        // being the old and the new id of change i.  The ranges' 16-byte
        // chunks are numbered consecutively so that all threads share one scan.
        __shared__ int2 parts[kChgParts];
        __shared__ int pchunk[kChgParts + 1];
        const uint8_t* onb = reinterpret_cast<const uint8_t*>(a.chg_on + (int64_t)h * a.chg_stride);
        const int* tk = a.chg_tok + (int64_t)h * a.chg_stride;
        for (int p = tid; p < kChgParts; p += kUpdThreads) parts[p] = a.chg_parts[(int64_t)h * kChgParts + p];
        if (tid < kMaxGroup) dcnt[tid] = touched[tid] = 0;
        if (tid < 2 * kMaxGroup) bcnt[tid] = 0;
        if (tid == 0) { ibig = 0; n_raw = 0; }
        clear_sums();
        __syncthreads();
        if (warp == 0) {
            // exclusive prefix of the ranges' chunk counts, kChgParts / 32 per lane
            constexpr int PL = kChgParts / 32;
            int c[PL], sum = 0;
#pragma unroll
            for (int r = 0; r < PL; ++r) {
                c[r] = (2 * parts[lane * PL + r].y + 15) >> 4;
                sum += c[r];
            }
            int inc = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += u;
            }
            int run = inc - sum;
#pragma unroll
            for (int r = 0; r < PL; ++r) {
                pchunk[lane * PL + r] = run;
                run += c[r];
            }
            if (lane == 31) pchunk[kChgParts] = run;
        }
        __syncthreads();
        const int n_chunks = pchunk[kChgParts];
        // the chunk q of the changes: its first byte and the end of its range
        auto locate = [&](int q, int64_t& at, int64_t& lim) {
            int lo_p = 0, hi_p = kChgParts - 1;                    // the range holding chunk q
            while (lo_p < hi_p) {
                const int mid = (lo_p + hi_p + 1) >> 1;
                if (pchunk[mid] <= q) lo_p = mid; else hi_p = mid - 1;
            }
            at = 2 * (int64_t)parts[lo_p].x + 16 * (int64_t)(q - pchunk[lo_p]);
            lim = 2 * ((int64_t)parts[lo_p].x + parts[lo_p].y);
        };
        // the entry of change byte j (old id at even j, new at odd)
        auto entry = [&](int64_t j, uint32_t v) {
            const int k = (int)v - c0, leaving = (int)(~j & 1);
            return (tk[j >> 1] << 5) | (2 * k + leaving);
        };
        // one scan of all chunks: every member byte appended to raw while it
        // has room (n_raw counts them all), one shared atomic per warp and round
        {
            const uint32_t mask4 = keep * 0x01010101u, want4 = (uint32_t)c0 * 0x01010101u;
            for (int q0 = warp * 32 * kScanR; q0 < n_chunks; q0 += kScanR * kUpdThreads) {
                uint32_t w[kScanR][4], z[kScanR][4];
                int64_t at[kScanR];
                int m = 0;
#pragma unroll
                for (int r = 0; r < kScanR; ++r) {
                    const int q = q0 + 32 * r + lane;
                    int64_t lim = 0;
                    at[r] = 0;
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (q < n_chunks) {
                        locate(q, at[r], lim);
                        v = __ldg(reinterpret_cast<const uint4*>(onb + at[r]));
                    }
                    w[r][0] = v.x; w[r][1] = v.y; w[r][2] = v.z; w[r][3] = v.w;
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) {
                        const int64_t rem = q < n_chunks ? lim - at[r] - 4 * qq : 0;   // valid bytes of the word
                        uint32_t zz = zero_bytes((w[r][qq] & mask4) ^ want4);
                        if (rem <= 0) zz = 0;
                        else if (rem < 4) zz &= (1u << (8 * rem)) - 1u;
                        z[r][qq] = zz;
                        m += __popc(zz);
                    }
                }
                int slot = warp_reserve(m, &n_raw, lane);
#pragma unroll
                for (int r = 0; r < kScanR; ++r)
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq)
                        for (uint32_t zz = z[r][qq]; zz; zz &= zz - 1u) {
                            const int byte = (__ffs(zz) - 1) >> 3;
                            if (slot < kListCap) raw[slot] = entry(at[r] + 4 * qq + byte, (w[r][qq] >> (8 * byte)) & 0xFFu);
                            ++slot;
                        }
            }
        }
        __syncthreads();
        if (n_raw <= kListCap) {
            count_raw(bcnt, 2 * G);
            if (tid < G) {
                dcnt[tid] = bcnt[2 * tid] - bcnt[2 * tid + 1];
                touched[tid] = (bcnt[2 * tid] | bcnt[2 * tid + 1]) != 0;
            }
            sort_raw(bcnt, 2 * G);
            sum_list(true);
            fold(false);
        } else {
            // more rows than the list holds: runs of chunks holding at most
            // kListCap / 2 changes, each scanned again entry by entry
            for (int cb = 0; cb < n_chunks; cb += kListCap / 16) {
                const int ce = min(n_chunks, cb + kListCap / 16);
                __syncthreads();
                if (tid < 2 * kMaxGroup) bcnt[tid] = 0;
                if (tid == 0) n_raw = 0;
                __syncthreads();
                for (int q = cb + tid; q < ce; q += kUpdThreads) {
                    int64_t at, lim;
                    locate(q, at, lim);
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(onb + at));
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    for (int b = 0; b < 16 && at + b < lim; ++b) {
                        const uint32_t byte = (w[b >> 2] >> (8 * (b & 3))) & 0xFFu;
                        if ((byte & keep) == (uint32_t)c0) {
                            const int e = entry(at + b, byte);
                            atomicAdd(&bcnt[e & 31], 1);
                            raw[atomicAdd(&n_raw, 1)] = e;
                        }
                    }
                }
                __syncthreads();
                if (tid < G) {
                    dcnt[tid] += bcnt[2 * tid] - bcnt[2 * tid + 1];
                    if (bcnt[2 * tid] | bcnt[2 * tid + 1]) touched[tid] = 1;
                }
                sort_raw(bcnt, 2 * G);
                sum_list(true);
                fold(false);
            }
        }
        if (!(amax < kWinMax)) ibig = 1;
        __syncthreads();
        if (!ibig) {
            if (tid < ng) {
                dcnt[tid] += kc[tid];                  // the new counts
                kc[tid] = dcnt[tid];
            }
            __syncthreads();
            // clusters that a change touched are rounded again (a token leaving
            // and another arriving may leave the count as it was); an emptied
            // one keeps its centroid
            for (int i = tid; i < ng * D; i += kUpdThreads) {
                const int k = i / D, d = i % D;
                if (touched[k] && dcnt[k] != 0) ch[i] = mean_of(k, d, false, dcnt[k]);
            }
            return;
        }
        // a changed row holds a value >= 2^14: the full update below redoes the group
        __syncthreads();
    }

    // ---- full update
    if (tid < kMaxGroup) cnt[tid] = 0;
    if (tid == 0) { n_raw = 0; big = 0; }
    clear_sums();
    __syncthreads();
    const bool packable = N < kPackLimit;
    if (packable) {
        // one scan of the ids: every member appended to raw while it has room
        // (n_raw counts them all), one shared atomic per warp and round; the
        // unaligned head and tail (at most 30 bytes) one atomic per member
        const uint32_t mask4 = keep * 0x01010101u, want4 = (uint32_t)c0 * 0x01010101u;
        int64_t pre = (int64_t)((16u - ((uint32_t)(uintptr_t)idh & 15u)) & 15u);
        if (pre > N) pre = N;
        const int64_t body = (N - pre) >> 4;
        const uint4* pb = reinterpret_cast<const uint4*>(idh + pre);
        auto put1 = [&](int64_t n, uint32_t v) {
            if ((v & keep) == (uint32_t)c0) {
                const int pos = atomicAdd(&n_raw, 1);
                if (pos < kListCap) raw[pos] = ((int)n << 5) | ((int)v - c0);
            }
        };
        for (int64_t i = tid; i < pre; i += kUpdThreads) put1(i, idh[i]);
        for (int64_t n = pre + 16 * body + tid; n < N; n += kUpdThreads) put1(n, idh[n]);
        for (int64_t i0 = (int64_t)warp * 32 * kScanR; i0 < body; i0 += kScanR * kUpdThreads) {
            uint32_t w[kScanR][4], z[kScanR][4];
            int m = 0;
#pragma unroll
            for (int r = 0; r < kScanR; ++r) {
                const int64_t i = i0 + 32 * r + lane;
                const uint4 v = i < body ? __ldg(pb + i) : make_uint4(0, 0, 0, 0);
                w[r][0] = v.x; w[r][1] = v.y; w[r][2] = v.z; w[r][3] = v.w;
#pragma unroll
                for (int qq = 0; qq < 4; ++qq) {
                    const uint32_t zz = i < body ? zero_bytes((w[r][qq] & mask4) ^ want4) : 0u;
                    z[r][qq] = zz;
                    m += __popc(zz);
                }
            }
            int slot = warp_reserve(m, &n_raw, lane);
#pragma unroll
            for (int r = 0; r < kScanR; ++r)
#pragma unroll
                for (int qq = 0; qq < 4; ++qq)
                    for (uint32_t zz = z[r][qq]; zz; zz &= zz - 1u) {
                        const int byte = (__ffs(zz) - 1) >> 3;
                        const int64_t n = pre + 16 * (i0 + 32 * r + lane) + 4 * qq + byte;
                        if (slot < kListCap) raw[slot] = ((int)n << 5) | ((int)((w[r][qq] >> (8 * byte)) & 0xFFu) - c0);
                        ++slot;
                    }
        }
    }
    __syncthreads();
    const bool one = packable && n_raw <= kListCap;
    amax = 0.0f;
    if (one) {
        count_raw(cnt, G);
        sort_raw(cnt, G);
        sum_list(false);
        __syncthreads();
        for (int i = tid; i < ng * 3 * D; i += kUpdThreads) ks[i] = (long long)hi[i] * 32768 + lo[i];
    } else {
        // more members than the list holds: token spans sized from the
        // member count to fill about three quarters of it (a span that still
        // overflows is halved; kListCap tokens never can)
        int64_t span = kListCap;
        if (packable && n_raw > 0) {
            const int64_t fit = (int64_t)((double)(3 * kListCap / 4) * (double)N / (double)n_raw);
            if (fit > span) span = fit;
        }
        bool first = true;
        for (int64_t t0 = 0; t0 < N;) {
            const int64_t t1 = min(N, t0 + span);
            if (tid < 2 * kMaxGroup) bcnt[tid] = 0;
            __syncthreads();
            for_matching_bytes(idh, t0, t1, keep, (uint32_t)c0, [&](int64_t, uint32_t v) { atomicAdd(&bcnt[(int)v - c0], 1); });
            __syncthreads();
            int members = 0;
            for (int b = 0; b < G; ++b) members += bcnt[b];
            __syncthreads();               // every thread has read the counts (the same decision) before they change
            if (members > kListCap) {
                span = span / 2 > kListCap ? span / 2 : kListCap;
                continue;
            }
            if (tid < G) cnt[tid] += bcnt[tid];
            set_offsets(bcnt, G);
            for_matching_bytes(idh, t0, t1, keep, (uint32_t)c0,
                               [&](int64_t n, uint32_t v) { list[atomicAdd(&cur[(int)v - c0], 1)] = (int)n; });
            __syncthreads();
            sum_list(false);
            fold(first);
            first = false;
            t0 = t1;
        }
    }
    if (!(amax < kWinMax)) big = 1;
    if (tid < ng) kc[tid] = cnt[tid];
    __syncthreads();
    if (tid == 0) *kb = big;
    if (!big) {
        for (int i = tid; i < ng * D; i += kUpdThreads) {
            const int k = i / D, d = i % D;
            if (cnt[k] != 0) ch[i] = mean_of(k, d, one, cnt[k]);   // an empty cluster keeps its centroid
        }
        return;
    }
    // a value outside the first window: sum the group again with 128-bit
    // integers, one thread per (slot, channel)
    i128* s128 = reinterpret_cast<i128*>(lo);
    for (int i = tid; i < G * D; i += kUpdThreads) s128[i] = 0;
    __syncthreads();
    auto exact_list = [&]() {
        for (int i = tid; i < ng * D; i += kUpdThreads) {
            const int k = i / D, d = i % D;
            i128 t = 0;
            for (int p = off[k]; p < off[k + 1]; ++p) t += bf16_to_i128_units(xh[(int64_t)list[p] * a.token_stride + d]);
            s128[i] += t;
        }
        __syncthreads();
    };
    if (one) {
        exact_list();                                // the sorted list is still in place
    } else {
        for (int64_t t0 = 0; t0 < N; t0 += kListCap) {
            const int64_t t1 = min(N, t0 + kListCap);
            if (tid < 2 * kMaxGroup) bcnt[tid] = 0;
            __syncthreads();
            for_matching_bytes(idh, t0, t1, keep, (uint32_t)c0, [&](int64_t, uint32_t v) { atomicAdd(&bcnt[(int)v - c0], 1); });
            set_offsets(bcnt, G);
            for_matching_bytes(idh, t0, t1, keep, (uint32_t)c0,
                               [&](int64_t n, uint32_t v) { list[atomicAdd(&cur[(int)v - c0], 1)] = (int)n; });
            __syncthreads();
            exact_list();
        }
    }
    for (int i = tid; i < ng * D; i += kUpdThreads) {
        const int k = i / D;
        if (cnt[k] != 0) ch[i] = mean_bf16_bits_fast(s128[i], (uint32_t)cnt[k]);
    }
}

// Clusters per CTA: the largest power of two up to kMaxGroup that still
// gives two CTAs per SM and, on average, fills at most three quarters of the
// list.  Every CTA scans all N ids of its head, so larger groups scan less in
// all (H * C / G * N bytes).
int update_group_log2(int D, int H, int C, int64_t N) {
    int lg = 0;
    while ((1 << (lg + 1)) <= kMaxGroup && (int64_t)H * ((C + (2 << lg) - 1) >> (lg + 1)) >= 2 * 148 &&
           4 * N * (2 << lg) <= 3 * (int64_t)C * kListCap && (D << (lg + 1)) <= kMaxGroupChannels)
        ++lg;
    return lg;
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
cudaError_t update_d(const UpdateArgs& a0, cudaStream_t s) {
    if (a0.n_tokens == 0) return cudaSuccess;
    UpdateArgs a = a0;
    if (a.group_log2 < 0) a.group_log2 = update_group_log2(D, a.H, a.C, a.n_tokens);
    if ((1 << a.group_log2) > kMaxGroup || (D << a.group_log2) > kMaxGroupChannels) return cudaErrorInvalidValue;
    const size_t smem = update_smem(D, a.group_log2);
    cudaError_t e = cudaFuncSetAttribute(kmeans_update_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.C + (1 << a.group_log2) - 1) >> a.group_log2), (unsigned)a.H);
    kmeans_update_kernel<D><<<grid, kUpdThreads, smem, s>>>(a);
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

cudaError_t launch_assign(int D, int H, const AssignArgs& a, cudaStream_t s, bool* recorded) {
    bool launched = false;
    const cudaError_t e = launch_assign_tc(D, H, a, &launched, s);
    if (recorded) *recorded = launched && a.chg_parts != nullptr;
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
