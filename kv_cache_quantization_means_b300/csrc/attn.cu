// Attention whose keys and values are read straight from the compressed cache
// (Quant VideoGen explainer, sec. 3, key contributions: fused dequantisation
// kernels; the 33-method Self-Forcing KV-cache study, abstract: integrations
// that rebuild full BF16 K/V buffers around attention lose the memory that
// compression saved).  No bf16 K/V buffer is written: each 64-key tile is
// decoded into shared memory, used, and overwritten by the next.
//
// Per head h and query i (non-causal; every query sees keys 0 .. n_keys-1):
//   s_n = scale * <q_i, k_hat_n>,  o_i = sum_n exp(s_n) v_hat_n / sum_n exp(s_n),
// where k_hat, v_hat are the bf16 reconstructions that the decoder writes,
// bit for bit: x_hat = bf16(((c[id] + d_1) + d_2) ...), d_s = q_s*s_s + z_s in
// fp32 (Quant VideoGen explainer, Sommario tecnico sec. 2B item 3).  The
// decode below calls the same per-16-channel routines as the decode kernel.
//
// One CTA = 64 queries of one head, four warps of 16 query rows.  Per key tile:
//  1. all 128 threads decode 64 rows of K and of V, 16 channels per item,
//     into padded shared memory (row stride D + 8 bf16: conflict-free
//     ldmatrix); with at most two code and meta words per item, the raw
//     words of the next tile are loaded into registers while this tile's
//     products run, and decoded after them;
//  2. each warp computes S = Q K^T (16 x 64) with bf16 mma.sync m16n8k16,
//     fp32 accumulation, Q held in registers for the whole kernel;
//  3. online softmax in fp32 with base-2 exponentials (scale * log2 e folded
//     into one multiply), the running maximum and sum per query row;
//  4. O += P V with P rounded to bf16 (the score fragment is the A fragment
//     of the second product) and V read by transposing ldmatrix.
// The output is O / l in fp32.
#include <math.h>

#include "attn.h"
#include "common.cuh"
#include "prq16.cuh"

namespace qvg {

namespace {

constexpr int kAttnWarps = 4;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kQTile = 16 * kAttnWarps;   // queries per CTA
constexpr int kKTile = 64;                // keys per tile

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

// d += a (16 x 16 bf16, row) * b (16 x 8 bf16, col), fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// PF: the next key tile's ids, code words and meta words are loaded into
// registers before the current tile's products, so that their latency is
// spent under the tensor work (needs S * B / 2 <= 2 code words and S <= 2
// meta words per item); otherwise each tile is loaded and decoded in turn.
template <int D, int B, bool PF>
__global__ void __launch_bounds__(kAttnThreads) attention_decode_kernel(AttnArgs a) {
    constexpr int LD = D + 8;             // bf16 row stride in shared memory
    constexpr int CPR = D / 16;           // 16-channel items per row
    constexpr int ITEMS = 2 * kKTile * CPR;
    constexpr int IPT = ITEMS / kAttnThreads;
    constexpr int WPT = B / 2;            // code words per item and stage
    constexpr int WPR = D * B / 32;       // code words per row and stage
    static_assert(ITEMS % kAttnThreads == 0, "whole items per thread");
    __shared__ __align__(16) uint16_t ks[kKTile * LD];
    __shared__ __align__(16) uint16_t vs[kKTile * LD];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y;
    const int64_t q0 = (int64_t)blockIdx.x * kQTile;

    // queries of this CTA, staged through ks (zero rows past n_queries)
    for (int v = tid; v < kQTile * (D / 8); v += kAttnThreads) {
        const int r = v / (D / 8), c = v % (D / 8);
        uint4 val = make_uint4(0, 0, 0, 0);
        if (q0 + r < a.n_queries) val = ldg_nc_v4(a.q + h * a.q_head_stride + (q0 + r) * a.q_token_stride + c * 8);
        *reinterpret_cast<uint4*>(ks + r * LD + c * 8) = val;
    }
    __syncthreads();
    uint32_t qf[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        ldsm_x4(smem_addr(ks + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8), qf[kk]);
    __syncthreads();

    float o[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r) o[i][r] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY};   // running maximum (base-2 units) of rows g, g + 8
    float l[2] = {0.0f, 0.0f};             // this thread's part of the running sums
    const int qd = lane & 3;
    const int brow = (lane & 7) + ((lane >> 4) << 3), bk = ((lane >> 3) & 1) * 8;
    const int64_t stage_rows = (int64_t)a.H * a.cap;

    // item k of this thread: v = tid + k * kAttnThreads; K for v < ITEMS / 2, V after
    uint32_t pid[IPT], pcode[IPT][2], pmeta[IPT][2];
    uint32_t pvalid = 0;
    const int mpr = D / a.G;

    // raw words of the tile starting at n (PF)
    auto prefetch = [&](int64_t n) {
        pvalid = 0;
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const int v = tid + k * kAttnThreads;
            const bool is_v = v >= ITEMS / 2;
            const int rem = is_v ? v - ITEMS / 2 : v;
            const int r = rem / CPR, c = rem % CPR;
            pid[k] = 0;
            pcode[k][0] = pcode[k][1] = 0;
            pmeta[k][0] = pmeta[k][1] = 0;
            if (n + r < a.n_keys) {
                pvalid |= 1u << k;
                const int64_t row = (int64_t)h * a.cap + n + r;
                const uint32_t* codes = is_v ? a.v_codes : a.k_codes;
                const uint32_t* meta = is_v ? a.v_meta : a.k_meta;
                if (a.C > 0) pid[k] = (is_v ? a.v_ids : a.k_ids)[row];
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2) {
                    if (s2 >= a.S) continue;
                    const int64_t srow = (int64_t)s2 * stage_rows + row;
                    if constexpr (B == 2) pcode[k][s2] = __ldg(codes + srow * WPR + c * WPT);
                    else if (s2 == 0) {
                        pcode[k][0] = __ldg(codes + srow * WPR + c * WPT);
                        pcode[k][1] = __ldg(codes + srow * WPR + c * WPT + 1);
                    }
                    pmeta[k][s2] = __ldg(meta + srow * mpr + (c * 16) / a.G);
                }
            }
        }
    };
    // centroid rows, dequantisation and the stores to shared memory (PF)
    auto finish = [&]() {
#pragma unroll
        for (int k = 0; k < IPT; ++k) {
            const int v = tid + k * kAttnThreads;
            const bool is_v = v >= ITEMS / 2;
            const int rem = is_v ? v - ITEMS / 2 : v;
            const int r = rem / CPR, c = rem % CPR;
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
            if (pvalid & (1u << k)) {
                float acc[16];
                if (a.C > 0) {
                    const uint16_t* cr = (is_v ? a.v_cent : a.k_cent) +
                                         ((int64_t)h * a.C + min((int)pid[k], a.C - 1)) * D + c * 16;
                    unpack16(__ldg(reinterpret_cast<const uint4*>(cr)), __ldg(reinterpret_cast<const uint4*>(cr + 8)),
                             acc);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
                }
                if constexpr (B == 2) {
#pragma unroll
                    for (int s2 = 0; s2 < 2; ++s2)
                        if (s2 < a.S) dequant_add16(acc, pcode[k][s2], pmeta[k][s2]);
                } else {
                    dequant_add8x4(acc, pcode[k][0], pmeta[k][0]);
                    dequant_add8x4(acc + 8, pcode[k][1], pmeta[k][0]);
                }
                pack16_bf16(acc, o0, o1);
            }
            uint16_t* dst = (is_v ? vs : ks) + r * LD + c * 16;
            *reinterpret_cast<uint4*>(dst) = o0;
            *reinterpret_cast<uint4*>(dst + 8) = o1;
        }
    };
    // load and decode the tile starting at n in one pass (not PF)
    auto decode_tile = [&](int64_t n) {
#pragma unroll 2
        for (int v = tid; v < ITEMS; v += kAttnThreads) {
            const bool is_v = v >= ITEMS / 2;
            const int rem = is_v ? v - ITEMS / 2 : v;
            const int r = rem / CPR, c = rem % CPR;
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
            if (n + r < a.n_keys) {
                const int64_t row = (int64_t)h * a.cap + n + r;
                if (is_v)
                    decode_chunk<D, B>(a.v_codes, a.v_meta, a.v_ids, a.v_cent, row, h, c, stage_rows, a.C, a.S, a.G,
                                       o0, o1);
                else
                    decode_chunk<D, B>(a.k_codes, a.k_meta, a.k_ids, a.k_cent, row, h, c, stage_rows, a.C, a.S, a.G,
                                       o0, o1);
            }
            uint16_t* dst = (is_v ? vs : ks) + r * LD + c * 16;
            *reinterpret_cast<uint4*>(dst) = o0;
            *reinterpret_cast<uint4*>(dst + 8) = o1;
        }
    };

    // 1. the first tile of K (items 0 .. ITEMS/2-1) and V (the rest)
    if constexpr (PF) {
        prefetch(0);
        finish();
    } else {
        decode_tile(0);
    }
    __syncthreads();

    for (int64_t n0 = 0; n0 < a.n_keys; n0 += kKTile) {
        const int64_t next = n0 + kKTile;
        if constexpr (PF) {
            if (next < a.n_keys) prefetch(next);   // in flight during the products below
        }

        // 2. S = Q K^T: n-tile j holds keys n0 + 8j .. n0 + 8j + 7
        float sc[kKTile / 8][4];
#pragma unroll
        for (int j = 0; j < kKTile / 8; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) sc[j][r] = 0.0f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
            for (int np = 0; np < kKTile / 16; ++np) {
                uint32_t b[4];
                ldsm_x4(smem_addr(ks + (np * 16 + brow) * LD + kk * 16 + bk), b);
                mma_bf16(sc[2 * np], qf[kk], b[0], b[1]);
                mma_bf16(sc[2 * np + 1], qf[kk], b[2], b[3]);
            }
        }

        // 3. online softmax; element r of a fragment is row g + 8*(r >> 1),
        //    key n0 + 8j + 2*qd + (r & 1)
        float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < kKTile / 8; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int64_t key = n0 + 8 * j + 2 * qd + (r & 1);
                const float v = key < a.n_keys ? sc[j][r] * a.scale_log2 : -INFINITY;
                sc[j][r] = v;
                tmax[r >> 1] = fmaxf(tmax[r >> 1], v);
            }
        float corr[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 1));
            tmax[i] = fmaxf(tmax[i], __shfl_xor_sync(0xffffffffu, tmax[i], 2));
            // the tile holds at least one key, so the new maximum is finite
            const float mn = fmaxf(m[i], tmax[i]);
            corr[i] = exp2f(m[i] - mn);       // 0 on the first tile (m = -inf)
            m[i] = mn;
            l[i] *= corr[i];
        }
#pragma unroll
        for (int j = 0; j < kKTile / 8; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float p = exp2f(sc[j][r] - m[r >> 1]);
                sc[j][r] = p;
                l[r >> 1] += p;
            }
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            o[i][0] *= corr[0]; o[i][1] *= corr[0];
            o[i][2] *= corr[1]; o[i][3] *= corr[1];
        }

        // 4. O += P V: keys 16kk .. 16kk+15 of the tile are n-tiles 2kk, 2kk+1
#pragma unroll
        for (int kk = 0; kk < kKTile / 16; ++kk) {
            uint32_t pa[4];
            pa[0] = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
            pa[1] = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
            pa[2] = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
            pa[3] = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {
                uint32_t b[4];
                ldsm_x4_trans(smem_addr(vs + (kk * 16 + (lane & 15)) * LD + np * 16 + (lane >> 4) * 8), b);
                mma_bf16(o[2 * np], pa, b[0], b[1]);
                mma_bf16(o[2 * np + 1], pa, b[2], b[3]);
            }
        }
        __syncthreads();   // the next tile's decode overwrites ks / vs
        if (next < a.n_keys) {
            if constexpr (PF) finish();
            else decode_tile(next);
            __syncthreads();
        }
    }

    // O / l, rows g and g + 8 of the warp
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        l[i] += __shfl_xor_sync(0xffffffffu, l[i], 1);
        l[i] += __shfl_xor_sync(0xffffffffu, l[i], 2);
    }
    const float inv[2] = {1.0f / l[0], 1.0f / l[1]};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int64_t qi = q0 + warp * 16 + (lane >> 2) + 8 * half;
        if (qi >= a.n_queries) continue;
        float* orow = a.out + h * a.out_head_stride + qi * a.out_token_stride;
#pragma unroll
        for (int i = 0; i < D / 8; ++i)
            *reinterpret_cast<float2*>(orow + 8 * i + 2 * qd) =
                make_float2(o[i][2 * half] * inv[half], o[i][2 * half + 1] * inv[half]);
    }
}

template <int D>
cudaError_t launch_d(const AttnArgs& a, cudaStream_t s) {
    dim3 grid((unsigned)((a.n_queries + kQTile - 1) / kQTile), (unsigned)a.H);
    if (a.bits == 2 && a.S <= 2) attention_decode_kernel<D, 2, true><<<grid, kAttnThreads, 0, s>>>(a);
    else if (a.bits == 2) attention_decode_kernel<D, 2, false><<<grid, kAttnThreads, 0, s>>>(a);
    else if (a.bits == 4 && a.S == 1) attention_decode_kernel<D, 4, true><<<grid, kAttnThreads, 0, s>>>(a);
    else if (a.bits == 4) attention_decode_kernel<D, 4, false><<<grid, kAttnThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention_decode(int D, const AttnArgs& a, cudaStream_t s) {
    if (a.n_queries == 0) return cudaSuccess;
    if (D == 128) return launch_d<128>(a, s);
    if (D == 64) return launch_d<64>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace qvg
