// Progressive residual quantisation: encoder and decoder kernels.
//
// Quant VideoGen explainer, Sommario tecnico sec. 2A item 3 (subtract each
// token's centroid) and sec. 2B items 1-3 (re-quantise the residual stage by
// stage; decode = dequantise, sum the stages, add the centroid back).
//
// Both kernels are HBM-streaming: one lane owns 8 consecutive channels of a
// token row (one 16-byte bf16 vector), D/8 lanes cover a row, a warp covers
// 32/(D/8) rows per step and 16 rows in all.  Group min/max are warp-shuffle
// reductions over the G/8 lanes of a group; each lane packs its 8 2-bit codes
// into one 16-bit half of a code word, so a warp's code store is contiguous.
#include "common.cuh"
#include "kernels.h"

namespace qvg {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerWarp = 16;

template <int D>
struct RowMap {
    static constexpr int LPR = D / 8;           // lanes per row
    static constexpr int RPS = 32 / LPR;        // rows per warp step
    static constexpr int STEPS = kRowsPerWarp / RPS;
    static constexpr int ROWS_PER_CTA = kRowsPerWarp * (kThreads / 32);
};

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

template <int D, int G, bool HAS_C>
__global__ void __launch_bounds__(kThreads) prq_encode_kernel(EncodeArgs a) {
    using M = RowMap<D>;
    constexpr int LPG = G / 8;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % M::LPR, rw = lane / M::LPR;
    const int h = blockIdx.y;
    const int64_t row0 = (int64_t)blockIdx.x * M::ROWS_PER_CTA + (int64_t)warp * kRowsPerWarp + rw;

    const uint16_t* xh = a.x + (int64_t)h * a.head_stride + sub * 8;
    const uint8_t* idh = HAS_C ? a.ids + (int64_t)h * a.cap + a.tok_offset : nullptr;
    const uint16_t* ch = HAS_C ? a.cent + (int64_t)h * a.C * D + sub * 8 : nullptr;
    uint16_t* codes16 = reinterpret_cast<uint16_t*>(a.codes);

    // Register double-buffering of the next row's input.
    uint4 xv = make_uint4(0, 0, 0, 0);
    int idv = 0;
    if (row0 < a.n_tokens) {
        xv = ldg_nc_v4(xh + row0 * a.token_stride);
        if (HAS_C) idv = idh[row0];
    }
#pragma unroll 1
    for (int st = 0; st < M::STEPS; ++st) {
        const int64_t n = row0 + (int64_t)st * M::RPS;
        const bool valid = n < a.n_tokens;
        const int64_t nn = n + M::RPS;
        uint4 xnext = make_uint4(0, 0, 0, 0);
        int idnext = 0;
        if (st + 1 < M::STEPS && nn < a.n_tokens) {
            xnext = ldg_nc_v4(xh + nn * a.token_stride);
            if (HAS_C) idnext = idh[nn];
        }
        float r[8];
        unpack8(xv, r);
        if (HAS_C) {
            uint4 cv = valid ? __ldg(reinterpret_cast<const uint4*>(ch + (int64_t)min(idv, a.C - 1) * D))
                             : make_uint4(0, 0, 0, 0);
            float c[8];
            unpack8(cv, c);
#pragma unroll
            for (int i = 0; i < 8; ++i) r[i] = __fsub_rn(r[i], c[i]);
        }
        const int64_t rowoff = (int64_t)h * a.cap + a.tok_offset + n;
        for (int s = 0; s < a.S; ++s) {
            float mn = r[0], mx = r[0];
#pragma unroll
            for (int i = 1; i < 8; ++i) { mn = fminf(mn, r[i]); mx = fmaxf(mx, r[i]); }
#pragma unroll
            for (int off = 1; off < LPG; off <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            }
            // a zero extreme is taken as +0 so the stored bits do not depend
            // on the reduction order
            mn = __fadd_rn(mn, 0.0f);
            mx = __fadd_rn(mx, 0.0f);
            const GroupParams p = group_params(mn, mx);
            uint32_t code = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t q = quant_code(r[i], p);
                code |= q << (2 * i);
                if (s + 1 < a.S) r[i] = __fsub_rn(r[i], dequant(q, p.s, p.z));
            }
            if (valid) {
                const int64_t srow = (int64_t)s * a.H * a.cap + rowoff;
                codes16[srow * (D / 8) + sub] = (uint16_t)code;
                if (sub % LPG == 0) a.meta[srow * (D / G) + sub / LPG] = p.meta;
            }
        }
        xv = xnext;
        idv = idnext;
    }
}

template <int D, int G, bool HAS_C, bool VERSIONED>
__global__ void __launch_bounds__(kThreads) prq_decode_kernel(DecodeArgs a) {
    using M = RowMap<D>;
    constexpr int LPG = G / 8;
    extern __shared__ int64_t chunk_smem[];   // VERSIONED: offsets[n_chunks + 1], versions[n_chunks]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = lane % M::LPR, rw = lane / M::LPR;
    const int h = blockIdx.y;
    if (VERSIONED) {
        int32_t* vers = reinterpret_cast<int32_t*>(chunk_smem + a.n_chunks + 1);
        for (int i = threadIdx.x; i <= a.n_chunks; i += kThreads) chunk_smem[i] = a.chunk_offset[i];
        for (int i = threadIdx.x; i < a.n_chunks; i += kThreads) vers[i] = a.chunk_version[i];
        __syncthreads();
    }
    const int64_t n_rows = a.tok_end - a.tok_begin;
    const int64_t row0 = (int64_t)blockIdx.x * M::ROWS_PER_CTA + (int64_t)warp * kRowsPerWarp + rw;
    const uint16_t* codes16 = reinterpret_cast<const uint16_t*>(a.codes);
    const int64_t stage_stride = (int64_t)a.H * a.cap;
    const int64_t version_stride = (int64_t)a.H * a.C * D;

#pragma unroll 1
    for (int st = 0; st < M::STEPS; ++st) {
        const int64_t i = row0 + (int64_t)st * M::RPS;
        if (i >= n_rows) break;
        const int64_t n = a.tok_begin + i;
        const int64_t row = (int64_t)h * a.cap + n;
        float acc[8];
        if (HAS_C) {
            const uint16_t* cbase = a.cent;
            if (VERSIONED) {
                const int32_t* vers = reinterpret_cast<const int32_t*>(chunk_smem + a.n_chunks + 1);
                int lo = 0, hi = a.n_chunks - 1;     // last chunk whose offset <= n
                while (lo < hi) {
                    int mid = (lo + hi + 1) >> 1;
                    if (chunk_smem[mid] <= n) lo = mid; else hi = mid - 1;
                }
                cbase += (int64_t)vers[lo] * version_stride;
            }
            const int id = min((int)a.ids[row], a.C - 1);
            uint4 cv = __ldg(reinterpret_cast<const uint4*>(cbase + ((int64_t)h * a.C + id) * D + sub * 8));
            unpack8(cv, acc);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
        }
        for (int s = 0; s < a.S; ++s) {
            const int64_t srow = (int64_t)s * stage_stride + row;
            const uint32_t code = codes16[srow * (D / 8) + sub];
            const uint32_t m = __ldg(a.meta + srow * (D / G) + sub / LPG);
            const float sc = f16_bits_to_f32(m), z = f16_bits_to_f32(m >> 16);
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = __fadd_rn(acc[k], dequant((code >> (2 * k)) & 3u, sc, z));
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        stg_v4_stream(a.out + (int64_t)h * a.out_head_stride + i * a.out_token_stride + sub * 8, o);
    }
}

template <int D, int G>
cudaError_t encode_dg(const EncodeArgs& a, cudaStream_t s) {
    using M = RowMap<D>;
    if (a.n_tokens == 0) return cudaSuccess;
    dim3 grid((unsigned)((a.n_tokens + M::ROWS_PER_CTA - 1) / M::ROWS_PER_CTA), (unsigned)a.H);
    if (a.C > 0) prq_encode_kernel<D, G, true><<<grid, kThreads, 0, s>>>(a);
    else prq_encode_kernel<D, G, false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t decode_dg(const DecodeArgs& a, cudaStream_t s) {
    using M = RowMap<D>;
    const int64_t rows = a.tok_end - a.tok_begin;
    if (rows <= 0) return cudaSuccess;
    dim3 grid((unsigned)((rows + M::ROWS_PER_CTA - 1) / M::ROWS_PER_CTA), (unsigned)a.H);
    if (a.C > 0 && a.chunk_offset) {
        size_t smem = sizeof(int64_t) * (a.n_chunks + 1) + sizeof(int32_t) * a.n_chunks;
        prq_decode_kernel<D, G, true, true><<<grid, kThreads, smem, s>>>(a);
    } else if (a.C > 0) {
        prq_decode_kernel<D, G, true, false><<<grid, kThreads, 0, s>>>(a);
    } else {
        prq_decode_kernel<D, G, false, false><<<grid, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

#define QVG_DG_SWITCH(FN, D, G, A, S)                                   \
    switch (D * 1000 + G) {                                             \
        case 32016: return FN<32, 16>(A, S);                            \
        case 32032: return FN<32, 32>(A, S);                            \
        case 64016: return FN<64, 16>(A, S);                            \
        case 64032: return FN<64, 32>(A, S);                            \
        case 64064: return FN<64, 64>(A, S);                            \
        case 128016: return FN<128, 16>(A, S);                          \
        case 128032: return FN<128, 32>(A, S);                          \
        case 128064: return FN<128, 64>(A, S);                          \
        case 128128: return FN<128, 128>(A, S);                         \
        case 256016: return FN<256, 16>(A, S);                          \
        case 256032: return FN<256, 32>(A, S);                          \
        case 256064: return FN<256, 64>(A, S);                          \
        case 256128: return FN<256, 128>(A, S);                         \
        default: return cudaErrorInvalidValue;                          \
    }

cudaError_t launch_encode(int D, int G, const EncodeArgs& a, cudaStream_t s) {
    QVG_DG_SWITCH(encode_dg, D, G, a, s)
}

cudaError_t launch_decode(int D, int G, const DecodeArgs& a, cudaStream_t s) {
    QVG_DG_SWITCH(decode_dg, D, G, a, s)
}

}  // namespace qvg
