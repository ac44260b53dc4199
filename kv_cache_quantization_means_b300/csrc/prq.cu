// Progressive residual quantisation: encoder and decoder kernels.
//
// Quant VideoGen explainer, Sommario tecnico sec. 2A item 3 (subtract each
// token's centroid) and sec. 2B items 1-3 (re-quantise the residual stage by
// stage; decode = dequantise, sum the stages, add the centroid back).
//
// Both kernels stream HBM.  A thread owns 16 consecutive channels of a token
// row (two 16-byte bf16 vectors, one 32-bit code word per stage); D/16 lanes
// cover a row and a warp covers 32/(D/16) rows at a time.  Group min/max are
// warp-shuffle reductions over the G/16 lanes of a group.  Every load of a
// row is issued before any of its arithmetic (the encoder also prefetches
// the next row), so each warp keeps several rows of HBM traffic in flight.
#include "common.cuh"
#include "kernels.h"
#include "prq16.cuh"

namespace qvg {

namespace {

constexpr int kThreads = 256;
constexpr int kEncRowsPerThread = 4;   // encoder: rows per thread (pipelined)
constexpr int kDecRowsPerThread = 2;   // decoder: rows per thread (loads hoisted)

template <int D>
struct Map16 {
    static constexpr int TPR = D / 16;                   // threads per row
    static constexpr int RPW = 32 / TPR;                 // rows per warp step
    static constexpr int RPS = RPW * (kThreads / 32);    // rows per CTA step
};

template <int D, int G, bool HAS_C>
__global__ void __launch_bounds__(kThreads, 4) prq_encode_kernel(EncodeArgs a) {
    using M = Map16<D>;
    constexpr int TPG = G / 16;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = lane % M::TPR;
    const int h = blockIdx.y;
    // rows of this thread: base + k * RPS, k < kEncRowsPerThread
    const int64_t base = (int64_t)blockIdx.x * M::RPS * kEncRowsPerThread + (int64_t)warp * M::RPW + lane / M::TPR;

    const uint16_t* xh = a.x + (int64_t)h * a.head_stride + t * 16;
    const uint8_t* idh = HAS_C ? a.ids + (int64_t)h * a.cap + a.tok_offset : nullptr;
    const uint16_t* ch = HAS_C ? a.cent + (int64_t)h * a.C * D + t * 16 : nullptr;
    const int64_t stage_rows = (int64_t)a.H * a.cap;
    const int64_t row0 = (int64_t)h * a.cap + a.tok_offset;

    uint4 xa = make_uint4(0, 0, 0, 0), xb = xa, ca = xa, cb = xa;
    if (base < a.n_tokens) {
        const uint16_t* p = xh + base * a.token_stride;
        xa = ldg_nc_v4(p);
        xb = ldg_nc_v4(p + 8);
        if (HAS_C) {
            const int id = min((int)idh[base], a.C - 1);
            ca = __ldg(reinterpret_cast<const uint4*>(ch + (int64_t)id * D));
            cb = __ldg(reinterpret_cast<const uint4*>(ch + (int64_t)id * D + 8));
        }
    }
#pragma unroll 1
    for (int k = 0; k < kEncRowsPerThread; ++k) {
        const int64_t n = base + (int64_t)k * M::RPS;
        const bool valid = n < a.n_tokens;
        // prefetch the next row of this thread
        const int64_t nn = n + M::RPS;
        uint4 nxa = make_uint4(0, 0, 0, 0), nxb = nxa;
        int nid = 0;
        const bool nvalid = (k + 1 < kEncRowsPerThread) && nn < a.n_tokens;
        if (nvalid) {
            const uint16_t* p = xh + nn * a.token_stride;
            nxa = ldg_nc_v4(p);
            nxb = ldg_nc_v4(p + 8);
            if (HAS_C) nid = min((int)idh[nn], a.C - 1);
        }
        float r[16];
        unpack16(xa, xb, r);
        if (HAS_C) {
            float c[16];
            unpack16(ca, cb, c);
            sub16(r, c);
        }
        const int64_t row = row0 + n;
        for (int s = 0; s < a.S; ++s) {
            uint32_t meta;
            const uint32_t code = quant_stage16<TPG>(r, s + 1 < a.S, nullptr, meta);
            if (valid) {
                const int64_t srow = (int64_t)s * stage_rows + row;
                a.codes[srow * (D / 16) + t] = code;
                if (t % TPG == 0) a.meta[srow * (D / G) + t / TPG] = meta;
            }
        }
        xa = nxa;
        xb = nxb;
        if (HAS_C && nvalid) {
            ca = __ldg(reinterpret_cast<const uint4*>(ch + (int64_t)nid * D));
            cb = __ldg(reinterpret_cast<const uint4*>(ch + (int64_t)nid * D + 8));
        }
    }
}

// Centroid version of token n: the last chunk whose first token is <= n.
__device__ __forceinline__ int chunk_of(const int64_t* offs, int n_chunks, int64_t n) {
    int lo = 0, hi = n_chunks - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (offs[mid] <= n) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <int D, int G, bool HAS_C, bool VERSIONED>
__global__ void __launch_bounds__(kThreads, 4) prq_decode_kernel(DecodeArgs a) {
    using M = Map16<D>;
    constexpr int NR = kDecRowsPerThread;
    extern __shared__ int64_t chunk_smem[];   // VERSIONED: offsets[n_chunks + 1], versions[n_chunks]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = lane % M::TPR;
    const int h = blockIdx.y;
    if (VERSIONED) {
        int32_t* vers = reinterpret_cast<int32_t*>(chunk_smem + a.n_chunks + 1);
        for (int i = threadIdx.x; i <= a.n_chunks; i += kThreads) chunk_smem[i] = a.chunk_offset[i];
        for (int i = threadIdx.x; i < a.n_chunks; i += kThreads) vers[i] = a.chunk_version[i];
        __syncthreads();
    }
    const int64_t n_rows = a.tok_end - a.tok_begin;
    const int64_t base = (int64_t)blockIdx.x * M::RPS * NR + (int64_t)warp * M::RPW + lane / M::TPR;
    const int64_t stage_rows = (int64_t)a.H * a.cap;
    constexpr int WPR = D / 16, MPR = D / G;
    const int mi = (t * 16) / G;

    int64_t ii[NR];
    bool ok[NR];
    int id[NR];
    uint32_t code[NR][kMaxStages], meta[NR][kMaxStages];
#pragma unroll
    for (int k = 0; k < NR; ++k) {
        ii[k] = base + (int64_t)k * M::RPS;
        ok[k] = ii[k] < n_rows;
        const int64_t row = (int64_t)h * a.cap + a.tok_begin + ii[k];
        id[k] = 0;
        if (HAS_C && ok[k]) id[k] = a.ids[row];
#pragma unroll
        for (int s = 0; s < kMaxStages; ++s) {
            code[k][s] = 0;
            meta[k][s] = 0;
            if (s < a.S && ok[k]) {
                const int64_t srow = (int64_t)s * stage_rows + row;
                code[k][s] = __ldg(a.codes + srow * WPR + t);
                meta[k][s] = __ldg(a.meta + srow * MPR + mi);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < NR; ++k) {
        if (!ok[k]) continue;
        float acc[16];
        if (HAS_C) {
            const uint16_t* cbase = a.cent;
            if (VERSIONED) {
                const int32_t* vers = reinterpret_cast<const int32_t*>(chunk_smem + a.n_chunks + 1);
                const int c = chunk_of(chunk_smem, a.n_chunks, a.tok_begin + ii[k]);
                cbase += (int64_t)vers[c] * a.H * a.C * D;
            }
            const uint16_t* cr = cbase + ((int64_t)h * a.C + min(id[k], a.C - 1)) * D + t * 16;
            const uint4 c0 = __ldg(reinterpret_cast<const uint4*>(cr));
            const uint4 c1 = __ldg(reinterpret_cast<const uint4*>(cr + 8));
            unpack16(c0, c1, acc);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        }
#pragma unroll
        for (int s = 0; s < kMaxStages; ++s)
            if (s < a.S) dequant_add16(acc, code[k][s], meta[k][s]);
        uint4 o0, o1;
        pack16_bf16(acc, o0, o1);
        uint16_t* op = a.out + (int64_t)h * a.out_head_stride + ii[k] * a.out_token_stride + t * 16;
        stg_v4_stream(op, o0);
        stg_v4_stream(op + 8, o1);
    }
}

template <int D, int G>
cudaError_t encode_dg(const EncodeArgs& a, cudaStream_t s) {
    using M = Map16<D>;
    if (a.n_tokens == 0) return cudaSuccess;
    const int64_t rows_per_cta = (int64_t)M::RPS * kEncRowsPerThread;
    dim3 grid((unsigned)((a.n_tokens + rows_per_cta - 1) / rows_per_cta), (unsigned)a.H);
    if (a.C > 0) prq_encode_kernel<D, G, true><<<grid, kThreads, 0, s>>>(a);
    else prq_encode_kernel<D, G, false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t decode_dg(const DecodeArgs& a, cudaStream_t s) {
    using M = Map16<D>;
    const int64_t rows = a.tok_end - a.tok_begin;
    if (rows <= 0) return cudaSuccess;
    const int64_t rows_per_cta = (int64_t)M::RPS * kDecRowsPerThread;
    dim3 grid((unsigned)((rows + rows_per_cta - 1) / rows_per_cta), (unsigned)a.H);
    if (a.C > 0 && a.chunk_offset) {
        const size_t smem = sizeof(int64_t) * (a.n_chunks + 1) + sizeof(int32_t) * a.n_chunks;
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
