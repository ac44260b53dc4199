// Progressive residual quantisation: encoder and decoder kernels.
//
// Quant VideoGen explainer, Sommario tecnico sec. 2A item 3 (subtract each
// token's centroid) and sec. 2B items 1-3 (re-quantise the residual stage by
// stage; decode = dequantise, sum the stages, add the centroid back).
//
// Both kernels stream HBM.  In the encoder a thread owns CPT = min(G, 32)
// consecutive channels of a token row -- a whole group, or a 1/TPG share of a
// 64- or 128-channel group whose extremes are combined with shuffles -- so
// the group's scale and zero-point are formed once; its channels
// arrive as 16-byte bf16 vectors and its codes leave as one vector store per
// stage.  In the write-heavy decoder a thread owns 16 consecutive channels,
// so a warp's stores cover whole contiguous row segments.  Every load of a
// row is issued before any of its arithmetic.  Codes are 2-bit (the QVG
// codec) or 4-bit (the PRQ_INT4 variant of the KV Cache Quantization for
// Self-Forcing Video Generation study, read as the same scheme with 15
// steps); B is a template parameter of both kernels.
#include "common.cuh"
#include "kernels.h"
#include "prq16.cuh"

namespace qvg {

namespace {

constexpr int kThreads = 256;

constexpr int kDecRowsPerThread = 2;   // decoder: rows per thread (loads hoisted)

// Decoder mapping: a thread owns 16 consecutive channels (one code word per
// stage), so each warp store instruction writes whole contiguous row segments.
template <int D>
struct Map16 {
    static constexpr int TPR = D / 16;                   // threads per row
    static constexpr int RPW = 32 / TPR;                 // rows per warp step
    static constexpr int RPS = RPW * (kThreads / 32);    // rows per CTA step
};

template <int D, int G, int B>
struct GMap {
    static constexpr int CPT = G < 32 ? G : 32;   // channels per thread
    static constexpr int TPG = G / CPT;           // threads per group (1 or 2)
    static constexpr int TPR = D / CPT;           // threads per row
    static constexpr int RPW = 32 / TPR;          // rows per warp
    static constexpr int RPC = RPW * (kThreads / 32);
    static constexpr int NV = CPT / 8;            // 16-byte bf16 vectors per thread
    static constexpr int NW = CPT * B / 32;       // code words per thread and stage
    static constexpr int WPR = D * B / 32;        // code words per row and stage
};

// 16-byte load through L1 (a thread's consecutive vectors share sectors).
__device__ __forceinline__ uint4 ldg_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

template <int NW>
__device__ __forceinline__ void store_words(uint32_t* p, const uint32_t* w) {
    if constexpr (NW == 4) *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    else if constexpr (NW == 2) *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
    else *p = w[0];
}

template <int NW>
__device__ __forceinline__ void load_words(const uint32_t* p, uint32_t* w) {
    if constexpr (NW == 4) {
        const uint4 v = ldg_v4(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (NW == 2) {
        const uint2 v = __ldg(reinterpret_cast<const uint2*>(p));
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = __ldg(p);
    }
}

// SC: the stage count when it is a compile-time constant (the loop over
// stages then unrolls), 0 when it is read from the arguments.
template <int D, int G, bool HAS_C, int B, int SC>
__global__ void __launch_bounds__(kThreads, 4) prq_encode_kernel(EncodeArgs a) {
    using M = GMap<D, G, B>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t = lane % M::TPR;
    const int h = blockIdx.y;
    const int64_t n = (int64_t)blockIdx.x * M::RPC + (int64_t)warp * M::RPW + lane / M::TPR;
    const bool valid = n < a.n_tokens;
    // every lane takes part in the group reductions; `valid` gates memory only
    float r[M::CPT];
    {
        uint4 xv[M::NV], cv[M::NV];
        // the cluster id first: the centroid loads depend on it and then
        // overlap the token loads
        const int id = (HAS_C && valid) ? min((int)a.ids[(int64_t)h * a.cap + a.tok_offset + n], a.C - 1) : 0;
        const uint16_t* xp = a.x + (int64_t)h * a.head_stride + (valid ? n : 0) * a.token_stride + t * M::CPT;
#pragma unroll
        for (int k = 0; k < M::NV; ++k) xv[k] = valid ? ldg_v4(xp + 8 * k) : make_uint4(0, 0, 0, 0);
        if (HAS_C) {
            const uint16_t* cp = a.cent + ((int64_t)h * a.C + id) * D + t * M::CPT;
#pragma unroll
            for (int k = 0; k < M::NV; ++k) cv[k] = valid ? __ldg(reinterpret_cast<const uint4*>(cp + 8 * k)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < M::NV; k += 2) {
            float c[16];
            unpack16(xv[k], xv[k + 1], r + 8 * k);
            if (HAS_C) {
                unpack16(cv[k], cv[k + 1], c);
                sub16(r + 8 * k, c);
            }
        }
    }
    const int64_t row = (int64_t)h * a.cap + a.tok_offset + n;
    const int64_t stage_rows = (int64_t)a.H * a.cap;
    const int S = SC ? SC : a.S;
#pragma unroll
    for (int s = 0; s < (SC ? SC : kMaxStages); ++s) {
        if (!SC && s >= S) break;
        uint32_t code[M::NW], meta;
        quant_stage<M::CPT, M::TPG, B>(r, s + 1 < S, nullptr, code, meta);
        if (valid) {
            const int64_t srow = (int64_t)s * stage_rows + row;
            store_words<M::NW>(a.codes + srow * M::WPR + t * M::NW, code);
            if (t % M::TPG == 0) a.meta[srow * (D / G) + t / M::TPG] = meta;
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

template <int D, int G, bool HAS_C, bool VERSIONED, int B>
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
    constexpr int WPT = 16 * B / 32;          // code words per thread and stage (1 or 2)
    constexpr int WPR = D * B / 32, MPR = D / G;
    const int mi = (t * 16) / G;

    int64_t ii[NR];
    bool ok[NR];
    int id[NR];
    uint32_t code[NR][kMaxStages][WPT], meta[NR][kMaxStages];
#pragma unroll
    for (int k = 0; k < NR; ++k) {
        ii[k] = base + (int64_t)k * M::RPS;
        ok[k] = ii[k] < n_rows;
        const int64_t row = (int64_t)h * a.cap + a.tok_begin + ii[k];
        id[k] = 0;
        if (HAS_C && ok[k]) id[k] = a.ids[row];
#pragma unroll
        for (int s = 0; s < kMaxStages; ++s) {
#pragma unroll
            for (int w = 0; w < WPT; ++w) code[k][s][w] = 0;
            meta[k][s] = 0;
            if (s < a.S && ok[k]) {
                const int64_t srow = (int64_t)s * stage_rows + row;
                load_words<WPT>(a.codes + srow * WPR + t * WPT, code[k][s]);
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
        for (int s = 0; s < kMaxStages; ++s) {
            if (s >= a.S) continue;
            if constexpr (B == 2) {
                dequant_add16(acc, code[k][s][0], meta[k][s]);
            } else {
                dequant_add8x4(acc, code[k][s][0], meta[k][s]);
                dequant_add8x4(acc + 8, code[k][s][1], meta[k][s]);
            }
        }
        uint4 o0, o1;
        pack16_bf16(acc, o0, o1);
        uint16_t* op = a.out + (int64_t)h * a.out_head_stride + ii[k] * a.out_token_stride + t * 16;
        stg_v4_stream(op, o0);
        stg_v4_stream(op + 8, o1);
    }
}

template <int D, int G, int B>
cudaError_t encode_dgb(const EncodeArgs& a, cudaStream_t s) {
    using M = GMap<D, G, B>;
    dim3 grid((unsigned)((a.n_tokens + M::RPC - 1) / M::RPC), (unsigned)a.H);
    auto kern = a.C > 0 ? prq_encode_kernel<D, G, true, B, 0> : prq_encode_kernel<D, G, false, B, 0>;
    if constexpr (D == 64 || D == 128) {
        // the head dims of the measured workloads get the unrolled stage loop
        switch (a.S) {
#define QVG_ENC_SC(SV) \
            case SV: kern = a.C > 0 ? prq_encode_kernel<D, G, true, B, SV> : prq_encode_kernel<D, G, false, B, SV>; break;
            QVG_ENC_SC(1) QVG_ENC_SC(2) QVG_ENC_SC(3) QVG_ENC_SC(4)
#undef QVG_ENC_SC
            default: break;
        }
    }
    kern<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t encode_dg(const EncodeArgs& a, cudaStream_t s) {
    if (a.n_tokens == 0) return cudaSuccess;
    if (a.bits == 4) return encode_dgb<D, G, 4>(a, s);
    if (a.bits == 2) return encode_dgb<D, G, 2>(a, s);
    return cudaErrorInvalidValue;
}

template <int D, int G, int B>
cudaError_t decode_dgb(const DecodeArgs& a, cudaStream_t s) {
    using M = Map16<D>;
    const int64_t rows = a.tok_end - a.tok_begin;
    const int64_t rows_per_cta = (int64_t)M::RPS * kDecRowsPerThread;
    dim3 grid((unsigned)((rows + rows_per_cta - 1) / rows_per_cta), (unsigned)a.H);
    if (a.C > 0 && a.chunk_offset) {
        const size_t smem = sizeof(int64_t) * (a.n_chunks + 1) + sizeof(int32_t) * a.n_chunks;
        prq_decode_kernel<D, G, true, true, B><<<grid, kThreads, smem, s>>>(a);
    } else if (a.C > 0) {
        prq_decode_kernel<D, G, true, false, B><<<grid, kThreads, 0, s>>>(a);
    } else {
        prq_decode_kernel<D, G, false, false, B><<<grid, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t decode_dg(const DecodeArgs& a, cudaStream_t s) {
    if (a.tok_end - a.tok_begin <= 0) return cudaSuccess;
    if (a.bits == 4) return decode_dgb<D, G, 4>(a, s);
    if (a.bits == 2) return decode_dgb<D, G, 2>(a, s);
    return cudaErrorInvalidValue;
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
    bool launched = false;
    cudaError_t e = launch_decode_tma(D, G, a, &launched, s);
    if (e != cudaSuccess || launched) return e;
    QVG_DG_SWITCH(decode_dg, D, G, a, s)
}

}  // namespace qvg
