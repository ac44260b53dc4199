// Coral-KV cross-layer residual coding (news items on the Coral-KV preprint,
// section "cross-layer prediction"): layer l+1 is predicted from the
// reconstruction of layer l by a block-DPLR map -- a dense D x D block per
// head (channel mixing inside the head) plus one global rank-R term (mixing
// across heads) -- and only the prediction residual is quantised, here with
// the same multi-stage 2-bit group quantiser as Quant VideoGen's PRQ.
//
// Two kernels per layer:
//  1. lowrank: t = xhat W ([N x H*D] x [H*D x R], bf16 tensor cores, fp32).
//  2. predict + code: per (64-token tile, head) pred = xhat_h B_h^T + t U_h^T
//     on the tensor cores, t carried as a bf16 hi/lo pair so the low-rank
//     term keeps ~16 significand bits; the fp32 prediction is staged in
//     shared memory and each token row is then PRQ-coded (encode) or
//     rebuilt from its codes (decode).  Encode and decode run the identical
//     prediction code, so the encoder's reconstruction equals the decoder's
//     bit for bit.  Given a smoothed residual's ids and centroids the decode
//     adds c[id] to the stages and rounds that residual to bf16 before adding
//     it to the prediction (the Coral + SAS hybrid).
#include "common.cuh"
#include "kernels.h"
#include "prq16.cuh"

namespace qvg {

namespace {

constexpr int kThreads = 256;
constexpr int kLrTile = 128;     // tokens per low-rank CTA
constexpr int kLrK = 64;         // K chunk of the low-rank GEMM
constexpr int kTok = 64;         // tokens per predict CTA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// t[n][r] = sum_j xhat[n][j] W[j][r]; one CTA = 128 tokens x R, warps own 16 rows.
template <int R>
__global__ void __launch_bounds__(kThreads) coral_lowrank_kernel(const uint16_t* xh, const uint16_t* W,
                                                                 int64_t N, int HD, float* t) {
    constexpr int LDA = kLrK + 8, LDB = R + 8;
    __shared__ __align__(16) uint16_t as[kLrTile * LDA];
    __shared__ __align__(16) uint16_t bs[kLrK * LDB];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t n0 = (int64_t)blockIdx.x * kLrTile;
    float acc[R / 8][4];
#pragma unroll
    for (int i = 0; i < R / 8; ++i)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[i][r] = 0.0f;
    for (int k0 = 0; k0 < HD; k0 += kLrK) {
        for (int v = tid; v < kLrTile * (kLrK / 8); v += kThreads) {
            const int r = v / (kLrK / 8), c = v % (kLrK / 8);
            uint4 val = make_uint4(0, 0, 0, 0);
            if (n0 + r < N) val = ldg_nc_v4(xh + (n0 + r) * HD + k0 + c * 8);
            *reinterpret_cast<uint4*>(as + r * LDA + c * 8) = val;
        }
        for (int v = tid; v < kLrK * (R / 8); v += kThreads) {
            const int r = v / (R / 8), c = v % (R / 8);
            *reinterpret_cast<uint4*>(bs + r * LDB + c * 8) =
                __ldg(reinterpret_cast<const uint4*>(W + (int64_t)(k0 + r) * R) + c);
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < kLrK / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(smem_u32(as + (warp * 16 + (lane & 15)) * LDA + kk * 16 + (lane >> 4) * 8), a[0], a[1], a[2],
                    a[3]);
#pragma unroll
            for (int np = 0; np < R / 16; ++np) {
                uint32_t b0, b1, b2, b3;
                // [k][n] storage, transposed load: lanes 0-15 rows k (lo/hi 8) at n-tile 2np,
                // lanes 16-31 the same rows at n-tile 2np+1
                ldsm_x4_t(smem_u32(bs + (kk * 16 + (lane & 15)) * LDB + np * 16 + (lane >> 4) * 8), b0, b1, b2, b3);
                mma16816(acc[2 * np], a, b0, b1);
                mma16816(acc[2 * np + 1], a, b2, b3);
            }
        }
        __syncthreads();
    }
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int nt = 0; nt < R / 8; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int64_t n = n0 + warp * 16 + g + 8 * (r >> 1);
            if (n < N) t[n * R + nt * 8 + 2 * q + (r & 1)] = acc[nt][r];
        }
}

// Prediction + residual coding of one (64-token tile, head).
template <int D, int G, bool ENCODE>
__global__ void __launch_bounds__(kThreads, 2) coral_predict_kernel(CoralArgs a) {
    constexpr int LDX = D + 8;           // bf16 rows
    constexpr int LDP = D + 4;           // fp32 prediction rows
    extern __shared__ __align__(16) unsigned char smem[];
    const int R = a.R, R2 = 2 * a.R, LDU = 2 * a.R + 8;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem);          // [kTok][LDX]
    uint16_t* bsm = xs + kTok * LDX;                            // [D][LDX], reused as pred [kTok][LDP] fp32
    uint16_t* us = bsm + D * LDX;                               // [D][LDU]
    uint16_t* ts = us + D * LDU;                                // [kTok][LDU]
    float* ps = reinterpret_cast<float*>(bsm);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.y, H = a.H;
    const int HD = H * D;
    const int64_t n0 = (int64_t)blockIdx.x * kTok;
    const bool has_pred = a.xprev != nullptr;

    if (has_pred) {
        for (int v = tid; v < kTok * (D / 8); v += kThreads) {
            const int r = v / (D / 8), c = v % (D / 8);
            uint4 val = make_uint4(0, 0, 0, 0);
            if (n0 + r < a.n_tokens) val = ldg_nc_v4(a.xprev + (n0 + r) * HD + h * D + c * 8);
            *reinterpret_cast<uint4*>(xs + r * LDX + c * 8) = val;
        }
        for (int v = tid; v < D * (D / 8); v += kThreads) {
            const int r = v / (D / 8), c = v % (D / 8);
            *reinterpret_cast<uint4*>(bsm + r * LDX + c * 8) =
                __ldg(reinterpret_cast<const uint4*>(a.B + ((int64_t)h * D + r) * D) + c);
        }
        if (R > 0) {
            for (int v = tid; v < D * (R / 8); v += kThreads) {
                const int r = v / (R / 8), c = v % (R / 8);
                const uint4 u = __ldg(reinterpret_cast<const uint4*>(a.U + ((int64_t)h * D + r) * R) + c);
                *reinterpret_cast<uint4*>(us + r * LDU + c * 8) = u;
                *reinterpret_cast<uint4*>(us + r * LDU + R + c * 8) = u;
            }
            for (int v = tid; v < kTok * R; v += kThreads) {
                const int r = v / R, c = v % R;
                const float tv = (n0 + r < a.n_tokens) ? a.lowrank[(n0 + r) * R + c] : 0.0f;
                const __nv_bfloat16 hi = __float2bfloat16_rn(tv);
                const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(tv, __bfloat162float(hi)));
                ts[r * LDU + c] = __bfloat16_as_ushort(hi);
                ts[r * LDU + R + c] = __bfloat16_as_ushort(lo);
            }
        }
        __syncthreads();

        // warp w: rows 16*(w%4).., columns 64*(w/4)..
        const int rb = (warp & 3) * 16, cb = (warp >> 2) * (D / 2);
        constexpr int NT = D / 2 / 8;
        float acc[NT][4];
#pragma unroll
        for (int i = 0; i < NT; ++i)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][r] = 0.0f;
        const int brow = (lane & 7) + ((lane >> 4) << 3), bk = ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t af[4];
            ldsm_x4(smem_u32(xs + (rb + (lane & 15)) * LDX + kk * 16 + (lane >> 4) * 8), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(bsm + (cb + np * 16 + brow) * LDX + kk * 16 + bk), b0, b1, b2, b3);
                mma16816(acc[2 * np], af, b0, b1);
                mma16816(acc[2 * np + 1], af, b2, b3);
            }
        }
        for (int kk = 0; kk < R2 / 16; ++kk) {
            uint32_t af[4];
            ldsm_x4(smem_u32(ts + (rb + (lane & 15)) * LDU + kk * 16 + (lane >> 4) * 8), af[0], af[1], af[2], af[3]);
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(us + (cb + np * 16 + brow) * LDU + kk * 16 + bk), b0, b1, b2, b3);
                mma16816(acc[2 * np], af, b0, b1);
                mma16816(acc[2 * np + 1], af, b2, b3);
            }
        }
        __syncthreads();   // B no longer needed: reuse its space for the prediction
        const int g = lane >> 2, q = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r)
                ps[(rb + g + 8 * (r >> 1)) * LDP + cb + nt * 8 + 2 * q + (r & 1)] = acc[nt][r];
        __syncthreads();
    }

    // ---- residual coding: a thread owns 16 consecutive channels of a token row
    constexpr int TPR = D / 16, RPW = 32 / TPR, TPG = G / 16;
    const int t = lane % TPR, rw = lane / TPR;
    const int64_t stage_stride = (int64_t)H * a.n_tokens;
    for (int r0 = warp * RPW; r0 < kTok; r0 += (kThreads / 32) * RPW) {
        const int row = r0 + rw;
        const int64_t n = n0 + row;
        const bool valid = n < a.n_tokens;
        float p[16];
        if (has_pred) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = *reinterpret_cast<const float4*>(ps + row * LDP + t * 16 + 4 * k);
                p[4 * k] = v.x; p[4 * k + 1] = v.y; p[4 * k + 2] = v.z; p[4 * k + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) p[i] = 0.0f;
        }
        const int64_t elem = n * HD + h * D + t * 16;
        if (valid && a.pred_out) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<float4*>(a.pred_out + elem + 4 * k) =
                    make_float4(p[4 * k], p[4 * k + 1], p[4 * k + 2], p[4 * k + 3]);
        }
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = p[i];
        const int64_t rowoff = (int64_t)h * a.n_tokens + n;
        if (ENCODE) {
            // every lane takes part in the group reductions; `valid` gates the stores only
            float rr[16];
            const uint4 x0 = valid ? ldg_nc_v4(a.xnext + elem) : make_uint4(0, 0, 0, 0);
            const uint4 x1 = valid ? ldg_nc_v4(a.xnext + elem + 8) : make_uint4(0, 0, 0, 0);
            unpack16(x0, x1, rr);
            sub16(rr, p);
            for (int s = 0; s < a.S; ++s) {
                uint32_t meta;
                const uint32_t code = quant_stage16<TPG>(rr, s + 1 < a.S, acc, meta);
                if (valid) {
                    const int64_t srow = (int64_t)s * stage_stride + rowoff;
                    a.codes[srow * (D / 16) + t] = code;
                    if (t % TPG == 0) a.meta[srow * (D / G) + t / TPG] = meta;
                }
            }
        } else if (valid && a.cent) {
            // a smoothed residual: r_hat = bf16(c[id] + d_1 + d_2 + ...), the QVG
            // decoder's sum and rounding, then x_hat = bf16(pred + r_hat)
            const uint16_t* cr = a.cent + ((int64_t)h * a.C + min((int)a.ids[rowoff], a.C - 1)) * D + t * 16;
            float rr[16];
            unpack16(ldg_nc_v4(cr), ldg_nc_v4(cr + 8), rr);
            for (int s = 0; s < a.S; ++s) {
                const int64_t srow = (int64_t)s * stage_stride + rowoff;
                dequant_add16(rr, __ldg(a.codes + srow * (D / 16) + t), __ldg(a.meta + srow * (D / G) + (t * 16) / G));
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = __fadd_rn(acc[i], __bfloat162float(__float2bfloat16_rn(rr[i])));
        } else if (valid) {
            for (int s = 0; s < a.S; ++s) {
                const int64_t srow = (int64_t)s * stage_stride + rowoff;
                dequant_add16(acc, __ldg(a.codes + srow * (D / 16) + t), __ldg(a.meta + srow * (D / G) + (t * 16) / G));
            }
        }
        if (valid && a.xhat) {
            uint4 o0, o1;
            pack16_bf16(acc, o0, o1);
            *reinterpret_cast<uint4*>(a.xhat + elem) = o0;
            *reinterpret_cast<uint4*>(a.xhat + elem + 8) = o1;
        }
    }
}

size_t predict_smem(int D, int R) {
    const int LDX = D + 8, LDU = 2 * R + 8;
    size_t b = (size_t)kTok * LDX * 2 + (size_t)D * LDX * 2 + (size_t)D * LDU * 2 + (size_t)kTok * LDU * 2;
    const size_t pred = (size_t)kTok * (D + 4) * 4;
    const size_t bpart = (size_t)D * LDX * 2;
    if (pred > bpart) b += pred - bpart;
    return b;
}

template <int D, int G>
cudaError_t coral_dg(bool encode, const CoralArgs& a, cudaStream_t s) {
    if (a.n_tokens == 0) return cudaSuccess;
    if (a.xprev && a.workspace && a.workspace_bytes >= coral_tc_scratch_bytes(a.H, a.n_tokens)) {
        // tensor-core path first; the kernels below serve every other shape
        auto a256 = [](size_t v) { return (v + 255) & ~(size_t)255; };
        const size_t N = (size_t)a.n_tokens, HD = (size_t)a.H * 128;
        uint8_t* base = static_cast<uint8_t*>(a.workspace);
        CoralTcScratch w;
        w.t2 = reinterpret_cast<uint16_t*>(base);
        w.wt = reinterpret_cast<uint16_t*>(base + a256(N * 64 * 2));
        w.ud = reinterpret_cast<uint16_t*>(base + a256(N * 64 * 2) + a256(32 * HD * 2));
        if (a.prepared) use_prepared(a.prepared, a.H, w);
        w.err = a.err_out ? a.err_out
                          : reinterpret_cast<uint32_t*>(base + coral_tc_scratch_bytes(a.H, a.n_tokens) - 256);
        bool launched = false;
        cudaError_t e = launch_coral_tc(D, G, encode, a, w, &launched, s);
        if (e != cudaSuccess || launched) return e;
    }
    const int HD = a.H * D;
    if (a.xprev && a.R > 0) {
        dim3 g((unsigned)((a.n_tokens + kLrTile - 1) / kLrTile));
        switch (a.R) {
            case 16: coral_lowrank_kernel<16><<<g, kThreads, 0, s>>>(a.xprev, a.W, a.n_tokens, HD, a.lowrank); break;
            case 32: coral_lowrank_kernel<32><<<g, kThreads, 0, s>>>(a.xprev, a.W, a.n_tokens, HD, a.lowrank); break;
            case 48: coral_lowrank_kernel<48><<<g, kThreads, 0, s>>>(a.xprev, a.W, a.n_tokens, HD, a.lowrank); break;
            case 64: coral_lowrank_kernel<64><<<g, kThreads, 0, s>>>(a.xprev, a.W, a.n_tokens, HD, a.lowrank); break;
            default: return cudaErrorInvalidValue;
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t smem = predict_smem(D, a.R);
    auto kern = encode ? coral_predict_kernel<D, G, true> : coral_predict_kernel<D, G, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.n_tokens + kTok - 1) / kTok), (unsigned)a.H);
    kern<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

// Coral + SAS hybrid: the prediction residual rounded to bf16 (the input of
// the k-means smoothing), and the reconstruction pred + r_hat rounded to bf16.
// Eight elements a thread and step.
__global__ void coral_residual_kernel(const uint16_t* __restrict__ xnext, const float* __restrict__ pred,
                                      int64_t count, uint16_t* __restrict__ r) {
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < count;
         i += (int64_t)gridDim.x * blockDim.x * 8) {
        const uint4 xv = ldg_nc_v4(xnext + i);
        const float4 p0 = *reinterpret_cast<const float4*>(pred + i), p1 = *reinterpret_cast<const float4*>(pred + i + 4);
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const float pp[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float lo = __fsub_rn(bf16_lo(xw[k]), pp[2 * k]), hi = __fsub_rn(bf16_hi(xw[k]), pp[2 * k + 1]);
            o[k] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
        }
        *reinterpret_cast<uint4*>(r + i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

__global__ void coral_recon_kernel(const float* __restrict__ pred, const uint16_t* __restrict__ rhat, int64_t count,
                                   uint16_t* __restrict__ xhat) {
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < count;
         i += (int64_t)gridDim.x * blockDim.x * 8) {
        const uint4 rv = ldg_nc_v4(rhat + i);
        const float4 p0 = *reinterpret_cast<const float4*>(pred + i), p1 = *reinterpret_cast<const float4*>(pred + i + 4);
        const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
        const float pp[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float lo = __fadd_rn(pp[2 * k], bf16_lo(rw[k])), hi = __fadd_rn(pp[2 * k + 1], bf16_hi(rw[k]));
            o[k] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
        }
        *reinterpret_cast<uint4*>(xhat + i) = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

unsigned elementwise_grid(int64_t count) {
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    const int64_t blocks = (count / 8 + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sms * 8;
    return (unsigned)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace

cudaError_t launch_coral_residual(const uint16_t* xnext, const float* pred, int64_t count, uint16_t* r,
                                  cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    coral_residual_kernel<<<elementwise_grid(count), kThreads, 0, s>>>(xnext, pred, count, r);
    return cudaGetLastError();
}

cudaError_t launch_coral_recon(const float* pred, const uint16_t* rhat, int64_t count, uint16_t* xhat,
                               cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    coral_recon_kernel<<<elementwise_grid(count), kThreads, 0, s>>>(pred, rhat, count, xhat);
    return cudaGetLastError();
}

cudaError_t launch_coral(int D, int G, bool encode, const CoralArgs& a, cudaStream_t s) {
    switch (D * 1000 + G) {
        case 64016: return coral_dg<64, 16>(encode, a, s);
        case 64032: return coral_dg<64, 32>(encode, a, s);
        case 64064: return coral_dg<64, 64>(encode, a, s);
        case 128016: return coral_dg<128, 16>(encode, a, s);
        case 128032: return coral_dg<128, 32>(encode, a, s);
        case 128064: return coral_dg<128, 64>(encode, a, s);
        case 128128: return coral_dg<128, 128>(encode, a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qvg
