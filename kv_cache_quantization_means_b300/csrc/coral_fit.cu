// Coral-KV adapted configuration: the per-head block predictors rebuilt for
// the current layer pair.
//
// Coral-KV news items, "cross-layer prediction": besides the reusable
// configuration (predictors calibrated offline) the pages describe an
// adapted one, in which the light block-diagonal predictors are rebuilt for
// the current video while the global low-rank part stays as calibrated.
// Per head h this computes the ridge-regularised least-squares block
//     B_h = argmin_B  sum_n || y_{n,h} - U_h t_n - B x_{n,h} ||^2 + lambda_h ||B||^2,
// x = the reconstruction x_hat_l, y = x_{l+1}, t_n = W^T x_hat_n,
// lambda_h = 2^-20 trace(G_h) / D with G_h = X_h^T X_h, by the normal equations
//     (G_h + lambda_h I) Z = X_h^T (Y_h - T U_h^T),   B_h = Z^T (bf16).
//
//  gram   grid (chunk of 1024 tokens, column block, head): X_h^T [X_h | Y_h | t]
//         with mma.sync bf16 -> fp32 (exact products, fp32 sums over the
//         chunk); x_hat and y are token-major, so both operands come from
//         shared memory through transposed ldmatrix.  One fp32 partial per
//         chunk.
//  reduce the partials added in chunk order, a thread per element
//         (deterministic).
//  solve  eight CTAs per head, 16 right-hand sides each: forms those columns
//         of C - P U_h^T (t as its bf16 hi + lo pair), adds the ridge,
//         factors G = L L^T (fp32, right-looking; every CTA of the head
//         factors the same G the same way) and solves its columns.
// The low-rank projection t comes from the tensor-core low-rank kernel.
#include "common.cuh"
#include "kernels.h"

namespace qvg {

namespace {

constexpr int kFD = 128;          // head dim
constexpr int kFR = 32;           // rank of the low-rank part
constexpr int kFStep = 32;        // tokens per shared-memory slice
constexpr int kLdX = kFD + 8;     // padded rows: the 8 rows of an ldmatrix hit distinct banks
constexpr int kFBlocks = 3;       // column blocks: x_h (128), y_h (128), t = (t_hi | t_lo) (64)

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t saddr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

struct GramArgs {
    const uint16_t* xh;   // [N][H*D]
    const uint16_t* y;    // [N][H*D]
    const uint16_t* t2;   // [N][64]: t_hi | t_lo
    int64_t n_tokens;
    int H, chunks;
    float* part;          // [H][kFBlocks][chunks][128][128]
};

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros (the
// source address must still be a valid one).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

constexpr int kGramStages = 3;    // token slices in flight

// grid (chunks, kFBlocks, H), 256 threads.  Warp w owns rows i in
// [16w, 16w + 16) of X_h^T B over the chunk's tokens, B = the column block
// (128 columns; 64 for t).  The 32-token slices of X_h and B stream through a
// three-stage ring of asynchronous copies, so a slice's loads overlap the
// MMAs of the two before it; the slices are summed in token order.
__global__ void __launch_bounds__(256) coral_gram_kernel(GramArgs a) {
    extern __shared__ __align__(16) uint16_t gram_smem[];
    auto xs = reinterpret_cast<uint16_t(*)[kFStep][kLdX]>(gram_smem);                                  // [stage][32][kLdX]
    auto bs = reinterpret_cast<uint16_t(*)[kFStep][kLdX]>(gram_smem + kGramStages * kFStep * kLdX);    // [stage][32][kLdX]
    const int chunk = blockIdx.x, cb = blockIdx.y, h = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t HD = (int64_t)a.H * kFD;
    const int64_t n0 = (int64_t)chunk * kFitChunkTokens;
    const int64_t n1 = min(n0 + (int64_t)kFitChunkTokens, a.n_tokens);
    const int ncol = cb == 2 ? 64 : 128;
    const uint16_t* bsrc = cb == 0 ? a.xh + h * kFD : (cb == 1 ? a.y + h * kFD : a.t2);
    const int64_t bstride = cb == 2 ? 64 : HD;
    float acc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
    const int mi = lane >> 3, rr = lane & 7;
    const int nslices = (int)((n1 - n0 + kFStep - 1) / kFStep);
    // slice sl's rows of X_h (32 x 128 bf16) and of the column block into stage st;
    // rows past the chunk and columns past the block are zero-filled
    auto load_slice = [&](int sl, int st) {
        const int64_t nb = n0 + (int64_t)sl * kFStep;
        for (int v = tid; v < kFStep * 16; v += 256) {
            const int r = v >> 4, k = v & 15;
            const int64_t n = nb + r;
            const bool in = n < n1;
            const int64_t nn = in ? n : n0;
            cp_async16(saddr(&xs[st][r][8 * k]), a.xh + nn * HD + h * kFD + 8 * k, in ? 16u : 0u);
            const bool col_ok = 8 * k < ncol;
            cp_async16(saddr(&bs[st][r][8 * k]), bsrc + nn * bstride + (col_ok ? 8 * k : 0), (in && col_ok) ? 16u : 0u);
        }
    };
#pragma unroll
    for (int sl = 0; sl < kGramStages - 1; ++sl) {
        if (sl < nslices) load_slice(sl, sl);
        cp_async_commit();
    }
    for (int sl = 0; sl < nslices; ++sl) {
        const int st = sl % kGramStages;
        cp_async_wait<kGramStages - 2>();       // this thread's copies of slice sl have landed
        __syncthreads();                        // everyone's; and slice sl - 1 is no longer read
        if (sl + kGramStages - 1 < nslices) load_slice(sl + kGramStages - 1, (sl + kGramStages - 1) % kGramStages);
        cp_async_commit();
#pragma unroll
        for (int kk = 0; kk < kFStep; kk += 16) {
            // A = X_h^T (rows i, columns = tokens): matrices (tok 0-7 | 8-15) x (i 0-7 | 8-15)
            uint32_t af[4];
            ldsm_x4_t(saddr(&xs[st][kk + ((mi >> 1) << 3) + rr][16 * warp + ((mi & 1) << 3)]), af[0], af[1], af[2],
                      af[3]);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                if (16 * p >= ncol) break;
                // B = block columns j (as the n dimension), tokens as k
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(saddr(&bs[st][kk + ((mi & 1) << 3) + rr][16 * p + ((mi >> 1) << 3)]), b0, b1, b2, b3);
                mma_bf16(acc[2 * p], af, b0, b1);
                mma_bf16(acc[2 * p + 1], af, b2, b3);
            }
        }
    }
    cp_async_wait<0>();
    float* out = a.part + (((int64_t)h * kFBlocks + cb) * a.chunks + chunk) * (kFD * kFD);
    const int g = lane >> 2, q = lane & 3;
#pragma unroll
    for (int jt = 0; jt < 16; ++jt) {
        if (8 * jt >= ncol) break;
        const int i = 16 * warp + g, j = 8 * jt + 2 * q;
        *reinterpret_cast<float2*>(out + (int64_t)i * kFD + j) = make_float2(acc[jt][0], acc[jt][1]);
        *reinterpret_cast<float2*>(out + (int64_t)(i + 8) * kFD + j) = make_float2(acc[jt][2], acc[jt][3]);
    }
}

// partials -> sums: element e of block (h, cb) summed over the chunks in
// order, a thread per element (coalesced)
__global__ void __launch_bounds__(256) coral_gram_reduce_kernel(const float* part, int chunks, int64_t total,
                                                                float* red) {
    const int64_t t = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (t >= total) return;
    const int64_t blkidx = t / (kFD * kFD), e = t % (kFD * kFD);
    const float* src = part + blkidx * chunks * (kFD * kFD) + e;
    float acc = 0.0f;
    for (int c = 0; c < chunks; ++c) acc += __ldg(src + (int64_t)c * (kFD * kFD));
    red[t] = acc;
}

constexpr int kLdS = kFD + 1;     // padded fp32 rows of the solve
constexpr int kSolveCols = 16;    // right-hand sides (columns of B_h^T) per solve CTA
constexpr int kLdR = kSolveCols + 1;

struct SolveArgs {
    const float* red;     // [H][kFBlocks][128][128]: X^T X, X^T Y, X^T t
    const uint16_t* U;    // [H*D][32]
    int H;
    uint16_t* B;          // [H][D][D] out
};

// One CTA per head, 256 threads.
__global__ void __launch_bounds__(256) coral_solve_kernel(SolveArgs a) {
    extern __shared__ float sm[];
    float* Gm = sm;                         // [128][kLdS]: G, then its Cholesky factor L (lower)
    float* Rm = Gm + kFD * kLdS;            // [128][kLdR]: this CTA's right-hand sides, then solutions
    float* Pm = Rm + kFD * kLdR;            // [128][64]: X_h^T (t_hi | t_lo)
    float* Us = Pm + kFD * 64;              // [kSolveCols][32]: the rows of U_h for those columns
    __shared__ float trace_s;
    const int tid = threadIdx.x, h = blockIdx.y, o0 = blockIdx.x * kSolveCols;
    const float* base = a.red + (int64_t)h * kFBlocks * (kFD * kFD);
    for (int e = tid; e < kFD * kFD; e += 256) {
        const int i = e >> 7, k = e & 127;
        Gm[i * kLdS + k] = base[e];
        if (k < 64) Pm[i * 64 + k] = base[2 * kFD * kFD + e];
    }
    for (int e = tid; e < kFD * kSolveCols; e += 256) {
        const int i = e / kSolveCols, c = e % kSolveCols;
        Rm[i * kLdR + c] = base[kFD * kFD + i * kFD + o0 + c];
    }
    for (int e = tid; e < kSolveCols * kFR; e += 256) Us[e] = bf16f(a.U[((int64_t)h * kFD + o0) * kFR + e]);
    __syncthreads();
    // right-hand sides C - P U_h^T, with P = X_h^T (t_hi + t_lo)
    for (int e = tid; e < kFD * kSolveCols; e += 256) {
        const int i = e / kSolveCols, c = e % kSolveCols;
        float s = 0.0f;
#pragma unroll 8
        for (int r = 0; r < kFR; ++r) s = fmaf(Pm[i * 64 + r] + Pm[i * 64 + kFR + r], Us[c * kFR + r], s);
        Rm[i * kLdR + c] -= s;
    }
    if (tid < 32) {
        float t = 0.0f;
        for (int i = tid; i < kFD; i += 32) t += Gm[i * kLdS + i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (tid == 0) trace_s = t;
    }
    __syncthreads();
    const float tr = trace_s;
    uint16_t* Bh = a.B + (int64_t)h * kFD * kFD;
    if (!(tr > 0.0f)) {
        for (int e = tid; e < kSolveCols * kFD; e += 256) Bh[(int64_t)o0 * kFD + e] = 0;
        return;
    }
    const float lambda = ldexpf(tr / kFD, -20);
    if (tid < kFD) Gm[tid * kLdS + tid] += lambda;
    __syncthreads();
    // right-looking Cholesky, G = L L^T in the lower triangle; the trailing
    // update of step j is spread over the threads element by element (16 x 16
    // thread grid), each element updated once per step, steps in order
    const int ty = tid >> 4, tx = tid & 15;
    for (int j = 0; j < kFD; ++j) {
        if (tid == 0) Gm[j * kLdS + j] = sqrtf(fmaxf(Gm[j * kLdS + j], 1e-30f));
        __syncthreads();
        const float d = Gm[j * kLdS + j];
        for (int i = j + 1 + tid; i < kFD; i += 256) Gm[i * kLdS + j] /= d;
        __syncthreads();
        for (int i = j + 1 + ty; i < kFD; i += 16) {
            const float lij = Gm[i * kLdS + j];
            for (int k = j + 1 + tx; k <= i; k += 16) Gm[i * kLdS + k] -= lij * Gm[k * kLdS + j];
        }
        __syncthreads();
    }
    // L u = r, then L^T z = u, for the CTA's columns: right-looking, a row's
    // value fixed by its division, then subtracted from the rows it feeds
    for (int i = 0; i < kFD; ++i) {
        if (tid < kSolveCols) Rm[i * kLdR + tid] /= Gm[i * kLdS + i];
        __syncthreads();
        for (int e = tid; e < (kFD - 1 - i) * kSolveCols; e += 256) {
            const int k = i + 1 + e / kSolveCols, c = e % kSolveCols;
            Rm[k * kLdR + c] -= Gm[k * kLdS + i] * Rm[i * kLdR + c];
        }
        __syncthreads();
    }
    for (int i = kFD - 1; i >= 0; --i) {
        if (tid < kSolveCols) Rm[i * kLdR + tid] /= Gm[i * kLdS + i];
        __syncthreads();
        for (int e = tid; e < i * kSolveCols; e += 256) {
            const int k = e / kSolveCols, c = e % kSolveCols;
            Rm[k * kLdR + c] -= Gm[i * kLdS + k] * Rm[i * kLdR + c];
        }
        __syncthreads();
    }
    // B[o][i] = z_o[i]
    for (int e = tid; e < kSolveCols * kFD; e += 256) {
        const int c = e >> 7, i = e & 127;
        Bh[(int64_t)(o0 + c) * kFD + i] = __bfloat16_as_ushort(__float2bfloat16_rn(Rm[i * kLdR + c]));
    }
}

}  // namespace

// partial sums [H][kFBlocks][chunks][128][128], then their totals [H][kFBlocks][128][128]
size_t coral_fit_part_bytes(int H, int64_t n_tokens) {
    const int64_t chunks = (n_tokens + kFitChunkTokens - 1) / kFitChunkTokens;
    return (size_t)H * kFBlocks * (size_t)((chunks > 0 ? chunks : 1) + 1) * kFD * kFD * sizeof(float);
}

cudaError_t launch_coral_fit(const uint16_t* xh, const uint16_t* y, const uint16_t* t2, const uint16_t* U,
                             int64_t n_tokens, int H, float* part, uint16_t* B, cudaStream_t s) {
    const int chunks = (int)((n_tokens + kFitChunkTokens - 1) / kFitChunkTokens);
    GramArgs ga{xh, y, t2, n_tokens, H, chunks, part};
    const size_t gsmem = sizeof(uint16_t) * 2 * kGramStages * kFStep * kLdX;
    cudaError_t ge = cudaFuncSetAttribute(coral_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gsmem);
    if (ge != cudaSuccess) return ge;
    coral_gram_kernel<<<dim3((unsigned)chunks, kFBlocks, (unsigned)H), 256, gsmem, s>>>(ga);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    float* red = part + (size_t)H * kFBlocks * chunks * kFD * kFD;
    const int64_t total = (int64_t)H * kFBlocks * kFD * kFD;
    coral_gram_reduce_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(part, chunks, total, red);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t smem = sizeof(float) * (kFD * kLdS + kFD * kLdR + kFD * 64 + kSolveCols * kFR);
    e = cudaFuncSetAttribute(coral_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    SolveArgs sa{red, U, H, B};
    coral_solve_kernel<<<dim3(kFD / kSolveCols, (unsigned)H), 256, smem, s>>>(sa);
    return cudaGetLastError();
}

}  // namespace qvg
