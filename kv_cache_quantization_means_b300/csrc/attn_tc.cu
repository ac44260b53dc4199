// Attention over a compressed K/V history on the tensor cores, staged by
// groups of heads (Quant VideoGen explainer, sec. 3, key contributions: fused
// dequantisation kernels; the 33-method Self-Forcing KV-cache study,
// abstract: integrations that rebuild full BF16 K/V buffers around attention
// lose the memory that compression saved).
//
// Same result definition as the in-CTA fused kernel (attn.cu):
//   s_n = scale * <q_i, k_hat_n>,  o_i = sum_n exp(s_n) v_hat_n / sum_n exp(s_n),
// with k_hat, v_hat the decoder's bf16 rows bit for bit, bf16 products with
// fp32 sums, fp32 online softmax, probabilities rounded to bf16 for the
// product with v_hat, fp32 output.
//
// Decoding every key tile once per 128-query tile would cost as much as the
// products (a decoded row is about a dozen instructions per element, against
// 4 * 128 flop per element spread over the tensor cores).  So each key row is
// decoded once per head: a group of up to four heads is decoded into a
// working buffer -- K as rows [n][D], V transposed as [D][n], 2 x 4 x n x D
// bf16, small enough to stay in L2 -- and the attention kernel reads its
// tiles from there; then the next group reuses the buffer.  No bf16 K/V of the
// whole history is ever formed.
//
// Attention kernel: one CTA per (head, 128 queries), 2 + 4 kFaNG warps.
//   warp 0   bulk tensor copies: the query tile once, then per 128-key tile
//            the K tile (one lane, a ring of three) and the V^T tile (another
//            lane, a ring of two); a K tile is released when its scores are
//            computed, a V^T tile when its product is;
//   warp 1   tcgen05.mma issuer: S_j = Q K_j^T into one of two tensor-memory
//            score buffers (128 x 128 fp32), then O += P_{j-1} V_{j-1} into
//            the output accumulator (128 x D fp32), P from shared memory;
//   the other warps softmax: the kFaNG warps on a tensor-memory lane quadrant
//            take 128 / kFaNG of each row's columns each and trade the row maximum
//            through shared memory.  Scores in base-2 units t = RN(s c),
//            c = scale log2(e); the running maximum m and sum l; p =
//            exp2(t - m) (ex2.approx, subnormals flushed) rounded to bf16
//            into P.  The maximum is only raised when a tile's exceeds it by
//            more than 8 (a factor 2^8), and then O is rescaled in tensor
//            memory; otherwise the stale m keeps every p below 2^8, which
//            changes no rounding (powers of two) and cannot overflow.  Each
//            group sums its p in four partial sums into its own l; the
//            groups' l are added at the end.
// Every wait is bounded; a wait that runs out records 0x7E000000 in the
// library's device error word, the roles drain what they issued and return.
#include <math.h>

#include "attn.h"
#include "common.cuh"
#include "kernels.h"
#include "prq16.cuh"
#include "tc_common.cuh"

namespace qvg {

namespace {

constexpr int kFaQ = 128;                 // queries per CTA
constexpr int kFaK = 128;                 // keys per tile
constexpr int kFaNG = 2;                  // softmax column groups: each row's S and O columns split in kFaNG parts
constexpr int kFaSoftWarps = 4 * kFaNG;
constexpr int kFaThreads = 32 * (2 + kFaSoftWarps);   // warp 0 copies, warp 1 MMA, the rest softmax
constexpr uint32_t kFaAtom = 128u * 128u; // one 64-element slab of 128 rows, 128-byte swizzle
constexpr uint32_t kFaErrTimeout = 0x7E000000u;
constexpr int kStageRows = 64;            // rows per CTA of the staging decode

// shared memory map (offsets from the 1024-byte aligned base): Q, a ring of
// kFaKS K tiles and one of kFaVS V^T tiles (K_j is released as soon as S_j
// has been computed, V_j after O += P_j V_j), P, barriers, exchange words
constexpr int kFaKS = 3, kFaVS = 2;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = 2 * kFaAtom;
constexpr uint32_t kOffV = kOffK + kFaKS * 2 * kFaAtom;
constexpr uint32_t kOffP = kOffV + kFaVS * 2 * kFaAtom;
constexpr uint32_t kOffBar = kOffP + 2 * kFaAtom;
constexpr uint32_t kOffMisc = kOffBar + 160;
constexpr uint32_t kOffX = kOffMisc + 16;                      // row maxima / sums / flags traded by the groups
constexpr uint32_t kFaSmem = kOffX + kFaNG * 128 * 4 + 2 * kFaNG * 128 + 1024;   // + alignment slack
static_assert(kFaSmem <= 232448, "shared memory of one CTA");

struct FaArgs {
    int64_t n_queries, n_keys;
    int h0;                          // first head of the group (query and output rows)
    float* out;
    int64_t out_head_stride, out_token_stride;
    float scale_log2;
    int q_head_inner;                // query map dims (D, H, N) rather than (D, N, H)
    CodecCtl ctl;
};

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2^x by the hardware approximation (ex2.approx, subnormal results flushed
// to zero: a probability below 2^-126 weighs nothing next to the row's
// largest, which is at least 1).
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// bf16 of lo in the low half, of hi in the high half (round to nearest even)
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// ------------------------------------------------------- staging decode
//
// Rows [n0, n0 + 64) of head h0 + blockIdx.y: K to kscr[hh][n][D], V
// transposed to vscr[hh][d][npad] through a shared-memory tile.
struct StageArgs {
    const uint32_t *k_codes, *k_meta, *v_codes, *v_meta;
    const uint8_t *k_ids, *v_ids;
    const uint16_t *k_cent, *v_cent;
    int64_t cap, n_keys, npad;
    int H, C, S, G, h0;
    uint16_t *kscr, *vscr;
};

// A thread's four items (16 channels of a row: two of K, two of V) have all
// their loads in flight at once: the ids first, then every centroid chunk,
// code word and scale/zero word, then the arithmetic of decode_chunk.
template <int D, int B, int S>
__global__ void __launch_bounds__(256) attn_stage_kernel(StageArgs a) {
    constexpr int CPR = D / 16, LD = D + 8, WPT = B / 2, WPR = D * B / 32;
    constexpr int PER = kStageRows * CPR;                 // items per tensor
    constexpr int IT = 2 * PER / 256;                     // items per thread
    static_assert(2 * PER % 256 == 0 && PER % 256 == 0, "whole items per thread, K before V");
    __shared__ __align__(16) uint16_t vt[kStageRows * LD];
    const int tid = threadIdx.x, hh = blockIdx.y, h = a.h0 + hh;
    const int64_t n0 = (int64_t)blockIdx.x * kStageRows;
    const int64_t stage_rows = (int64_t)a.H * a.cap;
    const int mpr = D / a.G;
    int64_t row[IT];
    int rr[IT], cc[IT], id[IT];
    bool valid[IT];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const bool is_v = it >= IT / 2;
        const int j = tid + 256 * (is_v ? it - IT / 2 : it);
        rr[it] = j / CPR;
        cc[it] = j % CPR;
        valid[it] = n0 + rr[it] < a.n_keys;
        row[it] = (int64_t)h * a.cap + n0 + rr[it];
        id[it] = (a.C > 0 && valid[it]) ? (is_v ? a.v_ids : a.k_ids)[row[it]] : 0;
    }
    uint4 c0[IT], c1[IT];
    uint32_t cw[IT][S][WPT], mw[IT][S];
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const bool is_v = it >= IT / 2;
        const uint32_t* codes = is_v ? a.v_codes : a.k_codes;
        const uint32_t* meta = is_v ? a.v_meta : a.k_meta;
        c0[it] = c1[it] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int s = 0; s < S; ++s) {
#pragma unroll
            for (int w = 0; w < WPT; ++w) cw[it][s][w] = 0;
            mw[it][s] = 0;
        }
        if (!valid[it]) continue;
        if (a.C > 0) {
            const uint16_t* cr = (is_v ? a.v_cent : a.k_cent) + ((int64_t)h * a.C + min(id[it], a.C - 1)) * D + cc[it] * 16;
            c0[it] = __ldg(reinterpret_cast<const uint4*>(cr));
            c1[it] = __ldg(reinterpret_cast<const uint4*>(cr + 8));
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t srow = (int64_t)s * stage_rows + row[it];
#pragma unroll
            for (int w = 0; w < WPT; ++w) cw[it][s][w] = __ldg(codes + srow * WPR + cc[it] * WPT + w);
            mw[it][s] = __ldg(meta + srow * mpr + (cc[it] * 16) / a.G);
        }
    }
#pragma unroll
    for (int it = 0; it < IT; ++it) {
        const bool is_v = it >= IT / 2;
        float acc[16];
        if (a.C > 0) {
            unpack16(c0[it], c1[it], acc);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        }
#pragma unroll
        for (int s = 0; s < S; ++s) {
            if constexpr (B == 2) {
                dequant_add16(acc, cw[it][s][0], mw[it][s]);
            } else {
                dequant_add8x4(acc, cw[it][s][0], mw[it][s]);
                dequant_add8x4(acc + 8, cw[it][s][1], mw[it][s]);
            }
        }
        uint4 o0 = make_uint4(0, 0, 0, 0), o1 = o0;
        if (valid[it]) pack16_bf16(acc, o0, o1);
        if (is_v) {
            *reinterpret_cast<uint4*>(vt + rr[it] * LD + 16 * cc[it]) = o0;
            *reinterpret_cast<uint4*>(vt + rr[it] * LD + 16 * cc[it] + 8) = o1;
        } else if (valid[it]) {
            uint16_t* kr = a.kscr + ((int64_t)hh * a.npad + n0 + rr[it]) * D + 16 * cc[it];
            *reinterpret_cast<uint4*>(kr) = o0;
            *reinterpret_cast<uint4*>(kr + 8) = o1;
        }
    }
    __syncthreads();
    // V^T: channel d, tokens n0 + 8u .. n0 + 8u + 7 per 16-byte store
    for (int it = tid; it < D * (kStageRows / 8); it += 256) {
        const int d = it / (kStageRows / 8), u = it % (kStageRows / 8);
        if (n0 + 8 * u >= a.npad) continue;
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = (uint32_t)vt[(8 * u + 2 * k) * LD + d] | ((uint32_t)vt[(8 * u + 2 * k + 1) * LD + d] << 16);
        *reinterpret_cast<uint4*>(a.vscr + ((int64_t)hh * D + d) * a.npad + n0 + 8 * u) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <int B>
cudaError_t launch_stage(const StageArgs& sa, dim3 grid, cudaStream_t s) {
    switch (sa.S) {
        case 1: attn_stage_kernel<128, B, 1><<<grid, 256, 0, s>>>(sa); break;
        case 2: attn_stage_kernel<128, B, 2><<<grid, 256, 0, s>>>(sa); break;
        case 3: attn_stage_kernel<128, B, 3><<<grid, 256, 0, s>>>(sa); break;
        case 4: attn_stage_kernel<128, B, 4><<<grid, 256, 0, s>>>(sa); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// ------------------------------------------------------- attention kernel

__global__ void __launch_bounds__(kFaThreads, 1)
    attn_fa_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, FaArgs a) {
    extern __shared__ __align__(1024) uint8_t fa_smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(fa_smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sQ = smem_u32(base + kOffQ), sK = smem_u32(base + kOffK), sV = smem_u32(base + kOffV),
                   sP = smem_u32(base + kOffP);
    uint8_t* P = base + kOffP;
    const uint32_t bar0 = smem_u32(base + kOffBar);
    const uint32_t q_full = bar0, k_full = bar0 + 8, k_empty = k_full + 8 * kFaKS, v_full = k_empty + 8 * kFaKS,
                   v_empty = v_full + 8 * kFaVS, s_full = v_empty + 8 * kFaVS, s_free = s_full + 16,
                   p_full = s_free + 16, pv_done = p_full + 8;
    uint32_t* misc = reinterpret_cast<uint32_t*>(base + kOffMisc);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hh = blockIdx.y, h = a.h0 + hh;
    const int64_t q0 = (int64_t)blockIdx.x * kFaQ;
    const int nkt = (int)((a.n_keys + kFaK - 1) / kFaK);
    const unsigned long long lim = a.ctl.limit;

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int st = 0; st < kFaKS; ++st) {
            mbar_init(k_full + 8 * st, 1);
            mbar_init(k_empty + 8 * st, 1);
        }
        for (int st = 0; st < kFaVS; ++st) {
            mbar_init(v_full + 8 * st, 1);
            mbar_init(v_empty + 8 * st, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + 8 * b, 1);
            mbar_init(s_free + 8 * b, kFaSoftWarps);
        }
        mbar_init(p_full, kFaSoftWarps);
        mbar_init(pv_done, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(misc)), "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ------------------------------------------------ copies: lane 0 Q and K, lane 1 V^T
        if (lane == 0) {
            mbar_arrive_tx(q_full, 2 * kFaAtom);
            for (int at = 0; at < 2; ++at) {
                if (a.q_head_inner) tma_load_3d(sQ + at * kFaAtom, &qmap, q_full, 64 * at, h, (int)q0);
                else tma_load_3d(sQ + at * kFaAtom, &qmap, q_full, 64 * at, (int)q0, h);
            }
            int armed = 0;
            for (int j = 0; j < nkt; ++j) {
                const int st = j % kFaKS;
                if (!mbar_wait(k_empty + 8 * st, ((uint32_t)(j / kFaKS) & 1u) ^ 1u, lim)) { atomicExch(misc + 1, 1u); break; }
                if (*(volatile uint32_t*)(misc + 1)) break;
                const uint32_t dst = sK + (uint32_t)st * 2 * kFaAtom;
                mbar_arrive_tx(k_full + 8 * st, 2 * kFaAtom);
                for (int at = 0; at < 2; ++at) tma_load_3d(dst + at * kFaAtom, &kmap, k_full + 8 * st, 64 * at, j * kFaK, hh);
                armed = j + 1;
            }
            // drain: every copy issued has landed before exit
            mbar_wait(q_full, 0u, lim);
            for (int j = armed - kFaKS > 0 ? armed - kFaKS : 0; j < armed; ++j)
                mbar_wait(k_full + 8 * (j % kFaKS), (uint32_t)(j / kFaKS) & 1u, lim);
        } else if (lane == 1) {
            int armed = 0;
            for (int j = 0; j < nkt; ++j) {
                const int st = j % kFaVS;
                if (!mbar_wait(v_empty + 8 * st, ((uint32_t)(j / kFaVS) & 1u) ^ 1u, lim)) { atomicExch(misc + 1, 1u); break; }
                if (*(volatile uint32_t*)(misc + 1)) break;
                const uint32_t dst = sV + (uint32_t)st * 2 * kFaAtom;
                mbar_arrive_tx(v_full + 8 * st, 2 * kFaAtom);
                for (int at = 0; at < 2; ++at)
                    tma_load_3d(dst + at * kFaAtom, &vmap, v_full + 8 * st, j * kFaK + 64 * at, 0, hh);
                armed = j + 1;
            }
            for (int j = armed - kFaVS > 0 ? armed - kFaVS : 0; j < armed; ++j)
                mbar_wait(v_full + 8 * (j % kFaVS), (uint32_t)(j / kFaVS) & 1u, lim);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kFaK >> 3) << 17) |
                                   ((uint32_t)(kFaQ >> 4) << 24);
            uint32_t last_bar = 0, last_ph = 0;
            bool ok = mbar_wait(q_full, 0u, lim);
            for (int j = 0; ok && j <= nkt; ++j) {
                if (j < nkt) {
                    const int st = j % kFaKS, b = j & 1;
                    if (!(ok = mbar_wait(k_full + 8 * st, (uint32_t)(j / kFaKS) & 1u, lim))) break;
                    if (!(ok = mbar_wait(s_free + 8 * b, ((uint32_t)(j >> 1) & 1u) ^ 1u, lim))) break;
                    if (*(volatile uint32_t*)(misc + 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t kb = sK + (uint32_t)st * 2 * kFaAtom;
#pragma unroll
                    for (int at = 0; at < 2; ++at)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_bf16(tmem + 128u * b, sw128_desc(sQ + at * kFaAtom + 32u * k),
                                      sw128_desc(kb + at * kFaAtom + 32u * k), idesc, (at | k) ? 1u : 0u);
                    umma_commit(s_full + 8 * b);
                    umma_commit(k_empty + 8 * st);
                    last_bar = s_full + 8 * b;
                    last_ph = (uint32_t)(j >> 1) & 1u;
                }
                if (j >= 1) {
                    const int jj = j - 1, st = jj % kFaVS;
                    if (!(ok = mbar_wait(v_full + 8 * st, (uint32_t)(jj / kFaVS) & 1u, lim))) break;
                    if (!(ok = mbar_wait(p_full, (uint32_t)jj & 1u, lim))) break;
                    if (*(volatile uint32_t*)(misc + 1)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t vb = sV + (uint32_t)st * 2 * kFaAtom;
#pragma unroll
                    for (int at = 0; at < 2; ++at)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_bf16(tmem + 256u, sw128_desc(sP + at * kFaAtom + 32u * k),
                                      sw128_desc(vb + at * kFaAtom + 32u * k), idesc, (jj | at | k) ? 1u : 0u);
                    umma_commit(pv_done);
                    umma_commit(v_empty + 8 * st);
                    last_bar = pv_done;
                    last_ph = (uint32_t)jj & 1u;
                }
            }
            if (!ok) atomicExch(misc + 1, 1u);
            // drain: the last commit arrives once every MMA issued has completed
            if (last_bar) mbar_wait(last_bar, last_ph, lim);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax
        // row = tensor-memory lane; the kFaNG warps on a row's quadrant take
        // CW of its S columns (keys) and of its O columns (channels) each.
        // They trade their maxima (at the end their sums) through shared
        // memory, so all keep the same m, and with them whether their waits
        // succeeded, so that all leave the loop at the same point.
        constexpr int CW = kFaK / kFaNG;
        static_assert(CW % 32 == 0, "whole 32-column tensor-memory loads per group");
        const int grp = (warp - 2) >> 2, quad = warp & 3;
        const int row = 32 * quad + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
        float* xch = reinterpret_cast<float*>(base + kOffX);                    // [grp][row]
        uint8_t* xok1 = base + kOffX + kFaNG * 128 * 4;                         // [grp][row]
        uint8_t* xok2 = xok1 + kFaNG * 128;
        auto group_sync = [&]() { asm volatile("bar.sync %0, %1;" ::"r"(1 + quad), "r"(32 * kFaNG) : "memory"); };
        auto all_ok = [&](const uint8_t* f) {
            bool r = true;
#pragma unroll
            for (int g = 0; g < kFaNG; ++g) r = r && f[g * 128 + row];
            return r;
        };
        // one lane probes the barrier, the warp follows (__syncwarp orders the
        // other lanes' reads after that lane's acquiring wait)
        auto warp_wait = [&](uint32_t bar, uint32_t parity) -> bool {
            uint32_t r = 0;
            if (lane == 0) r = mbar_wait(bar, parity, lim) ? 1u : 0u;
            r = __shfl_sync(0xffffffffu, r, 0);
            __syncwarp();
            return r != 0;
        };
        const float c2 = a.scale_log2;
        float m = -INFINITY, l = 0.0f;
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            const int b = j & 1;
            uint32_t s[CW];
            float e0 = 0.0f;
            bool okw = warp_wait(s_full + 8 * b, (uint32_t)(j >> 1) & 1u);
            if (okw) {
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < CW / 32; ++c) tmem_ld32(trow + 128u * b + (uint32_t)(CW * grp + 32 * c), s + 32 * c);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free + 8 * b);
                // keys past n_keys (last tile only) take the score that maps to -inf
                if (j == nkt - 1) {
                    const int64_t k0 = (int64_t)j * kFaK + CW * grp;
#pragma unroll
                    for (int c = 0; c < CW; ++c)
                        if (k0 + c >= a.n_keys) s[c] = __float_as_uint(c2 >= 0.0f ? -INFINITY : INFINITY);
                }
                // the group's extreme raw score (four chains), then in base-2 units
                float x4[4] = {__uint_as_float(s[0]), __uint_as_float(s[1]), __uint_as_float(s[2]),
                               __uint_as_float(s[3])};
                if (c2 >= 0.0f) {
#pragma unroll
                    for (int c = 4; c < CW; c += 8)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            x4[q] = c + 2 * q + 1 < CW ? fmax3(x4[q], __uint_as_float(s[c + 2 * q]), __uint_as_float(s[c + 2 * q + 1]))
                                                       : x4[q];
                    e0 = fmaxf(fmaxf(x4[0], x4[1]), fmaxf(x4[2], x4[3]));
                } else {
#pragma unroll
                    for (int c = 4; c < CW; c += 8)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            x4[q] = c + 2 * q + 1 < CW ? fmin3(x4[q], __uint_as_float(s[c + 2 * q]), __uint_as_float(s[c + 2 * q + 1]))
                                                       : x4[q];
                    e0 = fminf(fminf(x4[0], x4[1]), fminf(x4[2], x4[3]));
                }
            }
            xch[grp * 128 + row] = e0 * c2;
            xok1[grp * 128 + row] = okw ? 1 : 0;
            group_sync();
            if (!all_ok(xok1)) { ok = false; break; }
            float mx = xch[row];
#pragma unroll
            for (int g = 1; g < kFaNG; ++g) mx = fmaxf(mx, xch[g * 128 + row]);
            const float m_new = fmaxf(m, mx);
            // P and O are free once the previous product has completed
            okw = j == 0 || warp_wait(pv_done, (uint32_t)(j - 1) & 1u);
            if (okw) {
                tc_fence_after();
                if (__any_sync(0xffffffffu, m_new > m + 8.0f)) {
                    const bool raise = m_new > m + 8.0f;
                    const float alpha = raise ? exp2f(m - m_new) : 1.0f;
                    if (j >= 1) {
#pragma unroll
                        for (int c = 0; c < CW / 32; ++c) {
                            uint32_t o[32];
                            tmem_ld32(trow + 256u + (uint32_t)(CW * grp + 32 * c), o);
                            tmem_wait_ld_regs(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st32(trow + 256u + (uint32_t)(CW * grp + 32 * c), o);
                        }
                        tmem_wait_st();
                    }
                    if (raise) {
                        l *= alpha;
                        m = m_new;
                    }
                }
                // p = exp2(RN(s * c2) - m) (the row's largest score gives exactly
                // 1), summed in four partial sums, rounded to bf16 into P
                // (packed pairs: each lane of an fp32x2 operation rounds as the scalar one)
                const float2 c22 = make_float2(c2, c2), m2 = make_float2(m, m);
                float2 ps2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
                for (int c8 = 0; c8 < CW / 8; ++c8) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 t = f2_sub(f2_mul(make_float2(__uint_as_float(s[8 * c8 + 2 * e]),
                                                                   __uint_as_float(s[8 * c8 + 2 * e + 1])),
                                                       c22),
                                                m2);
                        const float2 p = make_float2(ex2_ftz(t.x), ex2_ftz(t.y));
                        ps2[e & 1] = f2_add(ps2[e & 1], p);
                        w[e] = cvt_bf16x2(p.x, p.y);
                    }
                    *reinterpret_cast<uint4*>(P + sw_off(row, CW * grp + 8 * c8, kFaAtom)) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                l += (ps2[0].x + ps2[1].x) + (ps2[0].y + ps2[1].y);
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full);
            }
            xok2[grp * 128 + row] = okw ? 1 : 0;
            group_sync();                     // also: the maxima are read before the next tile overwrites them
            if (!all_ok(xok2)) { ok = false; break; }
        }
        if (ok) ok = warp_wait(pv_done, (uint32_t)(nkt - 1) & 1u);
        // every group of a row reaches this trade (they leave the loop together)
        xch[grp * 128 + row] = ok ? l : -1.0f;
        group_sync();
        float lsum = 0.0f;
        bool good = ok;
#pragma unroll
        for (int g = 0; g < kFaNG; ++g) {
            const float v = xch[g * 128 + row];
            good = good && v >= 0.0f;
            lsum += v;
        }
        if (!good) {
            if (lane == 0) atomicExch(misc + 1, 1u);
        } else {
            tc_fence_after();
            const int64_t qi = q0 + row;
            const float inv = 1.0f / lsum;
            float* orow = a.out + (int64_t)h * a.out_head_stride + qi * a.out_token_stride + CW * grp;
#pragma unroll
            for (int c = 0; c < CW / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(trow + 256u + (uint32_t)(CW * grp + 32 * c), o);
                tmem_wait_ld_regs(o);
                if (qi < a.n_queries)
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(orow + 32 * c + e) =
                            make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                        __uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && misc[1] && a.ctl.err) atomicExch(a.ctl.err, kFaErrTimeout);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    }
}

bool encode_map(CUtensorMap* map, const void* ptr, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t attention_staged_bytes(int D, int H, int64_t n_keys) {
    const int64_t npad = (n_keys + 7) / 8 * 8;
    const int hg = H < kAttnGroupHeads ? H : kAttnGroupHeads;
    return (size_t)2 * hg * (size_t)npad * D * sizeof(uint16_t);
}

cudaError_t launch_attention_staged(int D, const AttnArgs& a, void* ws, size_t ws_bytes, bool* launched,
                                    cudaStream_t s) {
    *launched = false;
    if (D != 128 || a.n_queries == 0 || !ws || ws_bytes < attention_staged_bytes(D, a.H, a.n_keys)) return cudaSuccess;
    if (!(a.bits == 2 || a.bits == 4) || a.S < 1 || a.S > 4) return cudaSuccess;
    if (a.n_keys > (int64_t)INT32_MAX - kFaK || a.n_queries > (int64_t)INT32_MAX - kFaQ) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) || (reinterpret_cast<uintptr_t>(a.q) & 15u)) return cudaSuccess;
    CodecCtl ctl;
    if (!codec_ctl(&ctl)) return cudaSuccess;
    const int64_t npad = (a.n_keys + 7) / 8 * 8;
    const int hg_max = a.H < kAttnGroupHeads ? a.H : kAttnGroupHeads;
    uint16_t* kscr = static_cast<uint16_t*>(ws);
    uint16_t* vscr = kscr + (size_t)hg_max * npad * D;

    // the query map: dims innermost first, the token and head dimensions in stride order
    CUtensorMap qmap, kmap, vmap;
    const bool head_inner = a.q_head_stride <= a.q_token_stride;
    {
        cuuint64_t dims[3], strides[2];
        cuuint32_t box[3];
        dims[0] = (cuuint64_t)D;
        if (head_inner) {
            dims[1] = (cuuint64_t)a.H; dims[2] = (cuuint64_t)a.n_queries;
            strides[0] = (cuuint64_t)a.q_head_stride * 2; strides[1] = (cuuint64_t)a.q_token_stride * 2;
            box[0] = 64; box[1] = 1; box[2] = kFaQ;
        } else {
            dims[1] = (cuuint64_t)a.n_queries; dims[2] = (cuuint64_t)a.H;
            strides[0] = (cuuint64_t)a.q_token_stride * 2; strides[1] = (cuuint64_t)a.q_head_stride * 2;
            box[0] = 64; box[1] = kFaQ; box[2] = 1;
        }
        if (a.H == 1) {
            if (head_inner) strides[0] = (cuuint64_t)D * 2;
            else strides[1] = strides[0] * (cuuint64_t)a.n_queries;
        }
        if (!encode_map(&qmap, a.q, dims, strides, box)) return cudaSuccess;
    }
    {
        // K rows of the group: (D, n_keys, heads), row stride D, head stride npad * D
        const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.n_keys, (cuuint64_t)hg_max};
        const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)npad * D * 2};
        const cuuint32_t box[3] = {64, kFaK, 1};
        if (!encode_map(&kmap, kscr, dims, strides, box)) return cudaSuccess;
    }
    {
        // V^T of the group: (n_keys, D, heads), row stride npad, head stride D * npad
        const cuuint64_t dims[3] = {(cuuint64_t)a.n_keys, (cuuint64_t)D, (cuuint64_t)hg_max};
        const cuuint64_t strides[2] = {(cuuint64_t)npad * 2, (cuuint64_t)D * npad * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)D, 1};
        if (!encode_map(&vmap, vscr, dims, strides, box)) return cudaSuccess;
    }
    cudaError_t e = cudaFuncSetAttribute(attn_fa_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFaSmem);
    if (e != cudaSuccess) return e;

    StageArgs sa;
    sa.k_codes = a.k_codes; sa.k_meta = a.k_meta; sa.v_codes = a.v_codes; sa.v_meta = a.v_meta;
    sa.k_ids = a.k_ids; sa.v_ids = a.v_ids; sa.k_cent = a.k_cent; sa.v_cent = a.v_cent;
    sa.cap = a.cap; sa.n_keys = a.n_keys; sa.npad = npad;
    sa.H = a.H; sa.C = a.C; sa.S = a.S; sa.G = a.G;
    sa.kscr = kscr; sa.vscr = vscr;
    FaArgs fa;
    fa.n_queries = a.n_queries; fa.n_keys = a.n_keys;
    fa.out = a.out; fa.out_head_stride = a.out_head_stride; fa.out_token_stride = a.out_token_stride;
    fa.scale_log2 = a.scale_log2;
    fa.q_head_inner = head_inner ? 1 : 0;
    fa.ctl = ctl;
    for (int h0 = 0; h0 < a.H; h0 += hg_max) {
        const int hg = a.H - h0 < hg_max ? a.H - h0 : hg_max;
        sa.h0 = h0;
        const dim3 sgrid((unsigned)((a.n_keys + kStageRows - 1) / kStageRows), (unsigned)hg);
        e = a.bits == 2 ? launch_stage<2>(sa, sgrid, s) : launch_stage<4>(sa, sgrid, s);
        if (e != cudaSuccess) return e;
        fa.h0 = h0;
        const dim3 grid((unsigned)((a.n_queries + kFaQ - 1) / kFaQ), (unsigned)hg);
        attn_fa_kernel<<<grid, kFaThreads, kFaSmem, s>>>(qmap, kmap, vmap, fa);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    *launched = true;
    return cudaSuccess;
}

}  // namespace qvg
