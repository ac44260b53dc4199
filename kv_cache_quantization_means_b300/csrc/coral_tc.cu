// Coral-KV cross-layer prediction on the 5th-generation tensor cores (sm_103a).
//
// Coral-KV news items, section "cross-layer prediction": layer l+1 is
// predicted from the reconstruction of layer l by a block-DPLR map -- a dense
// D x D block per head plus one global rank-R term -- and only the residual
// is quantised.  Per layer (one tensor, N tokens, H heads of D = 128, R = 32):
//
//  prep       Wt = W^T ([R][H*D]) and Ud = [U | U] ([H*D][2R]), bf16, so every
//             GEMM operand is K-major with 128-byte rows.
//  lowrank    t = xhat W: one CTA per 128-token tile streams the H*D/64
//             channel slabs of xhat and Wt through TMA into shared memory;
//             tcgen05.mma accumulates the [128 x 32] fp32 result in TMEM;
//             the epilogue stores t as a bf16 pair (hi, lo = t - hi), i.e. a
//             [128 x 64] K-major operand that keeps ~16 significant bits.
//  predict    persistent CTAs over (token tile, head) items: TMA brings
//             xhat_h (128 x 128), B_h (128 x 128), t (128 x 64) and Ud_h
//             (128 x 64); 8 + 4 MMAs (K = 16) form
//                 pred = xhat_h B_h^T + t_hi U_h^T + t_lo U_h^T
//             in one of two TMEM accumulators; two epilogue groups of four
//             warps drain them, a thread per token row, 32 channels (or one
//             64-channel group) at a time: encode subtracts pred from x_{l+1}, runs the same
//             per-thread PRQ stages as the other kernels and writes codes,
//             scale/zero words and x_hat_{l+1} = bf16(((pred + d_1) + d_2)..);
//             decode rebuilds x_hat_{l+1} from the codes.  Encoder and decoder
//             run the identical prediction, so their reconstructions agree
//             bit for bit.  Two decoder forms serve the Coral + SAS hybrid:
//             S = 0 stores the prediction alone, and with the residual's ids
//             and centroids the stages code a k-means-smoothed residual,
//             x_hat_{l+1} = bf16(pred + bf16(c[id] + d_1 + d_2 ..)).
// Every wait is a bounded mbarrier wait; on expiry the kernel records an
// error code, drains its own copies and MMAs and frees its tensor memory.
#include "common.cuh"
#include "kernels.h"
#include "prq16.cuh"
#include "tc_common.cuh"

namespace qvg {

namespace {

constexpr int kT = 128;                 // tokens per tile (UMMA M)
constexpr int kR = 32;                  // rank handled here
constexpr int kDh = 128;                // head dim handled here
constexpr int kSlab = kT * 128;         // one [128 x 64] bf16 operand slab, bytes
constexpr uint32_t kErrTimeout = 0x7E000000u;

// ------------------------------------------------------------------ prep

// W [H*D][32] -> Wt [32][H*D] and U [H*D][32] -> Ud [H*D][64] = [U | U].  A
// CTA takes kPrepRows channel rows: W and U are read along their rows and Ud
// written along its rows (coalesced); Wt, the transpose, goes out through a
// shared tile so that its rows are written along too.
constexpr int kPrepRows = 32;

__global__ void __launch_bounds__(256) coral_prep_kernel(const uint16_t* W, const uint16_t* U, int HD, uint16_t* Wt,
                                                         uint16_t* Ud) {
    __shared__ uint16_t tile[kR][kPrepRows + 2];
    const int j0 = blockIdx.x * kPrepRows, tid = threadIdx.x;
    for (int e = tid; e < kPrepRows * kR; e += 256) {
        const int jr = e / kR, r = e % kR, j = j0 + jr;
        if (j < HD) {
            tile[r][jr] = W[(int64_t)j * kR + r];
            const uint16_t u = U[(int64_t)j * kR + r];
            Ud[(int64_t)j * 2 * kR + r] = u;
            Ud[(int64_t)j * 2 * kR + kR + r] = u;
        }
    }
    __syncthreads();
    for (int e = tid; e < kR * kPrepRows; e += 256) {
        const int r = e / kPrepRows, jr = e % kPrepRows, j = j0 + jr;
        if (j < HD) Wt[(int64_t)r * HD + j] = tile[r][jr];
    }
}

// --------------------------------------------------------------- lowrank

constexpr int kLrStages = 8;
constexpr int kLrThreads = 64 + 128;    // TMA warp, MMA warp, 4 epilogue warps

struct LrArgs {
    int64_t n_tokens;
    int HD;
    uint16_t* t2;          // [N][64] bf16: t_hi | t_lo
    uint32_t* err;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__global__ void __launch_bounds__(kLrThreads, 1)
    coral_lowrank_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                            LrArgs a) {
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, derived from the shared array so that accesses stay in
    // the shared window
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    constexpr int kWBytes = kR * 128;                   // Wt slab [32 x 64]
    uint8_t* Xs = base;                                  // kLrStages x [128 x 64]
    uint8_t* Ws = base + kLrStages * kSlab;              // kLrStages x [32 x 64]
    const uint32_t bar0 = smem_u32(base + kLrStages * (kSlab + kWBytes));
    const uint32_t full_bar = bar0, empty_bar = bar0 + 8 * kLrStages, done_bar = bar0 + 16 * kLrStages;
    uint32_t* misc = reinterpret_cast<uint32_t*>(base + kLrStages * (kSlab + kWBytes) + 8 * (2 * kLrStages + 1));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tok0 = blockIdx.x * kT;
    const int nk = a.HD / 64;
    if (tid == 0) {
        for (int s = 0; s < kLrStages; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, 1);
        }
        mbar_init(done_bar, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(misc)),
                     "r"(32u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    if (warp == 0) {
        if (lane == 0) {
            int armed = 0;
            for (int k = 0; k < nk; ++k) {
                const int s = k % kLrStages;
                if (!mbar_wait(empty_bar + 8 * s, ((uint32_t)(k / kLrStages) & 1u) ^ 1u)) { misc[1] = 1; break; }
                mbar_arrive_tx(full_bar + 8 * s, (uint32_t)(kSlab + kWBytes));
                tma_load_2d(smem_u32(Xs + (size_t)s * kSlab), &tm_x, full_bar + 8 * s, k * 64, tok0);
                tma_load_2d(smem_u32(Ws + (size_t)s * kWBytes), &tm_w, full_bar + 8 * s, k * 64, 0);
                armed = k + 1;
            }
            for (int k = armed - kLrStages > 0 ? armed - kLrStages : 0; k < armed; ++k)
                mbar_wait(full_bar + 8 * (k % kLrStages), (uint32_t)(k / kLrStages) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kR >> 3) << 17) |
                                   ((uint32_t)(kT >> 4) << 24);
            bool ok = true;
            for (int k = 0; k < nk; ++k) {
                const int s = k % kLrStages;
                if (!mbar_wait(full_bar + 8 * s, (uint32_t)(k / kLrStages) & 1u)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem, sw128_desc(smem_u32(Xs + (size_t)s * kSlab) + 32u * kk),
                              sw128_desc(smem_u32(Ws + (size_t)s * kWBytes) + 32u * kk), idesc,
                              (k | kk) != 0 ? 1u : 0u);
                umma_commit(empty_bar + 8 * s);          // stage free once these MMAs are done
            }
            if (ok) umma_commit(done_bar);
            else misc[1] = 1;
        }
        __syncwarp();
    } else {
        const int q = warp & 3, row = q * 32 + lane;
        const bool ok = mbar_wait(done_bar, 0);
        if (!ok) misc[1] = 1;
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16), v);
        tmem_wait_ld();
        const int64_t n = (int64_t)tok0 + row;
        if (ok && n < a.n_tokens) {
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int r = 0; r < kR; r += 2) {
                const float t0 = __uint_as_float(v[r]), t1 = __uint_as_float(v[r + 1]);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(t0, t1);
                const float2 hf = __bfloat1622float2(hi);
                const __nv_bfloat162 lo = __floats2bfloat162_rn(__fsub_rn(t0, hf.x), __fsub_rn(t1, hf.y));
                hw[r / 2] = *reinterpret_cast<const uint32_t*>(&hi);
                lw[r / 2] = *reinterpret_cast<const uint32_t*>(&lo);
            }
            uint4* dst = reinterpret_cast<uint4*>(a.t2 + n * 2 * kR);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = make_uint4(hw[4 * k], hw[4 * k + 1], hw[4 * k + 2], hw[4 * k + 3]);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[4 + k] = make_uint4(lw[4 * k], lw[4 * k + 1], lw[4 * k + 2], lw[4 * k + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && misc[1] && a.err) atomicExch(a.err, kErrTimeout);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(32u) : "memory");
    }
}

// --------------------------------------------------------------- predict

constexpr int kPrStages = 2;
// TMA warp, MMA warp, two groups of eight epilogue warps: in a group the two
// warps on one TMEM lane quadrant take the two 64-channel halves of its rows
constexpr int kPrEpi = 16;
constexpr int kPrThreads = 64 + 32 * kPrEpi;
constexpr int kResBytes = 3 * kSlab;    // resident per head: B_h (two slabs), [U_h | U_h]
constexpr int kPrBars = 2 * kPrStages + 4 + 2;   // full, empty, tfull, tempty, block full / free

// Stage bytes: x_hat tile (two slabs) and t2 (one slab); the encoder adds the
// x_{l+1} tile (two slabs).
__host__ __device__ constexpr int pr_stage_bytes(bool encode) { return (encode ? 5 : 3) * kSlab; }

struct PrArgs {
    int64_t n_tokens;
    int H, S, tiles;
    uint32_t* codes;         // [S][H][N][D/16]
    uint32_t* meta;          // [S][H][N][D/G]
    uint16_t* xhat;          // [N][H*D] out, or nullptr
    float* pred_out;         // optional [N][H*D]
    const uint8_t* ids;      // decoder, optional: the stages code a smoothed residual (ids [H][N],
    const uint16_t* cent;    // centroids [H][C][D]); see CoralArgs
    int C;
    uint32_t* err;
};

// 16-byte load through L1 (a thread's consecutive vectors share sectors).
__device__ __forceinline__ uint4 ldg_v4_l1(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// Items are (head, 128-token tile) pairs in head-major order; each CTA takes a
// contiguous run of them, so the head's B_h and [U_h | U_h] stay resident in
// shared memory and are reloaded only when the run crosses into the next head
// (the MMA warp signals "block free" once the MMAs that read the old ones are
// done).  A stage carries the item's x_hat tile and t2 -- and, in the encoder,
// its x_{l+1} tile, which the epilogue reads from shared memory; the encoder's
// stage is released by the MMAs and by the four epilogue warps that read it.
template <int G, bool ENCODE, int S>
__global__ void __launch_bounds__(kPrThreads, 1)
    coral_predict_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                            const __grid_constant__ CUtensorMap tm_t, const __grid_constant__ CUtensorMap tm_u,
                            const __grid_constant__ CUtensorMap tm_xn, PrArgs a) {
    constexpr int SB = pr_stage_bytes(ENCODE);
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned, derived from the shared array so that accesses stay in
    // the shared window
    uint8_t* base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* res = base;                                   // resident B_h, [U_h | U_h]
    uint8_t* stages = base + kResBytes;
    const uint32_t bar0 = smem_u32(stages + kPrStages * SB);
    const uint32_t full_bar = bar0, empty_bar = bar0 + 8 * kPrStages, tfull_bar = bar0 + 16 * kPrStages,
                   tempty_bar = tfull_bar + 16, bfull_bar = tempty_bar + 16, bfree_bar = bfull_bar + 8;
    uint32_t* misc = reinterpret_cast<uint32_t*>(stages + kPrStages * SB + 8 * kPrBars);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, HD = H * kDh;
    const int n_items = a.tiles * H;
    const int per = (n_items + (int)gridDim.x - 1) / (int)gridDim.x;
    const int i0 = (int)blockIdx.x * per;
    const int my_items = n_items - i0 < per ? (n_items - i0 > 0 ? n_items - i0 : 0) : per;
    if (tid == 0) {
        for (int s = 0; s < kPrStages; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, ENCODE ? 1 + kPrEpi / 2 : 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar + 8 * b, 1);
            mbar_init(tempty_bar + 8 * b, kPrEpi / 2);
        }
        mbar_init(bfull_bar, 1);
        mbar_init(bfree_bar, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(misc)),
                     "r"(256u)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            int armed = 0, nb = 0, hres = -1;
            for (int i = 0; i < my_items; ++i) {
                const int item = i0 + i;
                const int h = item / a.tiles, tile = item % a.tiles;
                if (h != hres) {
                    // the previous head's block is free once its MMAs are done
                    if (nb > 0 && !mbar_wait(bfree_bar, (uint32_t)(nb - 1) & 1u)) { misc[1] = 1; break; }
                    mbar_arrive_tx(bfull_bar, (uint32_t)kResBytes);
                    for (int at = 0; at < 2; ++at)
                        tma_load_2d(smem_u32(res + at * kSlab), &tm_b, bfull_bar, at * 64, h * kDh);
                    tma_load_2d(smem_u32(res + 2 * kSlab), &tm_u, bfull_bar, 0, h * kDh);
                    hres = h;
                    ++nb;
                }
                const int s = i % kPrStages;
                if (!mbar_wait(empty_bar + 8 * s, ((uint32_t)(i / kPrStages) & 1u) ^ 1u)) { misc[1] = 1; break; }
                uint8_t* st = stages + (size_t)s * SB;
                const uint32_t fb = full_bar + 8 * s;
                mbar_arrive_tx(fb, (uint32_t)SB);
                for (int at = 0; at < 2; ++at)
                    tma_load_2d(smem_u32(st + at * kSlab), &tm_x, fb, h * kDh + at * 64, tile * kT);
                tma_load_2d(smem_u32(st + 2 * kSlab), &tm_t, fb, 0, tile * kT);
                if (ENCODE)
                    for (int at = 0; at < 2; ++at)
                        tma_load_2d(smem_u32(st + (3 + at) * kSlab), &tm_xn, fb, h * kDh + at * 64, tile * kT);
                armed = i + 1;
            }
            // drain this warp's copies before the CTA exits
            for (int i = armed - kPrStages > 0 ? armed - kPrStages : 0; i < armed; ++i)
                mbar_wait(full_bar + 8 * (i % kPrStages), (uint32_t)(i / kPrStages) & 1u);
            if (nb > 0) mbar_wait(bfull_bar, (uint32_t)(nb - 1) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kDh >> 3) << 17) |
                                   ((uint32_t)(kT >> 4) << 24);
            const uint32_t rs = smem_u32(res);
            int issued = 0, nb = 0, hres = -1;
            bool ok = true;
            for (int i = 0; i < my_items && ok; ++i) {
                const int h = (i0 + i) / a.tiles;
                if (h != hres) {
                    if (nb > 0) umma_commit(bfree_bar);     // the old block is free once the MMAs so far are done
                    if (!mbar_wait(bfull_bar, (uint32_t)nb & 1u)) { ok = false; break; }
                    hres = h;
                    ++nb;
                }
                const int s = i % kPrStages, acc = i & 1;
                if (!mbar_wait(tempty_bar + 8 * acc, ((uint32_t)(i >> 1) & 1u) ^ 1u)) { ok = false; break; }
                if (!mbar_wait(full_bar + 8 * s, (uint32_t)(i / kPrStages) & 1u)) { ok = false; break; }
                tc_fence_after();
                const uint32_t st = smem_u32(stages + (size_t)s * SB);
                const uint32_t d = tmem + (uint32_t)acc * kDh;
#pragma unroll
                for (int at = 0; at < 2; ++at)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(d, sw128_desc(st + at * kSlab + 32u * kk), sw128_desc(rs + at * kSlab + 32u * kk),
                                  idesc, (at | kk) != 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(d, sw128_desc(st + 2 * kSlab + 32u * kk), sw128_desc(rs + 2 * kSlab + 32u * kk), idesc, 1u);
                umma_commit(empty_bar + 8 * s);        // operands consumed once these MMAs are done
                umma_commit(tfull_bar + 8 * acc);
                issued = i + 1;
            }
            if (!ok) misc[1] = 1;
            for (int i = issued - 2 > 0 ? issued - 2 : 0; i < issued; ++i)
                mbar_wait(tfull_bar + 8 * (i & 1), (uint32_t)(i >> 1) & 1u);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- epilogue
        // A thread owns one token row's half: 64 channels = one TMEM lane,
        // 64 accumulator columns; it works through them in passes of CPT.
        constexpr int CPT = G < 32 ? 32 : G;      // channels per pass (whole groups)
        constexpr int GPP = CPT / G;              // groups per pass
        constexpr int HALF = kDh / 2;
        constexpr int NP = HALF / CPT;            // passes per half row
        constexpr int WPR = kDh / 16, MPR = kDh / G;
        constexpr int WPH = HALF / 16, MPH = HALF / G > 0 ? HALF / G : 1;
        const int e = warp - 2, g = e >> 3, hf = (e >> 2) & 1, q = warp & 3;
        const int row = q * 32 + lane;
        const int64_t stage_rows = (int64_t)H * a.n_tokens;
        for (int i = g; i < my_items; i += 2) {
            const int item = i0 + i;
            const int h = item / a.tiles, tile = item % a.tiles;
            const int64_t n = (int64_t)tile * kT + row;
            const bool valid = n < a.n_tokens;
            const int64_t elem0 = n * HD + (int64_t)h * kDh + hf * HALF;
            const int64_t rowoff = (int64_t)h * a.n_tokens + n;
            // The decoder's loads do not depend on the MMA: the codes and
            // scale/zero words of the half row are issued before waiting for it.
            uint32_t code[ENCODE || S == 0 ? 1 : S][WPH], meta[ENCODE || S == 0 ? 1 : S][MPH];
            if (!ENCODE) {
#pragma unroll
                for (int s = 0; s < S; ++s) {
                    const int64_t srow = (int64_t)s * stage_rows + rowoff;
#pragma unroll
                    for (int w = 0; w < WPH; w += 4) {
                        const uint4 cw = valid ? ldg_v4_l1(a.codes + srow * WPR + hf * WPH + w) : make_uint4(0, 0, 0, 0);
                        code[s][w] = cw.x; code[s][w + 1] = cw.y; code[s][w + 2] = cw.z; code[s][w + 3] = cw.w;
                    }
#pragma unroll
                    for (int m = 0; m < MPH; ++m) meta[s][m] = valid ? __ldg(a.meta + srow * MPR + hf * MPH + m) : 0u;
                }
            }
            // a smoothed residual's centroid row (half of it), also ahead of the wait
            constexpr bool HYB = !ENCODE && S > 0;
            uint4 cv[HYB ? HALF / 8 : 1];
            if constexpr (HYB) {
                if (a.cent) {
                    const int id = valid ? min((int)a.ids[rowoff], a.C - 1) : 0;
                    const uint16_t* cr = a.cent + ((int64_t)h * a.C + id) * kDh + hf * HALF;
#pragma unroll
                    for (int v8 = 0; v8 < HALF / 8; ++v8) cv[v8] = valid ? ldg_v4_l1(cr + 8 * v8) : make_uint4(0, 0, 0, 0);
                }
            }
            if (!mbar_wait(tfull_bar + 8 * g, (uint32_t)(i >> 1) & 1u)) { misc[1] = 1; break; }
            // the encoder reads the stage's x_{l+1} tile: wait on the stage's own
            // arrival too, so the copy's bytes are visible to these threads
            const int si = i % kPrStages;
            if (ENCODE && !mbar_wait(full_bar + 8 * si, (uint32_t)(i / kPrStages) & 1u)) { misc[1] = 1; break; }
            // this thread's half row of the x_{l+1} tile: slab hf, 128-byte swizzled
            const uint8_t* xrow = stages + (size_t)si * SB + (3 + hf) * kSlab + (size_t)row * 128;
            tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)g * kDh + (uint32_t)(hf * HALF);
#pragma unroll
            for (int c = 0; c < NP; ++c) {
                const uint32_t tcol = tbase + (uint32_t)(c * CPT);
                // the encoder's codes and scale/zero words of this pass
                uint32_t ec[ENCODE && S > 0 ? S : 1][CPT / 16], em[ENCODE && S > 0 ? S : 1][GPP];
                if (ENCODE) {
                    // residual r = x_{l+1} - pred, 16 channels at a time
                    float r[CPT];
#pragma unroll
                    for (int k = 0; k < CPT / 16; ++k) {
                        uint32_t v[16];
                        tmem_ld16(tcol + 16u * k, v);
                        // channel ch of the half sits in 16-byte chunk ch / 8 of the
                        // row, stored at chunk position chunk ^ (row % 8)
                        const int ch = c * CPT + 16 * k;
                        const uint4 x0 = *reinterpret_cast<const uint4*>(xrow + ((((ch >> 3)) ^ (row & 7)) << 4));
                        const uint4 x1 = *reinterpret_cast<const uint4*>(xrow + ((((ch >> 3) + 1) ^ (row & 7)) << 4));
                        tmem_wait_ld_regs16(v);
                        float pk[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) pk[jj] = __uint_as_float(v[jj]);
                        if (valid && a.pred_out) {
#pragma unroll
                            for (int jj = 0; jj < 16; jj += 4)
                                *reinterpret_cast<float4*>(a.pred_out + elem0 + c * CPT + 16 * k + jj) =
                                    make_float4(pk[jj], pk[jj + 1], pk[jj + 2], pk[jj + 3]);
                        }
                        unpack16(x0, x1, r + 16 * k);
                        sub16(r + 16 * k, pk);
                    }
#pragma unroll
                    for (int s = 0; s < S; ++s) {
#pragma unroll
                        for (int gi = 0; gi < GPP; ++gi) {
                            uint32_t cw[G / 16], m;
                            quant_stage<G, 1>(r + gi * G, s + 1 < S, nullptr, cw, m);
#pragma unroll
                            for (int w = 0; w < G / 16; ++w) ec[s][(gi * G) / 16 + w] = cw[w];
                            em[s][gi] = m;
                        }
                        if (valid) {
                            const int64_t srow = (int64_t)s * stage_rows + rowoff;
                            uint32_t* cp = a.codes + srow * WPR + (hf * HALF + c * CPT) / 16;
                            if constexpr (CPT / 16 == 4) *reinterpret_cast<uint4*>(cp) = make_uint4(ec[s][0], ec[s][1], ec[s][2], ec[s][3]);
                            else *reinterpret_cast<uint2*>(cp) = make_uint2(ec[s][0], ec[s][1]);
#pragma unroll
                            for (int gi = 0; gi < GPP; ++gi) a.meta[srow * MPR + (hf * HALF + c * CPT) / G + gi] = em[s][gi];
                        }
                    }
                }
                // x_hat = ((pred + d_1) + d_2) + ..., identical in encoder and decoder
#pragma unroll
                for (int k = 0; k < CPT / 16; ++k) {
                    uint32_t v[16];
                    tmem_ld16(tcol + 16u * k, v);
                    tmem_wait_ld_regs16(v);
                    float acc[16];
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) acc[jj] = __uint_as_float(v[jj]);
                    const int ch = c * CPT + 16 * k;                 // channel within the half
                    if (!ENCODE && valid && a.pred_out) {
#pragma unroll
                        for (int jj = 0; jj < 16; jj += 4)
                            *reinterpret_cast<float4*>(a.pred_out + elem0 + ch + jj) =
                                make_float4(acc[jj], acc[jj + 1], acc[jj + 2], acc[jj + 3]);
                    }
                    if constexpr (ENCODE) {
#pragma unroll
                        for (int s = 0; s < S; ++s) dequant_add16(acc, ec[s][(16 * k) / 16], em[s][(16 * k) / G]);
                    } else if constexpr (HYB) {
                        if (a.cent) {
                            // r_hat = bf16(c[id] + d_1 + d_2 + ...), the QVG decoder's sum
                            // and rounding, then x_hat = bf16(pred + r_hat): one fp32 addition
                            float rr[16];
                            unpack16(cv[ch / 8], cv[ch / 8 + 1], rr);
#pragma unroll
                            for (int s = 0; s < S; ++s) dequant_add16(rr, code[s][ch / 16], meta[s][ch / G]);
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                acc[jj] = __fadd_rn(acc[jj], __bfloat162float(__float2bfloat16_rn(rr[jj])));
                        } else {
#pragma unroll
                            for (int s = 0; s < S; ++s) dequant_add16(acc, code[s][ch / 16], meta[s][ch / G]);
                        }
                    }
                    if (valid && a.xhat) {
                        uint4 o0, o1;
                        pack16_bf16(acc, o0, o1);
                        uint16_t* op = a.xhat + elem0 + ch;
                        *reinterpret_cast<uint4*>(op) = o0;
                        *reinterpret_cast<uint4*>(op + 8) = o1;
                    }
                }
            }
            // accumulator drained (and, in the encoder, the stage's x_{l+1} read)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(tempty_bar + 8 * g);
                if (ENCODE) mbar_arrive(empty_bar + 8 * si);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && misc[1] && a.err) atomicExch(a.err, kErrTimeout);
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256u) : "memory");
    }
}

bool encode_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// prep + low-rank: t = x_hat W into w.t2 as (hi, lo) bf16 pairs
cudaError_t lowrank_stage(const CoralArgs& a, const CoralTcScratch& w, const CUtensorMap& tx, const CUtensorMap& tw,
                          cudaStream_t s) {
    const int HD = a.H * kDh;
    const int64_t N = a.n_tokens;
    // the re-layout of W and U, unless the caller prepared it once
    if (!a.prepared)
        coral_prep_kernel<<<(unsigned)((HD + kPrepRows - 1) / kPrepRows), 256, 0, s>>>(a.W, a.U, HD, w.wt, w.ud);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int tiles = (int)((N + kT - 1) / kT);
    const size_t lr_smem = (size_t)kLrStages * (kSlab + kR * 128) + 8 * (2 * kLrStages + 1) + 32 + 1024;
    // at least 116 KB so that one CTA (and one TMEM allocation) lives per SM
    const size_t lr_req = lr_smem < 118784 ? 118784 : lr_smem;
    e = cudaFuncSetAttribute(coral_lowrank_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lr_req);
    if (e != cudaSuccess) return e;
    LrArgs la{N, HD, w.t2, w.err};
    coral_lowrank_tc_kernel<<<(unsigned)tiles, kLrThreads, lr_req, s>>>(tx, tw, la);
    return cudaGetLastError();
}

template <int G>
cudaError_t coral_tc_g(bool encode, const CoralArgs& a, const CoralTcScratch& w, bool* launched, cudaStream_t s) {
    const int H = a.H, HD = H * kDh;
    const int64_t N = a.n_tokens;
    CUtensorMap tx, tw, tb, tt, tu, txn;
    if (!encode_2d(&tx, a.xprev, (uint64_t)HD, (uint64_t)N, (uint64_t)HD * 2, 64, kT)) return cudaSuccess;
    if (encode && !encode_2d(&txn, a.xnext, (uint64_t)HD, (uint64_t)N, (uint64_t)HD * 2, 64, kT)) return cudaSuccess;
    if (!encode_2d(&tw, w.wt, (uint64_t)HD, (uint64_t)kR, (uint64_t)HD * 2, 64, kR)) return cudaSuccess;
    if (!encode_2d(&tb, a.B, (uint64_t)kDh, (uint64_t)HD, (uint64_t)kDh * 2, 64, kT)) return cudaSuccess;
    if (!encode_2d(&tt, w.t2, (uint64_t)(2 * kR), (uint64_t)N, (uint64_t)(4 * kR), 64, kT)) return cudaSuccess;
    if (!encode_2d(&tu, w.ud, (uint64_t)(2 * kR), (uint64_t)HD, (uint64_t)(4 * kR), 64, kT)) return cudaSuccess;
    cudaError_t e = lowrank_stage(a, w, tx, tw, s);
    if (e != cudaSuccess) return e;
    const int tiles = (int)((N + kT - 1) / kT);
    const size_t pr_smem = (size_t)kResBytes + (size_t)kPrStages * pr_stage_bytes(encode) + 8 * kPrBars + 32 + 1024;
    // the stage count is a template parameter: the epilogue's stage loops unroll
    auto kern = encode ? coral_predict_tc_kernel<G, true, 2> : coral_predict_tc_kernel<G, false, 2>;
    switch (a.S) {
        case 0:                       // the prediction alone (the Coral + SAS hybrid)
            if (encode) return cudaSuccess;
            kern = coral_predict_tc_kernel<G, false, 0>;
            break;
        case 1: kern = encode ? coral_predict_tc_kernel<G, true, 1> : coral_predict_tc_kernel<G, false, 1>; break;
        case 2: break;
        case 3: kern = encode ? coral_predict_tc_kernel<G, true, 3> : coral_predict_tc_kernel<G, false, 3>; break;
        case 4: kern = encode ? coral_predict_tc_kernel<G, true, 4> : coral_predict_tc_kernel<G, false, 4>; break;
        default: return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pr_smem);
    if (e != cudaSuccess) return e;
    PrArgs pa;
    pa.n_tokens = N; pa.H = H; pa.S = a.S; pa.tiles = tiles;
    pa.codes = a.codes; pa.meta = a.meta; pa.xhat = a.xhat; pa.pred_out = a.pred_out;
    pa.ids = encode ? nullptr : a.ids;
    pa.cent = encode ? nullptr : a.cent;
    pa.C = a.C;
    pa.err = w.err;
    const int items = tiles * H;
    const int grid = items < sm_count() ? items : sm_count();
    kern<<<(unsigned)grid, kPrThreads, pr_smem, s>>>(tx, tb, tt, tu, encode ? txn : tx, pa);
    if ((e = cudaGetLastError()) == cudaSuccess) *launched = true;
    return e;
}

}  // namespace

size_t coral_tc_scratch_bytes(int H, int64_t n_tokens) {
    const size_t HD = (size_t)H * kDh, N = (size_t)(n_tokens > 0 ? n_tokens : 1);
    auto a256 = [](size_t v) { return (v + 255) & ~(size_t)255; };
    return a256(N * 2 * kR * 2) + a256((size_t)kR * HD * 2) + a256(HD * 2 * kR * 2) + 256;
}

size_t coral_prepared_bytes(int H) {
    const size_t HD = (size_t)H * kDh;
    auto a256 = [](size_t v) { return (v + 255) & ~(size_t)255; };
    return a256((size_t)kR * HD * 2) + a256(HD * 2 * kR * 2);
}

void use_prepared(const uint16_t* prepared, int H, CoralTcScratch& w) {
    const size_t HD = (size_t)H * kDh;
    const size_t wt_bytes = ((size_t)kR * HD * 2 + 255) & ~(size_t)255;
    w.wt = const_cast<uint16_t*>(prepared);
    w.ud = const_cast<uint16_t*>(prepared) + wt_bytes / 2;
}

cudaError_t launch_coral_prep(const uint16_t* W, const uint16_t* U, int H, uint16_t* prepared, cudaStream_t s) {
    const int HD = H * kDh;
    CoralTcScratch w{};
    use_prepared(prepared, H, w);
    coral_prep_kernel<<<(unsigned)((HD + kPrepRows - 1) / kPrepRows), 256, 0, s>>>(W, U, HD, w.wt, w.ud);
    return cudaGetLastError();
}

cudaError_t launch_coral_lowrank_tc(const CoralArgs& a, const CoralTcScratch& w, cudaStream_t s) {
    const int HD = a.H * kDh;
    CUtensorMap tx, tw;
    if (!encode_2d(&tx, a.xprev, (uint64_t)HD, (uint64_t)a.n_tokens, (uint64_t)HD * 2, 64, kT) ||
        !encode_2d(&tw, w.wt, (uint64_t)HD, (uint64_t)kR, (uint64_t)HD * 2, 64, kR))
        return cudaErrorInvalidValue;
    return lowrank_stage(a, w, tx, tw, s);
}

cudaError_t launch_coral_tc(int D, int G, bool encode, const CoralArgs& a, const CoralTcScratch& w, bool* launched,
                            cudaStream_t s) {
    *launched = false;
    if (D != kDh || a.R != kR || !a.xprev || a.n_tokens == 0) return cudaSuccess;
    auto al = [](const void* p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; };
    if (!al(a.xprev, 16) || !al(a.B, 16) || !al(w.t2, 128) || !al(w.wt, 128) || !al(w.ud, 128)) return cudaSuccess;
    // the epilogue moves 16-byte vectors of x_{l+1}, x_hat, codes and the prediction
    if (!al(a.xnext, 16) || !al(a.xhat, 16) || !al(a.codes, 16) || !al(a.pred_out, 16) || !al(a.cent, 16))
        return cudaSuccess;
    switch (G) {
        case 16: return coral_tc_g<16>(encode, a, w, launched, s);
        case 32: return coral_tc_g<32>(encode, a, w, launched, s);
        case 64: return coral_tc_g<64>(encode, a, w, launched, s);
        default: return cudaSuccess;
    }
}

}  // namespace qvg
