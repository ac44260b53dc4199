// Progressive residual quantisation: the persistent decoder fed by the copy
// engine, for head_dim 64 and 128 (sm_103a).
//
// Quant VideoGen explainer, Sommario tecnico sec. 2B item 3 (decoding
// dequantises every stage, sums them and adds the centroid back) and sec. 3
// (centroid caching: each streaming chunk decodes against its own centroid
// version).
//
// One CTA per SM walks a contiguous run of (head, token tile) units.  Warp 15
// is the producer: one lane moves each tile's code rows, scale/zero words and
// cluster ids into a ring of shared-memory stages with cp.async.bulk (one copy
// per stage and array; the scale/zero and id copies take the 16-byte-aligned
// window around the tile's bytes, and a window that would run past the end of
// its buffer is left to plain loads), and the head's centroid table (C x D
// bf16, up to 64 KB) into its own buffer whenever the run enters another head
// or, streaming, another centroid version.  Warps 0-14 compute: lane l owns 16
// consecutive channels of R rows of the tile (8 lanes a row at D = 128, 4 at
// D = 64).  Consumers release a stage as soon as its words are in registers.
//
// Bank conflicts: a row of the table or of the output is D*2 bytes of 16-byte
// chunks; a lane reads its two chunks 2t, 2t+1 in the order that puts the
// eight lanes of a quarter-warp on eight different bank groups (lanes of the
// upper half of a row, and at D = 64 those of the second row of the
// quarter-warp, take the odd chunk first).  Registers then hold the channels
// in that order; the code words and output addresses follow it.
//
// Every wait is bounded (qvg_debug_set_wait changes the limit); a wait that
// runs out records kErrTimeout in the library's device error word (read with
// qvg_device_error), every role drains the copies it issued and the CTA
// returns.
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "prq16.cuh"
#include "tc_common.cuh"

namespace qvg {

namespace {

// 15 consumer warps + the producer = 16 warps, four per scheduler, which
// leaves each thread up to 128 registers (a scheduler's file holds 16,384; a
// fifth warp on one of them would cap every thread at 96).
constexpr int kCWarps = 15;                     // decoder consumer warps
constexpr int kPThreads = 32 * (kCWarps + 1);   // + the producer warp
constexpr int kMaxRing = 8;
constexpr uint32_t kErrTimeout = 0x7E000000u;

// Waits for the phase of parity `parity`; gives up after `limit` ns.
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, unsigned long long limit) {
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 7u) == 0 && global_ns() - t0 > limit) return false;
    }
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit) {
    return mbar_try(bar, parity) || wait_slow(bar, parity, limit);
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void record_timeout(uint32_t* err) { atomicExch(err, kErrTimeout); }

// Before a producer whose consumers may have given up returns: waits (bounded)
// until the copies of the last `nst` stages it issued have landed, so that no
// copy is still writing into the CTA's shared memory when the CTA exits.  A
// stage withheld by the test flag (stage 0) was never issued.
template <typename FullBar>
__device__ __forceinline__ void drain(int64_t issued, int nst, bool withhold, FullBar full_bar,
                                      unsigned long long limit) {
    const int64_t first = issued > nst ? issued - nst : 0;
    for (int64_t i = first; i < issued; ++i) {
        if (withhold && i == 0) continue;
        wait_bounded(full_bar((int)(i % nst)), (uint32_t)((i / nst) & 1), limit);
    }
}

template <int D, int R>
struct RowMap {
    static constexpr int TPR = D / 16;                 // lanes per row
    static constexpr int RPW = 32 / TPR;               // rows per warp and block
    static constexpr int BLOCK = kCWarps * RPW;        // rows of one pass of the 16 warps (64 or 128)
    static constexpr int TILE = BLOCK * R;             // rows per tile: R blocks, one row of each per lane
};

// Order of a lane's two 16-byte chunks (see the top of this file): 1 = the odd
// chunk first.
template <int D>
__device__ __forceinline__ int chunk_swap(int lane) {
    constexpr int TPR = D / 16;
    const int t = lane % TPR;
    const int second_row = (TPR == 4) ? ((lane >> 2) & 1) : 0;
    return (t >= TPR / 2 ? 1 : 0) ^ second_row;
}

// This CTA's run of units (head, tile), heads x tiles in head-major order:
// `count` units from (h0, t0).
struct UnitRun {
    int64_t count;
    int h0, t0;
};

__device__ __forceinline__ UnitRun unit_run(int H, int tiles) {
    const int64_t units = (int64_t)H * tiles;
    const int64_t u0 = units * blockIdx.x / gridDim.x, u1 = units * (blockIdx.x + 1) / gridDim.x;
    UnitRun r;
    r.count = u1 - u0;
    r.h0 = (int)(u0 / tiles);
    r.t0 = (int)(u0 - (int64_t)r.h0 * tiles);
    return r;
}

// Walks (head, tile) and (ring stage, phase) one unit forward.
struct Cursor {
    int h, tile, st;
    uint32_t ph;
    __device__ __forceinline__ void next(int tiles, int nst) {
        if (++tile == tiles) { tile = 0; ++h; }
        if (++st == nst) { st = 0; ph ^= 1u; }
    }
};


constexpr uint32_t kSmemLimit = 232448u;

inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

}  // namespace

// The error word of the kernels that take no workspace, one per device.
__device__ uint32_t g_codec_err = 0;

namespace {

std::atomic<unsigned long long> g_limit_ns{2000000000ull};
std::atomic<uint32_t> g_flags{0u};
std::mutex g_err_mu;
constexpr int kMaxDev = 64;
uint32_t* g_err_ptr[kMaxDev] = {};

}  // namespace

namespace {

// --------------------------------------------------------------- decoder --

struct DecTma {
    CodecCtl ctl;
    const uint32_t* codes;
    const uint32_t* meta;
    const uint8_t* ids;
    const uint16_t* cent;          // version-0 table, [V][H][C][D]
    const int64_t* chunk_offset;   // null: one version
    const int32_t* chunk_version;
    int n_chunks;
    int64_t cap, tok_begin, n_rows;
    uint16_t* out;
    int64_t out_head_stride, out_token_stride;
    int H, C, S, tiles, nst;
    int64_t meta_words, id_bytes;  // extents of the meta and id buffers
    uint32_t table_off, chunk_off, ring_off, slot_bytes, codes_bytes, meta_slot, bar_off;
};

// 16-byte-aligned window [ws, we) around [start, start + len) bytes of a
// buffer of `extent` bytes; false when it would run past the buffer's end.
__device__ __forceinline__ bool window16(int64_t start, int64_t len, int64_t extent, int64_t& ws, int64_t& we) {
    ws = start & ~(int64_t)15;
    we = (start + len + 15) & ~(int64_t)15;
    return we <= extent;
}

template <int D, int G, int B, int S, int R, bool HAS_C, bool VERSIONED>
__global__ void __launch_bounds__(kPThreads, 1) prq_decode_tma_kernel(DecTma a) {
    using M = RowMap<D, R>;
    constexpr int TILE = M::TILE, TPR = M::TPR, BLOCK = M::BLOCK;
    constexpr int WPR = D * B / 32, MPR = D / G, WPT = B / 2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the launch adds 1024 bytes of slack: the map is laid out from a 1024-byte boundary
    uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bars = smem_u32(sm + a.bar_off);
    auto full_bar = [&](int st) { return bars + 8u * st; };
    auto empty_bar = [&](int st) { return bars + 8u * (kMaxRing + st); };
    const uint32_t tab_full = bars + 8u * (2 * kMaxRing), tab_empty = tab_full + 8u;
    const unsigned long long limit = a.ctl.limit;
    int64_t* offs = reinterpret_cast<int64_t*>(sm + a.chunk_off);
    int32_t* vers = reinterpret_cast<int32_t*>(sm + a.chunk_off + 8 * (a.n_chunks + 1));
    if (threadIdx.x == 0) {
        for (int st = 0; st < a.nst; ++st) {
            mbar_init(full_bar(st), 1);
            mbar_init(empty_bar(st), kCWarps);
        }
        mbar_init(tab_full, 1);
        mbar_init(tab_empty, kCWarps);
        fence_mbar_init();
    }
    if (VERSIONED) {
        for (int i = threadIdx.x; i <= a.n_chunks; i += blockDim.x) offs[i] = a.chunk_offset[i];
        for (int i = threadIdx.x; i < a.n_chunks; i += blockDim.x) vers[i] = a.chunk_version[i];
    }
    __syncthreads();
    // centroid version of cache row n: that of the last chunk starting at or before it
    auto version_of = [&](int64_t n) -> int {
        if (!VERSIONED) return 0;
        int lo = 0, hi = a.n_chunks - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (offs[mid] <= n) lo = mid; else hi = mid - 1;
        }
        return vers[lo];
    };
    const UnitRun run = unit_run(a.H, a.tiles);
    const int64_t stage_rows = (int64_t)a.H * a.cap;
    const size_t table_elems = (size_t)a.C * D;
    const uint32_t ids_off = a.codes_bytes + (uint32_t)S * a.meta_slot;

    if (warp == kCWarps) {
        // ---------------- producer
        if (lane != 0) return;
        const bool withhold = (a.ctl.flags & 1u) != 0;
        bool ok = true;
        int head = -1, ver = -1;
        uint32_t tab_ph = 0;
        int64_t issued = 0;
        Cursor c{run.h0, run.t0, 0, 0u};
        for (int64_t k = 0; k < run.count; ++k, c.next(a.tiles, a.nst)) {
            const int64_t n0 = (int64_t)c.tile * TILE;
            const int rows = (int)min((int64_t)TILE, a.n_rows - n0);
            if (k >= a.nst && !wait_bounded(empty_bar(c.st), c.ph ^ 1u, limit)) { ok = false; break; }
            const uint32_t slot = smem_u32(sm + a.ring_off) + (uint32_t)c.st * a.slot_bytes;
            if (withhold && k == 0) {
                ++issued;   // test flag: the first stage never fills
            } else {
                // the bytes first (the barrier must expect them before any copy lands)
                uint32_t bytes = (uint32_t)S * rows * WPR * 4;
                int64_t ws, we;
                const int64_t row0 = (int64_t)c.h * a.cap + a.tok_begin + n0;
                for (int s = 0; s < S; ++s)
                    if (window16((s * stage_rows + row0) * MPR * 4, (int64_t)rows * MPR * 4, a.meta_words * 4, ws, we))
                        bytes += (uint32_t)(we - ws);
                if (HAS_C && window16(row0, rows, a.id_bytes, ws, we)) bytes += (uint32_t)(we - ws);
                mbar_arrive_tx(full_bar(c.st), bytes);
                for (int s = 0; s < S; ++s) {
                    const int64_t srow = s * stage_rows + row0;
                    bulk_g2s(slot + (uint32_t)s * TILE * WPR * 4, a.codes + srow * WPR, (uint32_t)rows * WPR * 4,
                             full_bar(c.st));
                    if (window16(srow * MPR * 4, (int64_t)rows * MPR * 4, a.meta_words * 4, ws, we))
                        bulk_g2s(slot + a.codes_bytes + (uint32_t)s * a.meta_slot,
                                 reinterpret_cast<const uint8_t*>(a.meta) + ws, (uint32_t)(we - ws), full_bar(c.st));
                }
                if (HAS_C && window16(row0, rows, a.id_bytes, ws, we))
                    bulk_g2s(slot + ids_off, a.ids + ws, (uint32_t)(we - ws), full_bar(c.st));
                ++issued;
            }
            if (HAS_C) {
                const int v = version_of(a.tok_begin + n0);
                if (c.h != head || v != ver) {
                    if (head >= 0) {
                        if (!wait_bounded(tab_empty, tab_ph, limit)) { ok = false; break; }
                        tab_ph ^= 1u;
                    }
                    const uint32_t tb = (uint32_t)(table_elems * 2);
                    mbar_arrive_tx(tab_full, tb);
                    bulk_g2s(smem_u32(sm + a.table_off), a.cent + ((size_t)v * a.H + c.h) * table_elems, tb,
                             tab_full);
                    head = c.h;
                    ver = v;
                }
            }
        }
        if (!ok) record_timeout(a.ctl.err);
        if (!ok || withhold) drain(issued, a.nst, withhold, full_bar, limit);
        if (withhold && HAS_C && head >= 0) wait_bounded(tab_full, tab_ph, limit);
        return;
    }

    // ---------------- consumers: lane owns 16 channels of rows j * BLOCK + rb, j < R
    const int rb = warp * M::RPW + lane / TPR;
    const int t = lane % TPR;
    const int sw = chunk_swap<D>(lane);
    const int c0 = 2 * t + sw, c1 = 2 * t + 1 - sw;
    const int mi = (16 * t) / G;
    int head = -1, ver = -1;
    uint32_t tab_ph = 0;
    bool ok = true;
    Cursor c{run.h0, run.t0, 0, 0u};
    for (int64_t k = 0; k < run.count; ++k, c.next(a.tiles, a.nst)) {
        const int64_t n0 = (int64_t)c.tile * TILE;
        const int rows = (int)min((int64_t)TILE, a.n_rows - n0);
        if (!wait_bounded(full_bar(c.st), c.ph, limit)) { ok = false; break; }
        const uint8_t* slot = sm + a.ring_off + (size_t)c.st * a.slot_bytes;
        uint32_t code[R][S][WPT], meta[R][S];
        int id[R];
        const int64_t row0 = (int64_t)c.h * a.cap + a.tok_begin + n0;
        int64_t ws, we;
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int64_t srow = s * stage_rows + row0;
            // scale/zero words: from the stage, or (a window that would pass the end of
            // the buffer, which the producer did not copy) straight from global memory
            const bool in_smem = window16(srow * MPR * 4, (int64_t)rows * MPR * 4, a.meta_words * 4, ws, we);
            const uint32_t* mb = reinterpret_cast<const uint32_t*>(slot + a.codes_bytes + (size_t)s * a.meta_slot +
                                                                   (srow * MPR * 4 - ws));
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int rin = j * BLOCK + rb;
                const uint32_t* cw = reinterpret_cast<const uint32_t*>(slot + (size_t)s * TILE * WPR * 4) + rin * WPR + WPT * t;
#pragma unroll
                for (int w = 0; w < WPT; ++w) code[j][s][w] = cw[w];
                if (in_smem) meta[j][s] = mb[rin * MPR + mi];
                else meta[j][s] = rin < rows ? __ldg(a.meta + (srow + rin) * MPR + mi) : 0u;
            }
        }
        if (HAS_C) {
            const bool in_smem = window16(row0, rows, a.id_bytes, ws, we);
#pragma unroll
            for (int j = 0; j < R; ++j) {
                const int rin = j * BLOCK + rb;
                int v = 0;
                if (in_smem) v = slot[ids_off + (row0 - ws) + rin];
                else if (rin < rows) v = __ldg(a.ids + row0 + rin);
                id[j] = min(v, a.C - 1);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(c.st));
        bool mixed = false;   // rows of more than one centroid version in this tile
        if (HAS_C) {
            const int v = version_of(a.tok_begin + n0);
            mixed = VERSIONED && version_of(a.tok_begin + n0 + rows - 1) != v;
            if (c.h != head || v != ver) {
                if (head >= 0) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tab_empty);
                }
                if (!wait_bounded(tab_full, tab_ph, limit)) { ok = false; break; }
                tab_ph ^= 1u;
                head = c.h;
                ver = v;
            }
        }
#pragma unroll
        for (int j = 0; j < R; ++j) {
            const int rin = j * BLOCK + rb;
            const bool valid = rin < rows;
            const int64_t n = n0 + rin;
            float acc[16];
            if (HAS_C) {
                const int rv = (mixed && valid) ? version_of(a.tok_begin + n) : ver;
                uint4 k0, k1;
                if (rv == ver) {
                    const uint8_t* crow = sm + a.table_off + (size_t)id[j] * D * 2;
                    k0 = *reinterpret_cast<const uint4*>(crow + 16 * c0);
                    k1 = *reinterpret_cast<const uint4*>(crow + 16 * c1);
                } else {
                    // a row of another centroid version inside this tile
                    const uint16_t* crow = a.cent + (((size_t)rv * a.H + c.h) * a.C + id[j]) * D;
                    k0 = __ldg(reinterpret_cast<const uint4*>(crow) + c0);
                    k1 = __ldg(reinterpret_cast<const uint4*>(crow) + c1);
                }
                unpack16(k0, k1, acc);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
            }
#pragma unroll
            for (int s = 0; s < S; ++s) {
                if constexpr (B == 2) {
                    // register slots 0-7 hold chunk c0: bring its codes to the low half
                    const uint32_t cw = sw ? ((code[j][s][0] >> 16) | (code[j][s][0] << 16)) : code[j][s][0];
                    dequant_add16(acc, cw, meta[j][s]);
                } else {
                    const uint32_t w0 = sw ? code[j][s][1] : code[j][s][0];
                    const uint32_t w1 = sw ? code[j][s][0] : code[j][s][1];
                    dequant_add8x4(acc, w0, meta[j][s]);
                    dequant_add8x4(acc + 8, w1, meta[j][s]);
                }
            }
            if (valid) {
                uint4 o0, o1;
                pack16_bf16(acc, o0, o1);
                uint16_t* op = a.out + (int64_t)c.h * a.out_head_stride + n * a.out_token_stride;
                stg_v4_stream(op + 8 * c0, o0);
                stg_v4_stream(op + 8 * c1, o1);
            }
        }
    }
    if (!ok) record_timeout(a.ctl.err);
}

// Shared-memory layout of the decoder for R rows per lane; false when it
// does not fit with at least three stages.
template <int D, int G, int B, int R>
bool decode_layout(const DecodeArgs& a, DecTma& t) {
    using M = RowMap<D, R>;
    constexpr int WPR = D * B / 32, MPR = D / G;
    const bool versioned = a.C > 0 && a.chunk_offset;
    t.tiles = (int)((t.n_rows + M::TILE - 1) / M::TILE);
    t.table_off = 0;
    uint32_t o = align_up(a.C > 0 ? (uint32_t)a.C * D * 2 : 0u, 128u);
    t.chunk_off = o;
    if (versioned) o = align_up(o + 8u * (a.n_chunks + 1) + 4u * a.n_chunks, 128u);
    t.ring_off = align_up(o, 128u);
    t.codes_bytes = (uint32_t)a.S * M::TILE * WPR * 4;
    t.meta_slot = align_up((uint32_t)M::TILE * MPR * 4 + 32u, 16u);
    t.slot_bytes = align_up(t.codes_bytes + (uint32_t)a.S * t.meta_slot + (uint32_t)M::TILE + 32u, 128u);
    t.nst = kMaxRing;
    while (t.nst > 3 && t.ring_off + (uint32_t)t.nst * t.slot_bytes + 256u + 1024u > kSmemLimit) --t.nst;
    t.bar_off = t.ring_off + (uint32_t)t.nst * t.slot_bytes;
    return t.bar_off + 8u * (2 * kMaxRing + 2) + 1024u <= kSmemLimit;
}

template <int D, int G, int B, int S, int R>
cudaError_t decode_tma_launch(const DecodeArgs& a, DecTma& t, bool* launched, cudaStream_t s) {
    const uint32_t smem = t.bar_off + 8u * (2 * kMaxRing + 2) + 1024u;
    const int64_t units = (int64_t)a.H * t.tiles;
    const int grid = (int)(units < sm_count() ? units : sm_count());
    auto kern = prq_decode_tma_kernel<D, G, B, S, R, false, false>;
    if (a.C > 0 && a.chunk_offset) kern = prq_decode_tma_kernel<D, G, B, S, R, true, true>;
    else if (a.C > 0) kern = prq_decode_tma_kernel<D, G, B, S, R, true, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kPThreads, smem, s>>>(t);
    e = cudaGetLastError();
    if (e == cudaSuccess) *launched = true;
    return e;
}

// Rows per lane: four while the stages' code words are small, else two.
template <int D, int G, int B, int S>
cudaError_t decode_tma_dgbs(const DecodeArgs& a, DecTma& t, bool* launched, cudaStream_t s) {
    constexpr int R = S * B <= 8 ? 4 : 2;
    if (!decode_layout<D, G, B, R>(a, t)) return cudaSuccess;
    return decode_tma_launch<D, G, B, S, R>(a, t, launched, s);
}

template <int D, int G, int B>
cudaError_t decode_tma_dgb(const DecodeArgs& a, bool* launched, cudaStream_t s) {
    constexpr int MPR = D / G;
    DecTma t;
    if (!codec_ctl(&t.ctl)) return cudaSuccess;
    t.codes = a.codes; t.meta = a.meta; t.ids = a.ids; t.cent = a.cent;
    t.chunk_offset = a.chunk_offset; t.chunk_version = a.chunk_version; t.n_chunks = a.n_chunks;
    t.cap = a.cap; t.tok_begin = a.tok_begin; t.n_rows = a.tok_end - a.tok_begin;
    t.out = a.out; t.out_head_stride = a.out_head_stride; t.out_token_stride = a.out_token_stride;
    t.H = a.H; t.C = a.C; t.S = a.S;
    t.meta_words = (int64_t)a.S * a.H * a.cap * MPR;
    t.id_bytes = (int64_t)a.H * a.cap;
    switch (a.S) {
        case 1: return decode_tma_dgbs<D, G, B, 1>(a, t, launched, s);
        case 2: return decode_tma_dgbs<D, G, B, 2>(a, t, launched, s);
        case 3: return decode_tma_dgbs<D, G, B, 3>(a, t, launched, s);
        case 4: return decode_tma_dgbs<D, G, B, 4>(a, t, launched, s);
        default: return cudaSuccess;
    }
}

template <int D, int G>
cudaError_t decode_tma_dg(const DecodeArgs& a, bool* launched, cudaStream_t s) {
    if (a.bits == 2) return decode_tma_dgb<D, G, 2>(a, launched, s);
    if (a.bits == 4) return decode_tma_dgb<D, G, 4>(a, launched, s);
    return cudaSuccess;
}

}  // namespace

#define QVG_TMA_SWITCH(FN, D, G, A, L, S)                  \
    switch (D * 1000 + G) {                                \
        case 64016: return FN<64, 16>(A, L, S);            \
        case 64032: return FN<64, 32>(A, L, S);            \
        case 64064: return FN<64, 64>(A, L, S);            \
        case 128016: return FN<128, 16>(A, L, S);          \
        case 128032: return FN<128, 32>(A, L, S);          \
        case 128064: return FN<128, 64>(A, L, S);          \
        case 128128: return FN<128, 128>(A, L, S);         \
        default: return cudaSuccess;                       \
    }

cudaError_t launch_decode_tma(int D, int G, const DecodeArgs& a, bool* launched, cudaStream_t s) {
    *launched = false;
    const int64_t rows = a.tok_end - a.tok_begin;
    if (rows <= 0 || a.C > kMaxClusters) return cudaSuccess;
    if (a.C > 0 && a.chunk_offset && a.n_chunks > 1024) return cudaSuccess;
    if (rows > (int64_t)INT32_MAX / 2) return cudaSuccess;
    QVG_TMA_SWITCH(decode_tma_dg, D, G, a, launched, s)
}

bool codec_ctl(CodecCtl* ctl) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
    {
        std::lock_guard<std::mutex> lock(g_err_mu);
        if (!g_err_ptr[dev]) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_codec_err) != cudaSuccess) return false;
            g_err_ptr[dev] = static_cast<uint32_t*>(p);
        }
        ctl->err = g_err_ptr[dev];
    }
    ctl->limit = g_limit_ns.load();
    ctl->flags = g_flags.load();
    return true;
}

uint32_t* codec_error_word() {
    CodecCtl c;
    return codec_ctl(&c) ? c.err : nullptr;
}

cudaError_t read_codec_error(uint32_t* out, bool clear, cudaStream_t s) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_codec_err, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && clear) {
        static const uint32_t zero = 0;
        e = cudaMemcpyToSymbolAsync(g_codec_err, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return e;
}

cudaError_t set_codec_debug(unsigned long long wait_limit_ns, uint32_t flags, cudaStream_t s) {
    cudaError_t e = cudaStreamSynchronize(s);   // calls already enqueued keep the old settings
    g_limit_ns.store(wait_limit_ns);
    g_flags.store(flags);
    return e;
}

}  // namespace qvg
