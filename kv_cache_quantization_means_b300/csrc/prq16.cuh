// One thread's share of progressive residual quantisation: a run of
// consecutive channels of a token row (Quant VideoGen explainer, Sommario tecnico
// sec. 2B: each stage re-quantises what the previous stages left; decoding
// dequantises and sums the stages onto the centroid).
//
// Arithmetic per element and stage (identical, operation for operation, to
// the plain statement of the quantiser):
//   t = r - z                    one IEEE single subtraction
//   y = t / s                    IEEE single division, correctly rounded
//   q = clamp(rint(y), 0, L)     rint by adding and subtracting 1.5 * 2^23,
//                                whose IEEE sum rounds to an integer with
//                                ties to even
//   d = fma(q, s, z)             q*s is exact, so this is q*s + z rounded once
//   r = r - d
// The division: with inv = RN(1/s), q0 = RN(t * inv) is within one ulp of
// t/s, the remainder t - q0*s is exact in one fma, and RN(q0 + rem * inv) is
// the correctly rounded quotient (Markstein's correction step: P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990).  That holds while nothing
// overflows or underflows near a rounding boundary.  A group whose extremes
// satisfy min r - z >= -s/2 and max r - z <= (L + 1/4) s has every quotient
// in [-1/2, L + 1/4] and so every rint(y) in [0, L] already (rounding is
// monotone): it needs neither the clamp nor any other range care.  When any
// group of the warp is not of that kind -- in practice one whose zero-point
// rounded far from its minimum, or non-finite values -- the whole warp clamps
// t to [-s, (L+1) s] before dividing and the quotient to [0, L] after, which
// is exact for every group.  All 32 lanes must call the stage together.
// Every 16 2-bit codes go to one 32-bit word, element k at bits 2k, 2k+1;
// with 4-bit codes (levels 0..15, s = range / 15) every 8 codes go to one
// word, element k at bits 4k .. 4k+3.  The words are assembled in fp32: each
// half-word is sum q_k * 2^(b k) accumulated exactly onto 2^23 by fmas, whose
// low 16 bits are then spliced together.
#pragma once

#include "common.cuh"

namespace qvg {

constexpr float kRintMagic = 12582912.0f;   // 1.5 * 2^23
constexpr uint32_t kQMagicBits = 0x4B000000u;  // bit pattern of 2^23

__device__ __forceinline__ void unpack16(const uint4& lo, const uint4& hi, float* f) {
    f[0] = bf16_lo(lo.x); f[1] = bf16_hi(lo.x);
    f[2] = bf16_lo(lo.y); f[3] = bf16_hi(lo.y);
    f[4] = bf16_lo(lo.z); f[5] = bf16_hi(lo.z);
    f[6] = bf16_lo(lo.w); f[7] = bf16_hi(lo.w);
    f[8] = bf16_lo(hi.x); f[9] = bf16_hi(hi.x);
    f[10] = bf16_lo(hi.y); f[11] = bf16_hi(hi.y);
    f[12] = bf16_lo(hi.z); f[13] = bf16_hi(hi.z);
    f[14] = bf16_lo(hi.w); f[15] = bf16_hi(hi.w);
}

__device__ __forceinline__ void pack16_bf16(const float* f, uint4& lo, uint4& hi) {
    lo.x = pack_bf16x2(f[0], f[1]);   lo.y = pack_bf16x2(f[2], f[3]);
    lo.z = pack_bf16x2(f[4], f[5]);   lo.w = pack_bf16x2(f[6], f[7]);
    hi.x = pack_bf16x2(f[8], f[9]);   hi.y = pack_bf16x2(f[10], f[11]);
    hi.z = pack_bf16x2(f[12], f[13]); hi.w = pack_bf16x2(f[14], f[15]);
}

// r[i] -= c[i] (fp32, exact for bf16 operands of close magnitude, one
// rounding otherwise).
__device__ __forceinline__ void sub16(float* r, const float* c) {
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        float2 d = f2_sub(make_float2(r[i], r[i + 1]), make_float2(c[i], c[i + 1]));
        r[i] = d.x; r[i + 1] = d.y;
    }
}

// Correctly rounded t / s from inv = RN(1/s) and ns = -s, two lanes at a
// time (Markstein's correction step, see the top of this file).
__device__ __forceinline__ float2 div2_rn(float2 t, float2 inv, float2 ns) {
    const float2 q0 = f2_mul(t, inv);
    const float2 rem = f2_fma(q0, ns, t);
    return f2_fma(rem, inv, q0);
}

__device__ __forceinline__ float div_rn_markstein(float t, float inv, float ns) {
    const float q0 = __fmul_rn(t, inv);
    const float rem = __fmaf_rn(q0, ns, t);
    return __fmaf_rn(rem, inv, q0);
}

// One code word from PER = 32/B codes held as exact small floats, pairs
// (q_2j, q_2j+1): each 16-bit half is sum q_k 2^(B k) accumulated exactly onto
// 2^23 (whose low mantissa bits then hold it), the two halves spliced.
template <int B>
__device__ __forceinline__ uint32_t pack_word(const float2* qv) {
    constexpr int PER = 32 / B, HALF = PER / 2;
    float2 lo = make_float2(8388608.0f, 0.0f), hi = make_float2(8388608.0f, 0.0f);
#pragma unroll
    for (int j = 0; j < HALF / 2; ++j) {
        const float2 w = make_float2((float)(1u << (B * 2 * j)), (float)(1u << (B * (2 * j + 1))));
        lo = f2_fma(qv[j], w, lo);
        hi = f2_fma(qv[j + HALF / 2], w, hi);
    }
    const float l = __fadd_rn(lo.x, lo.y), h = __fadd_rn(hi.x, hi.y);
    return prmt(__float_as_uint(l), __float_as_uint(h), 0x5410u);
}

// One stage over the thread's CPT channels (a multiple of 16); the group of
// G = CPT * TPG channels spans TPG consecutive lanes (TPG > 1: all 32 lanes
// must call this together).  B-bit codes (B = 2 or 4): writes CPT*B/32 code
// words to `codes`; `meta` receives the group's (scale, zero) word.  When
// `update` the residual is replaced by what the stage leaves; `acc` (may be
// null) gets the dequantised values added.
// The element work of one stage, given the group's parameters (see
// quant_stage); CLAMP selects the clamped form.
template <int CPT, int B, bool CLAMP>
__device__ __forceinline__ void quant_words(float* r, bool update, float* acc, uint32_t* codes, const GroupParams& p) {
    constexpr float L = (float)((1 << B) - 1);
    constexpr int PER = 32 / B;                      // codes per word
    const float lo = -p.s, hi = (L + 1.0f) * p.s;
    const float2 z2 = make_float2(p.z, p.z), inv2 = make_float2(p.inv, p.inv), ns2 = make_float2(-p.s, -p.s);
    const float2 s2 = make_float2(p.s, p.s), m2 = make_float2(kRintMagic, kRintMagic);
#pragma unroll
    for (int w = 0; w < CPT / PER; ++w) {
        float2 qv[PER / 2];
#pragma unroll
        for (int k = 0; k < PER; k += 2) {
            const int i = PER * w + k;
            float2 t = f2_sub(make_float2(r[i], r[i + 1]), z2);
            if (CLAMP) {
                t.x = fminf(fmaxf(t.x, lo), hi);
                t.y = fminf(fmaxf(t.y, lo), hi);
            }
            float2 y = div2_rn(t, inv2, ns2);
            if (CLAMP) {
                y.x = fminf(fmaxf(y.x, 0.0f), L);              // NaN -> 0
                y.y = fminf(fmaxf(y.y, 0.0f), L);
            }
            qv[k / 2] = f2_sub(f2_add(y, m2), m2);           // rint(y), in [0, L]
        }
        codes[w] = pack_word<B>(qv);
        if (update || acc) {
#pragma unroll
            for (int k = 0; k < PER; k += 2) {
                const int i = PER * w + k;
                const float2 d = f2_fma(qv[k / 2], s2, z2);
                if (update) {
                    const float2 nr = f2_sub(make_float2(r[i], r[i + 1]), d);
                    r[i] = nr.x; r[i + 1] = nr.y;
                }
                if (acc) {
                    const float2 na = f2_add(make_float2(acc[i], acc[i + 1]), d);
                    acc[i] = na.x; acc[i + 1] = na.y;
                }
            }
        }
    }
}

template <int CPT, int TPG, int B = 2, int OFF1 = 1, int OFF2 = 2, int OFF3 = 4>
__device__ __forceinline__ void quant_stage(float* r, bool update, float* acc, uint32_t* codes, uint32_t& meta) {
    static_assert(B == 2 || B == 4, "2- or 4-bit codes");
    constexpr float L = (float)((1 << B) - 1);
    float m0 = fmin3(r[0], r[1], r[2]), M0 = fmax3(r[0], r[1], r[2]);
    float m1 = fmin3(r[3], r[4], r[5]), M1 = fmax3(r[3], r[4], r[5]);
#pragma unroll
    for (int i = 6; i + 3 < CPT; i += 4) {
        m0 = fmin3(m0, r[i], r[i + 1]);
        M0 = fmax3(M0, r[i], r[i + 1]);
        m1 = fmin3(m1, r[i + 2], r[i + 3]);
        M1 = fmax3(M1, r[i + 2], r[i + 3]);
    }
    // CPT % 4 == 0: the loop stops with r[CPT-2], r[CPT-1] left
    float mn = fmin3(m0, m1, fminf(r[CPT - 2], r[CPT - 1]));
    float mx = fmax3(M0, M1, fmaxf(r[CPT - 2], r[CPT - 1]));
    // the lanes of a group: OFF1, OFF2, OFF3 apart (up to TPG = 8)
    if (TPG > 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, OFF1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, OFF1));
    }
    if (TPG > 2) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, OFF2));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, OFF2));
    }
    if (TPG > 4) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, OFF3));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, OFF3));
    }
    // a zero extreme is taken as +0 so the stored bits do not depend on the
    // order in which equal extremes are met
    mn = __fadd_rn(mn, 0.0f);
    mx = __fadd_rn(mx, 0.0f);
    const GroupParams p = group_params<(1 << B) - 1>(mn, mx);
    meta = p.meta;
    // Every quotient of the group lies between those of its extremes.  With
    // (min - z) >= -s/2 and (max - z) <= (L + 1/4) s (both products exact: s
    // is an fp16 value) every rint(y) is already in [0, L].
    const bool plain = __fsub_rn(mn, p.z) >= -0.5f * p.s && __fsub_rn(mx, p.z) <= (L + 0.25f) * p.s;
    // Otherwise (any lane of the warp, so that the branch is uniform) t is
    // clamped to [-s, (L+1) s] first (exact bounds): inside, the quotient is
    // unchanged and stays in [-1, L+1], where the division is exact; outside,
    // the clamped and the true quotient both give code 0 or L.  s = 0 gives
    // t = 0 and y = 0; a NaN goes to a bound, then to 0.  The clamped form is
    // exact for every group, so lanes whose own group is plain may take it too.
    const bool clamp = !__all_sync(0xffffffffu, plain);
    if (clamp) quant_words<CPT, B, true>(r, update, acc, codes, p);
    else quant_words<CPT, B, false>(r, update, acc, codes, p);
}

// 16-channel form (one code word).
template <int TPG>
__device__ __forceinline__ uint32_t quant_stage16(float* r, bool update, float* acc, uint32_t& meta) {
    uint32_t c;
    quant_stage<16, TPG>(r, update, acc, &c, meta);
    return c;
}

// acc[k] += q_k * s + z for the 16 codes of `code` (element k at bits 2k).
__device__ __forceinline__ void dequant_add16(float* acc, uint32_t code, uint32_t meta) {
    const float s = f16_bits_to_f32(meta), z = f16_bits_to_f32(meta >> 16);
    const float2 s2 = make_float2(s, s), z2 = make_float2(z, z);
    const float2 b2 = make_float2(8388608.0f, 8388608.0f);
    uint32_t t[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) t[i] = (code >> (2 * i)) & 0x03030303u;   // byte j = q_{4j+i}
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        const uint32_t ba = prmt(t[k & 3], kQMagicBits, 0x7650u | (uint32_t)(k >> 2));
        const uint32_t bb = prmt(t[(k + 1) & 3], kQMagicBits, 0x7650u | (uint32_t)((k + 1) >> 2));
        const float2 q = f2_sub(make_float2(__uint_as_float(ba), __uint_as_float(bb)), b2);
        const float2 d = f2_fma(q, s2, z2);
        const float2 na = f2_add(make_float2(acc[k], acc[k + 1]), d);
        acc[k] = na.x; acc[k + 1] = na.y;
    }
}

// acc[k] += q_k * s + z for the 8 four-bit codes of `code` (element k at bits 4k).
__device__ __forceinline__ void dequant_add8x4(float* acc, uint32_t code, uint32_t meta) {
    const float s = f16_bits_to_f32(meta), z = f16_bits_to_f32(meta >> 16);
    const float2 s2 = make_float2(s, s), z2 = make_float2(z, z);
    const float2 b2 = make_float2(8388608.0f, 8388608.0f);
    const uint32_t t[2] = {code & 0x0F0F0F0Fu, (code >> 4) & 0x0F0F0F0Fu};   // byte j of t[i] = q_{2j+i}
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        const uint32_t ba = prmt(t[0], kQMagicBits, 0x7650u | (uint32_t)(k >> 1));
        const uint32_t bb = prmt(t[1], kQMagicBits, 0x7650u | (uint32_t)(k >> 1));
        const float2 q = f2_sub(make_float2(__uint_as_float(ba), __uint_as_float(bb)), b2);
        const float2 d = f2_fma(q, s2, z2);
        const float2 na = f2_add(make_float2(acc[k], acc[k + 1]), d);
        acc[k] = na.x; acc[k + 1] = na.y;
    }
}

// Decodes channels 16c .. 16c+15 of one row of an encoded tensor to bf16:
// `row` indexes the [H][cap] plane (h * cap + token), stage s of the row
// lies stage_rows (= H * cap) rows further; the centroid (C > 0) is
// cent[h][ids[row]].
template <int D, int B>
__device__ __forceinline__ void decode_chunk(const uint32_t* codes, const uint32_t* meta, const uint8_t* ids,
                                             const uint16_t* cent, int64_t row, int h, int c, int64_t stage_rows,
                                             int C, int S, int G, uint4& o0, uint4& o1) {
    constexpr int WPT = B / 2;          // code words per 16 channels and stage
    constexpr int WPR = D * B / 32;     // code words per row and stage
    const int mpr = D / G;
    float acc[16];
    if (C > 0) {
        const int id = ids[row];
        const uint16_t* cr = cent + ((int64_t)h * C + min(id, C - 1)) * D + c * 16;
        const uint4 c0 = __ldg(reinterpret_cast<const uint4*>(cr));
        const uint4 c1 = __ldg(reinterpret_cast<const uint4*>(cr + 8));
        unpack16(c0, c1, acc);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
    }
    for (int s = 0; s < S; ++s) {
        const int64_t srow = (int64_t)s * stage_rows + row;
        const uint32_t* cw = codes + srow * WPR + c * WPT;
        const uint32_t mw = __ldg(meta + srow * mpr + (c * 16) / G);
        if constexpr (B == 2) {
            dequant_add16(acc, __ldg(cw), mw);
        } else {
            dequant_add8x4(acc, __ldg(cw), mw);
            dequant_add8x4(acc + 8, __ldg(cw + 1), mw);
        }
    }
    pack16_bf16(acc, o0, o1);
}

}  // namespace qvg
