// Exact cluster sums and their rounding to a bf16 mean, in integer
// arithmetic only (no FP64: the B300's double-precision rate is a small
// fraction of its integer rate).
//
// A token value x (bf16, held in fp32) is split into three fixed-point
// windows by the add-and-subtract-a-constant technique: adding 1.5 * 2^(23+u)
// rounds x to a multiple of 2^u and leaves that multiple, as an integer, in
// the low mantissa bits of the fp32 sum.  With units 2^-8, 2^-30 and 2^-52
// every bf16 value with 2^-45 <= |x| < 2^14 (and zero) is
//     x = a1 * 2^-8 + a2 * 2^-30 + a3 * 2^-52,   |a1|, |a2|, |a3| <= 2^22,
// exactly (checked over all 65,536 bf16 patterns).  Values with |x| >= 2^14
// take an exact 128-bit path; values below 2^-45 lose the part below 2^-52.
//
// The mean of a cluster is rounded as the plain definition does it: the
// quotient of the exact sum by the count rounded to double precision (53
// significant bits, nearest-even), then that double rounded to bf16
// (nearest-even).  Both roundings are decided with integer comparisons here
// (valid for means of magnitude 2^-84 .. 2^16).
#pragma once

#include <cstdint>

#include "common.cuh"

namespace qvg {

constexpr float kWin1 = 49152.0f;                // 1.5 * 2^15 -> unit 2^-8
constexpr float kWin2 = 0.01171875f;             // 1.5 * 2^-7 -> unit 2^-30
constexpr float kWin3 = 2.79396772384643555e-09f;  // 1.5 * 2^-29 -> unit 2^-52
constexpr float kWinMax = 16384.0f;              // 2^14: first window's range

typedef __int128 i128;
typedef unsigned __int128 u128;

// Adds x to the window accumulators (int32; each term is at most 2^22 in
// magnitude, so up to 2^8 terms cannot overflow).
__device__ __forceinline__ void window_add(float x, int& a1, int& a2, int& a3) {
    const float v1 = __fadd_rn(x, kWin1);
    a1 += (int)(__float_as_uint(v1) - __float_as_uint(kWin1));
    const float r1 = __fsub_rn(x, __fsub_rn(v1, kWin1));
    const float v2 = __fadd_rn(r1, kWin2);
    a2 += (int)(__float_as_uint(v2) - __float_as_uint(kWin2));
    const float r2 = __fsub_rn(r1, __fsub_rn(v2, kWin2));
    const float v3 = __fadd_rn(r2, kWin3);
    a3 += (int)(__float_as_uint(v3) - __float_as_uint(kWin3));
}

// The same for two values at once (packed fp32 pairs).
__device__ __forceinline__ void window_add2(float2 x, int* a1, int* a2, int* a3) {
    const float2 W1 = make_float2(kWin1, kWin1), W2 = make_float2(kWin2, kWin2), W3 = make_float2(kWin3, kWin3);
    const float2 v1 = f2_add(x, W1);
    a1[0] += (int)(__float_as_uint(v1.x) - __float_as_uint(kWin1));
    a1[1] += (int)(__float_as_uint(v1.y) - __float_as_uint(kWin1));
    const float2 r1 = f2_sub(x, f2_sub(v1, W1));
    const float2 v2 = f2_add(r1, W2);
    a2[0] += (int)(__float_as_uint(v2.x) - __float_as_uint(kWin2));
    a2[1] += (int)(__float_as_uint(v2.y) - __float_as_uint(kWin2));
    const float2 r2 = f2_sub(r1, f2_sub(v2, W2));
    const float2 v3 = f2_add(r2, W3);
    a3[0] += (int)(__float_as_uint(v3.x) - __float_as_uint(kWin3));
    a3[1] += (int)(__float_as_uint(v3.y) - __float_as_uint(kWin3));
}

__device__ __forceinline__ i128 windows_to_i128(int a1, int a2, int a3) {
    return ((i128)a1 << 44) + ((i128)a2 << 22) + (i128)a3;
}

// Exact value of a bf16 pattern in units of 2^-52 (|x| < 2^60; magnitudes
// below 2^-45 are truncated toward zero).
__device__ __forceinline__ i128 bf16_to_i128_units(uint32_t b) {
    const int e = (int)((b >> 7) & 0xFFu);
    int64_t m = (int64_t)((b & 0x7Fu) | (e ? 0x80u : 0u));
    const int ee = e ? e : 1;
    // x = m * 2^(ee - 134); in units 2^-52: m * 2^(ee - 82)
    i128 v;
    if (ee >= 82) v = (i128)m << min(ee - 82, 112);
    else v = (i128)(m >> min(82 - ee, 63));
    return (b & 0x8000u) ? -v : v;
}

__device__ __forceinline__ int clz128(u128 v) {
    const uint64_t hi = (uint64_t)(v >> 64), lo = (uint64_t)v;
    return hi ? __clzll(hi) : 64 + __clzll(lo);
}

// U * 2^sh compared with V * 2^sv (U, V unsigned 128-bit, shifts may be
// negative); returns -1, 0 or 1.  Operands stay below 2^120.
__device__ __forceinline__ int cmp_scaled(u128 U, int sh, u128 V, int sv) {
    const int m = sh < sv ? sh : sv;
    const u128 a = U << (sh - m), b = V << (sv - m);
    return a > b ? 1 : (a < b ? -1 : 0);
}

// bf16 bits of bf16_rn(f64_rn(I * 2^-52 / cnt)), cnt >= 1, from one fp32
// estimate and exact 128-bit comparisons (no division of the wide integer).
// q = U * 2^-52 / cnt (U = |I|) lies in a
// binade [2^ex, 2^(ex+1)) found from an fp32 estimate and confirmed exactly;
// there the bf16 values are k * 2^(ex-7), k = 128..256, and the result is
// one of the two neighbours of q.  With k0 = floor of the estimate of
// q / 2^(ex-7) and mid = (2 k0 + 1) * 2^(ex-8) (when q lies near mid, k0 is
// exact; otherwise either neighbouring midpoint is far), the side of q relative to mid
// is the sign of  U - (2 k0 + 1) * cnt * 2^(ex + 44).  A q within half a
// double ulp of mid (|q - mid| <= 2^(ex-53)) rounds to mid in double
// precision first and then to the even neighbour.
__device__ __forceinline__ uint16_t mean_bf16_bits(i128 I, uint32_t cnt) {
    if (I == 0) return 0;
    const bool neg = I < 0;
    const u128 U = neg ? (u128)(-I) : (u128)I;
    const int bl = 128 - clz128(U);
    const int sh = bl > 24 ? bl - 24 : 0;
    const float qf = __fdiv_rn((float)(uint32_t)(U >> sh), (float)cnt);   // q ~ qf * 2^(sh-52)
    int ex;
    frexpf(qf, &ex);                                   // qf in [2^(ex-1), 2^ex)
    ex = ex - 1 + sh - 52;                             // estimated binade of q
    // exact binade: 2^ex <= q < 2^(ex+1)  <=>  cnt * 2^(ex+52) <= U < cnt * 2^(ex+53)
    if (cmp_scaled(U, 0, (u128)cnt, ex + 52) < 0) --ex;
    else if (cmp_scaled(U, 0, (u128)cnt, ex + 53) >= 0) ++ex;
    // k estimate of q / 2^(ex-7), in [128, 256)
    const float kq = ldexpf(qf, sh - 52 - (ex - 7));
    const int k0 = (int)floorf(kq);                  // q/2^(ex-7) lies within 2^-12 of kq
    const u128 Mc = (u128)(uint32_t)(2 * k0 + 1) * (u128)cnt;
    // side of q relative to mid: U vs Mc * 2^(ex - 8 + 52)
    const int side = cmp_scaled(U, 0, Mc, ex + 44);
    // tie: |U - Mc * 2^(ex+44)| <= cnt * 2^(ex-1)   (both sides times 2^52)
    bool tie;
    {
        const int m = (ex - 1) < 0 ? (ex - 1) : 0;     // common unit 2^m (m <= 0)
        const u128 a = U << (0 - m), b = Mc << (ex + 44 - m);
        const u128 d = a > b ? a - b : b - a;
        tie = d <= ((u128)cnt << (ex - 1 - m));
    }
    int k = (tie || side == 0) ? ((k0 & 1) ? k0 + 1 : k0) : (side > 0 ? k0 + 1 : k0);
    int e = ex;
    if (k >= 256) { k >>= 1; ++e; }
    uint32_t bits;
    if (e + 127 >= 255) bits = 0x7F80u;
    else if (e + 127 <= 0) bits = 0u;
    else bits = ((uint32_t)(e + 127) << 7) | ((uint32_t)k & 0x7Fu);
    return (uint16_t)(bits | (neg ? 0x8000u : 0u));
}

// The same result, taken from the fp32 estimate alone when no bf16 rounding
// midpoint can lie between it and q.  The estimate U' / cnt with U' = U >> sh
// (24 significant bits) is within 2^-22 of q relative (truncation < 2^-23,
// the correctly rounded quotient 2^-24; cnt < 2^24 is exact in fp32), that is
// within 4 units in the last place of the estimate qf.  The bits of qf below
// the bf16 mantissa (r) are at least 16 units from the midpoint 0x8000, so q,
// RN_f64(q) and qf lie on the same side of every midpoint and round to the
// same bf16 value; the rounding carries into the exponent where it must
// (also when qf and q lie on either side of a power of two).  Otherwise, and
// near the ends of the bf16 range, the exact comparisons decide.
__device__ __forceinline__ uint16_t mean_bf16_bits_fast(i128 I, uint32_t cnt) {
    if (I == 0) return 0;
    const bool neg = I < 0;
    const u128 U = neg ? (u128)(-I) : (u128)I;
    const int bl = 128 - clz128(U);
    const int sh = bl > 24 ? bl - 24 : 0;
    const float qf = __fdiv_rn((float)(uint32_t)(U >> sh), (float)cnt);
    const uint32_t b = __float_as_uint(qf);
    const uint32_t r = b & 0xFFFFu;
    const int e = (int)(b >> 23) - 127 + sh - 52;           // q ~ 1.m * 2^e
    if (cnt < (1u << 24) && (r > 0x8000u + 16u || r + 16u < 0x8000u) && e > -126 && e < 126) {
        uint32_t bits = ((uint32_t)(e + 127) << 7) | ((b >> 16) & 0x7Fu);
        if (r > 0x8000u) ++bits;
        return (uint16_t)(bits | (neg ? 0x8000u : 0u));
    }
    return mean_bf16_bits(I, cnt);
}

}  // namespace qvg
