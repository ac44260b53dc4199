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
// (nearest-even).  Both roundings are done on integers here.
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

// bf16 bits of bf16_rn(f64_rn(I * 2^-52 / cnt)), cnt >= 1.
__device__ __forceinline__ uint16_t mean_bf16_bits(i128 I, uint32_t cnt) {
    if (I == 0) return 0;
    const bool neg = I < 0;
    u128 U = neg ? (u128)(-I) : (u128)I;
    const int bl = 128 - clz128(U);
    const int k = bl < 86 ? 86 - bl : 0;   // scale so the quotient has >= 54 bits
    U <<= k;
    // 128-bit by 32-bit long division, 32 bits at a time
    uint64_t rem = 0;
    u128 q = 0;
#pragma unroll
    for (int li = 3; li >= 0; --li) {
        const uint64_t cur = (rem << 32) | (uint64_t)(uint32_t)(U >> (32 * li));
        const uint64_t ql = cur / cnt;
        rem = cur - ql * cnt;
        q |= (u128)ql << (32 * li);
    }
    // first rounding: to 53 significant bits, nearest-even, remainder sticky
    int sh = (128 - clz128(q)) - 53;
    const u128 low = q & (((u128)1 << sh) - 1);
    const u128 half = (u128)1 << (sh - 1);
    uint64_t q53 = (uint64_t)(q >> sh);
    if (low > half || (low == half && (rem != 0 || (q53 & 1)))) ++q53;
    if (q53 >> 53) { q53 >>= 1; ++sh; }
    // second rounding: the double to 8 significant bits, nearest-even
    const uint64_t low2 = q53 & ((1ull << 45) - 1);
    uint32_t m8 = (uint32_t)(q53 >> 45);
    int sh2 = 45;
    if (low2 > (1ull << 44) || (low2 == (1ull << 44) && (m8 & 1))) ++m8;
    if (m8 == 256) { m8 = 128; ++sh2; }
    // value = m8 * 2^(sh + sh2 - 52 - k), m8 in [128, 255]
    const int E = 7 + sh + sh2 - 52 - k;
    uint32_t bits;
    if (E + 127 >= 255) bits = 0x7F80u;          // outside the supported range
    else if (E + 127 <= 0) bits = 0u;
    else bits = ((uint32_t)(E + 127) << 7) | (m8 & 0x7Fu);
    return (uint16_t)(bits | (neg ? 0x8000u : 0u));
}

}  // namespace qvg
