// Shared device helpers of the KV-cache codec kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/qvg.h"

namespace qvg {

constexpr int kMaxClusters = 256;
constexpr int kMaxStages = 4;

// ----------------------------------------------------------- conversions --

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFF)));
}

// fp64 -> bf16 with a single round-to-nearest-even: truncate to fp32 and
// make the fp32 sticky (round to odd), which then rounds correctly to the
// 8-bit bf16 significand (fp32 carries 16 more bits).
__device__ __forceinline__ uint16_t f64_to_bf16_rn(double v) {
    float t = __double2float_rz(v);
    uint32_t u = __float_as_uint(t);
    if ((double)t != v) u |= 1u;
    float f = __uint_as_float(u);
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------------- the quantiser

struct GroupParams {
    float s, z, inv;
    uint32_t meta;   // low half fp16 scale, high half fp16 zero
};

// Scale / zero / reciprocal of one group from its fp32 min and max, with
// L = 2^b - 1 levels above the zero-point (3 for 2-bit codes, 15 for 4-bit).
// s = fp16(range / L) needs the correctly rounded quotient: with y = RN(1/L),
// q0 = RN(range*y), rem = range - q0*L (exact in one fma) and RN(q0 + rem*y)
// is it (Markstein's correction step; for L = 3 and 15 it was checked
// against IEEE division for every finite non-negative fp32 range, subnormals
// included).  An infinite range is passed through, as division would.
template <int L>
__device__ __forceinline__ GroupParams group_params(float mn, float mx) {
    constexpr float Lf = (float)L, y = 1.0f / (float)L;
    GroupParams p;
    const float range = __fsub_rn(mx, mn);
    const float q0 = __fmul_rn(range, y);
    const float rem = __fmaf_rn(q0, -Lf, range);
    float s32 = __fmaf_rn(rem, y, q0);
    if (!(range < INFINITY)) s32 = range;
    const __half2 sz = __floats2half2_rn(s32, mn);    // low half: scale, high half: zero-point
    const float2 f = __half22float2(sz);
    p.s = f.x;
    p.z = f.y;
    p.inv = (p.s != 0.0f) ? __frcp_rn(p.s) : 0.0f;
    p.meta = *reinterpret_cast<const uint32_t*>(&sz);
    return p;
}

// --------------------------------------------- Blackwell packed fp32 pairs --
// FADD2 / FMUL2 / FFMA2 (sm_100+) perform two independent IEEE single-precision
// operations (round to nearest even) in one instruction; each lane gives
// exactly the result of the scalar operation.  a - b is formed as
// fma(b, -1, a): b * -1 is exact, so the single rounding is that of a - b.

__device__ __forceinline__ float2 f2_add(float2 a, float2 b) { return __fadd2_rn(a, b); }
// Caution: the code generator may fuse a packed product with a following
// packed addition into one FFMA2 -- even when both are written with explicit
// round-to-nearest -- so a product whose rounding matters must not feed an
// addition directly.  In the quantiser the clamp of t = (r - z) * inv sits
// between the product and the rounding addition.
__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) { return __fmul2_rn(a, b); }

__device__ __forceinline__ float2 f2_fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 f2_sub(float2 a, float2 b) {
    return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a);
}

// Three-input minimum / maximum (sm_100+), NaN-ignoring like fminf/fmaxf.
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// --------------------------------------------------------------- memory ----

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_v4_stream(void* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

}  // namespace qvg
