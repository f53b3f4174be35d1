// Element arithmetic of the operand quantiser, shared by the quantiser
// kernels (quant.cu) and the grouped GEMM's fused activation quantiser
// (gemm.cu), so that both produce the same codes and scales bit for bit.
// The formats, their rounding and the scale rule are stated in quant.cu.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

namespace fp8g {

// FMT 0: E4M3, 1: E5M2, 2: E2M1 (FP4, two codes per byte), 3: E2M3, 4: E3M2
// (FP6, four codes per three bytes).  Largest finite value kMax = mmax *
// 2^kEmax; kMantOver is the fp32 mantissa field above which a value m 2^E
// (1 <= m < 2) exceeds mmax * 2^E (mmax = 1.75, 1.5 or 1.875).
template <int FMT>
struct Fp8Fmt;
template <>
struct Fp8Fmt<0> {
    static constexpr float kMax = 448.0f;
    static constexpr int kEmax = 8;
    static constexpr uint32_t kMantOver = 0x600000u;
};
template <>
struct Fp8Fmt<1> {
    static constexpr float kMax = 57344.0f;
    static constexpr int kEmax = 15;
    static constexpr uint32_t kMantOver = 0x600000u;
};
template <>
struct Fp8Fmt<2> {
    static constexpr float kMax = 6.0f;
    static constexpr int kEmax = 2;
    static constexpr uint32_t kMantOver = 0x400000u;
};
template <>
struct Fp8Fmt<3> {
    static constexpr float kMax = 7.5f;
    static constexpr int kEmax = 2;
    static constexpr uint32_t kMantOver = 0x700000u;
};
template <>
struct Fp8Fmt<4> {
    static constexpr float kMax = 28.0f;
    static constexpr int kEmax = 4;
    static constexpr uint32_t kMantOver = 0x600000u;
};

// Two fp32 values -> their codes, lo first: FP8 and FP6 two bytes (lo at the
// lower address; FP6 codes in the low six bits), E2M1 one byte (lo in the low
// nibble).  NaN, which E2M1 and FP6 cannot hold, becomes their largest
// positive value (E2M1 code 7, FP6 code 0x1F).
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
    uint32_t v;
    if constexpr (FMT == 2) {
        asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
            : "=r"(v)
            : "f"(hi), "f"(lo));
        if (isnan(lo)) v = (v & 0xF0u) | 0x07u;
        if (isnan(hi)) v = (v & 0x0Fu) | 0x70u;
        return v;
    } else {
        uint16_t r;
        if constexpr (FMT == 0)
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
        else if constexpr (FMT == 1)
            asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
        else if constexpr (FMT == 3)
            asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
        else
            asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
        v = r;
    }
    constexpr uint32_t kNan = FMT >= 3 ? 0x1Fu : 0x7Fu;
    if (isnan(lo)) v = (v & 0xFF00u) | kNan;
    if (isnan(hi)) v = (v & 0x00FFu) | (kNan << 8);
    return v;
}

// Codes of four values, first value lowest.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x4(float x0, float x1, float x2, float x3) {
    return fp8x2<FMT>(x0, x1) | (fp8x2<FMT>(x2, x3) << (FMT == 2 ? 8 : 16));
}

__device__ __forceinline__ float absmax8(const float4 a, const float4 b) {
    // fmaxf ignores a NaN operand
    float m = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w)));
    m = fmaxf(m, fmaxf(fmaxf(fabsf(b.x), fabsf(b.y)), fmaxf(fabsf(b.z), fabsf(b.w))));
    return m;
}

// Smallest power of two s with fmax s >= amax (amax >= 0, not NaN), as an
// exponent clamped to [-126, 127].  With amax = m 2^E, 1 <= m < 2 and
// fmax = 1.75 2^emax: e = E - emax when m <= 1.75 and E - emax + 1 otherwise
// (m > 1.75 <=> mantissa field above 0x600000).
template <int FMT>
__device__ __forceinline__ float pow2_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    const uint32_t bits = __float_as_uint(amax);
    int e;
    if (bits >= 0x7F800000u) {
        e = 127;
    } else {
        const int ex = (int)(bits >> 23);
        if (ex == 0) {
            e = -126;
        } else {
            e = (ex - 127) - Fp8Fmt<FMT>::kEmax + ((bits & 0x7FFFFFu) > Fp8Fmt<FMT>::kMantOver ? 1 : 0);
        }
        e = max(-126, min(127, e));
    }
    return __uint_as_float((uint32_t)(e + 127) << 23);
}

// Eight bf16 values (one 16-byte word, first value lowest) widened exactly
// to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float4 &a, float4 &b) {
    a = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                    __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    b = make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u),
                    __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u));
}

// Eight consecutive values of the source at element offset `off` (a multiple
// of 8), fp32 or bf16 (widened exactly).
template <bool BF16>
__device__ __forceinline__ void load8(const void *x, int64_t off, float4 &a, float4 &b) {
    if constexpr (BF16) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + off));
        bf16x8_to_f32(u, a, b);
    } else {
        const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(x) + off);
        a = __ldg(p);
        b = __ldg(p + 1);
    }
}

// Divide by a power-of-two scale: x * (1/s) is exactly x / s (both are the
// exact real x 2^-e rounded once), and 1/s is exact for s in 2^-126..2^127.
template <int FMT>
__device__ __forceinline__ uint2 quant8_pow2(const float4 a, const float4 b, float s) {
    const float r = __frcp_rn(s);
    uint2 o;
    o.x = fp8x4<FMT>(__fmul_rn(a.x, r), __fmul_rn(a.y, r), __fmul_rn(a.z, r), __fmul_rn(a.w, r));
    o.y = fp8x4<FMT>(__fmul_rn(b.x, r), __fmul_rn(b.y, r), __fmul_rn(b.z, r), __fmul_rn(b.w, r));
    return o;
}

}  // namespace fp8g
