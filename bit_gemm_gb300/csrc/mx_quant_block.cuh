// mx_quant_block.cuh -- quantize_block for one block of 32 elements, on the
// device (sm_103a): the rounding shared by the quantize kernels and by the
// block_matmul kernel that quantizes its activations on the fly.
//
// quantize_block of "A Dialect Is a Set of Co-Designed Decisions: Designing for
// MX Quantization in MLIR" ("The four ops") with the element and scale
// encodings of "Bit Layout" ("The E2M1 element", "The E8M0 shared scale",
// "Reference encode and decode").  Built without flush-to-zero.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "mx_internal.h"

namespace mx {

// ------------------------------------------------------------ element round
//
// y = |x| * 2^-e is formed by one exact binary32 multiply (a power of two;
// it also normalizes subnormal inputs), then rounded with integer operations
// on the bits of y.  Every rule below rounds ties to the LOWER magnitude
// (the first-index argmin of "Reference encode and decode").

// E4M3FN, y in [2^-6, 512): keep 3 mantissa bits rounding the 20 dropped bits
// half-down (add 2^19 - 1, truncate; a carry moves into the exponent as it
// should), re-bias the exponent 127 -> 7 (subtract 120 << 23), and read the
// 7-bit code from bits 20..26 -- one add and one shift -- then saturate at
// 0x7E = 448.
__device__ __forceinline__ uint32_t e4m3_normal_code(uint32_t ybits) {
    return min((ybits + (0x7FFFFu - 0x3C000000u)) >> 20, 0x7Eu);
}

// E4M3FN, y in [0, 2^-6): the subnormal quantum is 2^-9, so the code is the
// nearest integer to 512 y with ties down, ceil(512 y - 1/2).  The fused
// multiply-add rounds once; the result is exact whenever 512 y >= 1/4, and
// below that every value rounds into [-1/2, -1/4], whose ceiling is 0.  k = 8
// is the first normal 2^-6, whose code is also 8.
__device__ __forceinline__ uint32_t e4m3_subnormal_code(float y) {
    return (uint32_t)__float2int_ru(__fmaf_rn(y, 512.0f, -0.5f));
}

// E2M1, y in [0, 8): for y >= 1 keep 1 mantissa bit rounding half-down (add
// 2^21 - 1), re-bias so that 1.0 is code 2 (subtract 252 << 22), saturate at
// 7 = 6.0; below 1 the grid is {0, 0.5, 1}, so count the midpoints 0.25 and
// 0.75 strictly below y.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
    const uint32_t b = __float_as_uint(y);
    const uint32_t hi = min((b + (0x1FFFFFu - 0x3F000000u)) >> 22, 7u);
    const uint32_t lo = (uint32_t)(y > 0.25f) + (uint32_t)(y > 0.75f);
    return y < 1.0f ? lo : hi;
}

// Quantize the 8 elements a thread owns, given the block's max and min
// |bits|.  Returns the scale byte; fills 8 codes (sign included).
//
// Fast path (the block's exponent e >= -120, so every element that reaches
// the normal code range is itself a normal binary32): dividing by 2^e is a
// subtraction of e from the exponent field, which folds into the rounding
// constant -- one add and one shift per element.  The sign of a nonzero
// element is its bit 31.  Elements below the format's smallest normal (rare;
// zeros included) and blocks with e < -120 take the exact multiply path.
template <int FMT>
__device__ __forceinline__ uint32_t quantize8(const uint32_t (&u)[8], uint32_t amax_bits, uint32_t amin_bits,
                                              uint32_t (&code)[8]) {
    constexpr int kEmax = FMT == FMT_E2M1 ? 2 : 8;
    constexpr uint32_t kSign = FMT == FMT_E2M1 ? 0x8u : 0x80u;
    if (amax_bits >= 0x7F800000u) {  // NaN or infinity in the block: poison it
#pragma unroll
        for (int i = 0; i < 8; ++i) code[i] = 0;
        return 0xFFu;
    }
    if (amax_bits == 0u) {  // all-zero block
#pragma unroll
        for (int i = 0; i < 8; ++i) code[i] = 0;
        return 127u;
    }
    // floor(log2 amax), exactly, from the bit pattern (subnormals included).
    const int fe = (int)(amax_bits >> 23);
    const int E = fe ? fe - 127 : (31 - __clz((int)amax_bits)) - 149;
    int e = E - kEmax;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    // smallest normal of the element format, as a bound on |x|: 2^-6 * 2^e
    // (E4M3) or 1.0 * 2^e (E2M1); below it the element takes the slow path
    const int small_exp = (FMT == FMT_E2M1 ? 0 : -6) + e;
    const bool fast = e >= -120;
    const uint32_t small_bits = fast ? (uint32_t)(small_exp + 127) << 23 : 0xFFFFFFFFu;
    if (fast && FMT == FMT_E4M3 && amin_bits >= small_bits) {
        // code = round-half-down to 3 mantissa bits of |x| / 2^e, re-biased:
        // ((bits(|x|) - (e << 23)) + 2^19 - 1 - (120 << 23)) >> 20, saturated at 0x7E
        const uint32_t k = 0x7FFFFu - 0x3C000000u - ((uint32_t)e << 23);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t a = u[i] & 0x7FFFFFFFu;
            code[i] = min((a + k) >> 20, 0x7Eu) | ((u[i] >> 24) & kSign);
        }
        return (uint32_t)(e + 127);
    }
    // exact multiply path: y = |x| * 2^-e (e <= 125, so 2^-e is a normal binary32)
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
    if (FMT == FMT_E2M1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y = __fmul_rn(__uint_as_float(u[i] & 0x7FFFFFFFu), inv);
            // sign bit when x < 0: the pattern is above 0x80000000 (-0.0 is not)
            code[i] = e2m1_code(y) | (u[i] > 0x80000000u ? kSign : 0u);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float y = __fmul_rn(__uint_as_float(u[i] & 0x7FFFFFFFu), inv);
            const uint32_t c = y < 0.015625f ? e4m3_subnormal_code(y) : e4m3_normal_code(__float_as_uint(y));
            code[i] = c | (u[i] > 0x80000000u ? kSign : 0u);
        }
    }
    return (uint32_t)(e + 127);
}

// ------------------------------------------------- bf16: one thread per block
//
// A bf16 element has 8 significant bits, so y = x * 2^-e * (1 - 2^-12) is
// exact in binary32 (8 + 12 bits).  It sits below x * 2^-e by less than 2^-11
// of its magnitude, which is less than the distance (at least one bf16 unit in
// the last place) from any value that is not a tie to the nearest rounding
// midpoint of either element grid; a tie moves strictly below its midpoint.
// The hardware conversion (round to nearest even, saturating at the largest
// finite code) therefore rounds every tie to the LOWER magnitude and every
// other value as exact rounding would: the first-index argmin rule of
// "Reference encode and decode".  The multiply is a fused multiply-add with
// +0 so that -0.0 becomes +0 (the sign bit is set only for x < 0), while a
// nonzero negative x keeps its sign even when it rounds to zero.  Saturation
// covers |x| 2^-e in (max, 2^(emax+1)), where the nearest grid point is the
// format's largest.

// 64 bytes of bf16 (one block) in two 256-bit loads; p is 32-byte aligned.
__device__ __forceinline__ void load_block_bf16(const __nv_bfloat16* p, uint32_t (&w)[16]) {
    asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
        : "l"(p));
    asm("ld.global.nc.L1::no_allocate.L2::evict_first.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]), "=r"(w[15])
        : "l"(p + 16));
}

// four binary32 -> four E4M3FN codes, element 0 in byte 0
__device__ __forceinline__ uint32_t cvt_e4m3x4(float a0, float a1, float a2, float a3) {
    uint32_t r;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(r)
        : "f"(a0), "f"(a1), "f"(a2), "f"(a3));
    return r;
}

// eight binary32 -> eight E2M1 codes, element 0 in the low nibble of byte 0
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&a)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(r)
        : "f"(a[0]), "f"(a[1]), "f"(a[2]), "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7]));
    return r;
}

// The larger magnitude in each bf16 half of a and b, one instruction: with
// the sign bits cleared afterwards, the result is the larger |x| of the two
// when both are numbers (the bit patterns of non-negative bf16 values order
// as the values do), the infinity when one is infinite, and the canonical NaN
// 0x7FFF when either is a NaN -- so a block's maximum over these is below
// 0x7F80 exactly when the block holds no NaN or infinity, and then equals the
// largest magnitude's bits.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// The scale of a bf16 block from m, the bf16 bits of its largest magnitude
// (sign cleared), and below 0x7F80 (no NaN or infinity, which poison the
// block: scale byte 0xFF, codes 0).  Returns the scale byte e + 127 and sets
// c = 2^-e (1 - 2^-12), the multiplier that pre-scales the block's elements.
template <int FMT>
__device__ __forceinline__ uint32_t bf16_block_scale(uint32_t m, float& c) {
    constexpr int kEmax = FMT == FMT_E2M1 ? 2 : 8;
    // floor(log2 amax) from the bits: normal 2^(field-127), subnormal m * 2^-133
    const int fe = (int)(m >> 7);
    const int E = fe ? fe - 127 : (31 - __clz((int)m)) - 133;
    int e = E - kEmax;
    e = e < -127 ? -127 : (e > 127 ? 127 : e);
    e = m ? e : 0;  // all-zero block: scale byte 127, codes +0
    // 2^-e * (1 - 2^-12) = 2^(-e-1) * (2 - 2^-11)
    c = __uint_as_float(((uint32_t)(126 - e) << 23) | 0x7FF000u);
    return (uint32_t)(e + 127);
}

// Quantize one block of 32 bf16 (16 words, low half = lower element).
// Returns the scale byte; fills 32 bytes (E4M3FN) or 16 bytes (E2M1) of codes.
template <int FMT>
__device__ __forceinline__ uint32_t quantize_block_bf16(const uint32_t (&w)[16], uint32_t (&out)[FMT == FMT_E2M1 ? 4 : 8]) {
    uint32_t m2 = w[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) m2 = bf16x2_absmax(m2, w[i]);
    m2 &= 0x7FFF7FFFu;
    const uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);  // bf16 bits of the block's amax
    if (m >= 0x7F80u) {  // NaN or infinity in the block: poison it
#pragma unroll
        for (int i = 0; i < (FMT == FMT_E2M1 ? 4 : 8); ++i) out[i] = 0;
        return 0xFFu;
    }
    float c;
    const uint32_t sbyte = bf16_block_scale<FMT>(m, c);
    float y[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        y[2 * i] = __fmaf_rn(__uint_as_float(w[i] << 16), c, 0.0f);
        y[2 * i + 1] = __fmaf_rn(__uint_as_float(w[i] & 0xFFFF0000u), c, 0.0f);
    }
    if (FMT == FMT_E2M1) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float a[8] = {y[8 * k], y[8 * k + 1], y[8 * k + 2], y[8 * k + 3],
                                y[8 * k + 4], y[8 * k + 5], y[8 * k + 6], y[8 * k + 7]};
            out[k] = cvt_e2m1x8(a);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) out[k] = cvt_e4m3x4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
    }
    return sbyte;
}

// Quantize the blocks of two neighbouring columns at once: w[i] holds row i
// of column 0 in its low half and of column 1 in its high half (one 32-bit
// load of a bf16 row).  The same scale and rounding as quantize_block_bf16.
// Returns the two scale bytes (column 1 in bits 8..15); fills each column's
// codes.
template <int FMT>
__device__ __forceinline__ uint32_t quantize_column_pair_bf16(const uint32_t (&w)[32],
                                                              uint32_t (&out0)[FMT == FMT_E2M1 ? 4 : 8],
                                                              uint32_t (&out1)[FMT == FMT_E2M1 ? 4 : 8]) {
    constexpr int kOut = FMT == FMT_E2M1 ? 4 : 8;
    uint32_t m2 = w[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) m2 = bf16x2_absmax(m2, w[i]);
    m2 &= 0x7FFF7FFFu;
    uint32_t sbytes = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t(&out)[kOut] = h ? out1 : out0;
        const uint32_t m = h ? m2 >> 16 : m2 & 0xFFFFu;
        uint32_t sbyte = 0xFFu;
        if (m >= 0x7F80u) {  // NaN or infinity in the block: poison it
#pragma unroll
            for (int i = 0; i < kOut; ++i) out[i] = 0;
        } else {
            float c;
            sbyte = bf16_block_scale<FMT>(m, c);
            float y[32];
#pragma unroll
            for (int i = 0; i < 32; ++i)
                y[i] = __fmaf_rn(__uint_as_float(h ? w[i] & 0xFFFF0000u : w[i] << 16), c, 0.0f);
            if (FMT == FMT_E2M1) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a[8] = {y[8 * k], y[8 * k + 1], y[8 * k + 2], y[8 * k + 3],
                                        y[8 * k + 4], y[8 * k + 5], y[8 * k + 6], y[8 * k + 7]};
                    out[k] = cvt_e2m1x8(a);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) out[k] = cvt_e4m3x4(y[4 * k], y[4 * k + 1], y[4 * k + 2], y[4 * k + 3]);
            }
        }
        sbytes |= sbyte << (8 * h);
    }
    return sbytes;
}

// Quantize one block of 32 elements given as binary32 bit patterns (bf16 inputs
// shifted up by 16; `bf16` selects the bf16 routine).  Returns the scale byte.
template <int FMT>
__device__ __forceinline__ uint32_t quantize_column_block(const uint32_t (&u)[32], bool bf16,
                                                          uint32_t (&out)[FMT == FMT_E2M1 ? 4 : 8]) {
    if (bf16) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = (u[2 * i] >> 16) | (u[2 * i + 1] & 0xFFFF0000u);
        return quantize_block_bf16<FMT>(w, out);
    }
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = max(m, u[i] & 0x7FFFFFFFu);
    uint32_t sbyte = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t mn = 0xFFFFFFFFu;
        uint32_t v[8], c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[i] = u[8 * q + i];
            mn = min(mn, v[i] & 0x7FFFFFFFu);
        }
        sbyte = quantize8<FMT>(v, m, mn, c);
        if (FMT == FMT_E2M1) {
            uint32_t wd = c[7];
#pragma unroll
            for (int i = 6; i >= 0; --i) wd = wd * 16u + c[i];
            out[q] = wd;
        } else {
            out[2 * q] = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
            out[2 * q + 1] = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
        }
    }
    return sbyte;
}

}  // namespace mx
