// mx_quant.cu -- MX quantize / dequantize / scale relayout kernels (sm_103a).
//
// quantize_block and dequantize_block of "A Dialect Is a Set of Co-Designed
// Decisions: Designing for MX Quantization in MLIR" ("The four ops"), with the
// element and scale encodings of "Bit Layout" ("The E2M1 element", "The E8M0
// shared scale", "Block structure and packing", "Reference encode and
// decode").
//
// Both kernels stream HBM.  A tensor of R x C (C % 32 == 0) is, in memory, a
// run of R*C/32 blocks of 32 contiguous elements, so the kernels index blocks
// directly: four threads own one block (8 elements each, one or two 16-byte
// loads), a warp owns 8 consecutive blocks (1 KB of f32 / 512 B of bf16, fully
// coalesced), and the block maximum is two xor-shuffles.  Rounding is integer
// and compare logic on the binary32 bits -- no math library calls -- and the
// file is built without flush-to-zero so subnormal inputs and outputs are exact.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // independent items per thread in flight (memory-level parallelism)
constexpr int kMinBlocks = 4; // 4 x 256 threads per SM: at most 64 registers per thread

// ------------------------------------------------------------------ loads

template <typename InT>
struct Load8;

template <>
struct Load8<float> {
    // 8 consecutive f32 -> their bit patterns.
    static __device__ __forceinline__ void run(const float* p, uint32_t (&u)[8]) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
        u[0] = __float_as_uint(a.x); u[1] = __float_as_uint(a.y);
        u[2] = __float_as_uint(a.z); u[3] = __float_as_uint(a.w);
        u[4] = __float_as_uint(b.x); u[5] = __float_as_uint(b.y);
        u[6] = __float_as_uint(b.z); u[7] = __float_as_uint(b.w);
    }
};

template <>
struct Load8<__nv_bfloat16> {
    // 8 consecutive bf16 -> the bit patterns of their (exact) f32 values.
    static __device__ __forceinline__ void run(const __nv_bfloat16* p, uint32_t (&u)[8]) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            u[2 * i] = w[i] << 16;
            u[2 * i + 1] = w[i] & 0xFFFF0000u;
        }
    }
};

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

// Padding of the tensor-core layout: rows up to a multiple of 128 and blocks
// per row up to a multiple of 4 are written as 0 (scale 2^-127, finite, so
// zero-filled operand padding contributes exactly 0).  Grid-strided.
__device__ __forceinline__ void write_mma_padding(uint8_t* __restrict__ scales, int64_t rows, int64_t nb) {
    const int64_t nb4 = round_up(nb, 4);
    const int64_t r128 = round_up(rows, 128);
    const int64_t pad_rows = (r128 - rows) * nb4;
    const int64_t pad_cols = rows * (nb4 - nb);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < pad_rows + pad_cols; p += stride) {
        int64_t r, j;
        if (p < pad_rows) {
            r = rows + p / nb4;
            j = p - (r - rows) * nb4;
        } else {
            const int64_t q = p - pad_rows;
            const int64_t w = nb4 - nb;
            r = q / w;
            j = nb + (q - r * w);
        }
        scales[mma_scale_offset(r, j, nb4)] = 0;
    }
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

// bf16 -> E4M3FN, two elements per 32-bit word (the low half is the lower
// element).  For a block whose exponent e >= -120 and whose elements all lie
// at or above the E4M3 normal range (|x| >= 2^(e-6)), each half h of a word
// gives its code as ((h - (e << 7)) + 7 - (120 << 7)) >> 4: subtract e from
// the bf16 exponent field, round the 4 dropped mantissa bits half-down,
// re-bias 127 -> 7.  Both halves are formed by one 32-bit add: the low half's
// carry into the high half is 1 exactly when the constant K is negative, so
// it is pre-subtracted from the high half of the constant.
__device__ __forceinline__ uint32_t bf16_pair_e4m3(uint32_t w, uint32_t k2) {
    const uint32_t t = (w & 0x7FFF7FFFu) + k2;                      // r_lo | r_hi << 16
    uint32_t c = __vminu2((t >> 4) & 0x00FF00FFu, 0x007E007Eu);      // saturate at 448
    return c | ((w >> 8) & 0x00800080u);                            // sign bits 15, 31 -> 7, 23
}

template <int LAYOUT, int kU, int kMB, int kPipe>
__global__ void __launch_bounds__(kThreads, kMB)
    quantize_bf16_e4m3_kernel(const __nv_bfloat16* __restrict__ x, int64_t nblocks, int64_t nb, int64_t rows,
                              uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int part = lane & 3;
    const int64_t nthreads = nblocks * 4;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t nb4 = round_up(nb, 4);
    uint4 v[kU], nxt[kPipe ? kU : 1];
    int64_t t0 = (int64_t)blockIdx.x * kThreads + threadIdx.x;
#pragma unroll
    for (int q = 0; q < kU; ++q) {
        const int64_t t = t0 + q * stride;
        v[q] = t < nthreads ? __ldcs(reinterpret_cast<const uint4*>(x) + t) : make_uint4(0, 0, 0, 0);
    }
    for (; t0 - lane < nthreads; t0 += stride * kU) {
        if (kPipe) {
            // issue the next round's loads before working on this round
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int64_t t = t0 + (kU + q) * stride;
                nxt[q % (kPipe ? kU : 1)] = t < nthreads ? __ldcs(reinterpret_cast<const uint4*>(x) + t) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t t = t0 + q * stride;
            if (t - lane >= nthreads) break;  // warp-uniform
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
            // |bits| max and min over the thread's 8 elements, 16 bits per lane
            uint32_t mx2 = __vmaxu2(__vmaxu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                    __vmaxu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
            uint32_t mn2 = __vminu2(__vminu2(w[0] & 0x7FFF7FFFu, w[1] & 0x7FFF7FFFu),
                                    __vminu2(w[2] & 0x7FFF7FFFu, w[3] & 0x7FFF7FFFu));
            uint32_t m = max(mx2 & 0xFFFFu, mx2 >> 16);
            const uint32_t mn16 = min(mn2 & 0xFFFFu, mn2 >> 16);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            const uint32_t amax_bits = m << 16;  // binary32 pattern of the bf16 amax
            uint32_t sbyte;
            uint2 out;
            // fast path conditions (a finite, nonzero block is required)
            const int fe = (int)(amax_bits >> 23);
            int e = (fe ? fe - 127 : (31 - __clz((int)amax_bits)) - 149) - 8;
            e = e < -127 ? -127 : (e > 127 ? 127 : e);
            const bool fast = amax_bits - 1u < 0x7F7FFFFFu  // nonzero and finite
                              && e >= -120 && mn16 >= (uint32_t)(e + 121) << 7;
            if (fast) {
                const int K = 7 - 0x3C00 - e * 128;
                const uint32_t k16 = (uint32_t)K & 0xFFFFu;
                const uint32_t k2 = k16 | (((k16 - (K < 0 ? 1u : 0u)) & 0xFFFFu) << 16);
                const uint32_t c0 = bf16_pair_e4m3(w[0], k2), c1 = bf16_pair_e4m3(w[1], k2);
                const uint32_t c2 = bf16_pair_e4m3(w[2], k2), c3 = bf16_pair_e4m3(w[3], k2);
                out.x = __byte_perm(c0, c1, 0x6420);
                out.y = __byte_perm(c2, c3, 0x6420);
                sbyte = (uint32_t)(e + 127);
            } else {
                uint32_t u[8], c[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    u[2 * i] = w[i] << 16;
                    u[2 * i + 1] = w[i] & 0xFFFF0000u;
                }
                sbyte = quantize8<FMT_E4M3>(u, amax_bits, mn16 << 16, c);
                out.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
                out.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
            }
            const bool valid = t < nthreads;
            const int64_t b = t >> 2;
            if (valid) __stcs(reinterpret_cast<uint2*>(codes) + t, out);
            const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 4);
            const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 8);
            const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 12);
            const bool words = (nb & 3) == 0;
            if (valid && (words ? (lane & 15) == 0 : part == 0)) {
                int64_t off;
                if (LAYOUT == LAYOUT_ROWMAJOR) {
                    off = b;
                } else {
                    const int64_t r = b / nb, j = b - r * nb;
                    off = mma_scale_offset(r, j, nb4);
                }
                if (words)
                    *reinterpret_cast<uint32_t*>(scales + off) = sbyte | (s1 << 8) | (s2 << 16) | (s3 << 24);
                else
                    scales[off] = (uint8_t)sbyte;
            }
        }
        if (kPipe) {
#pragma unroll
            for (int q = 0; q < kU; ++q) v[q] = nxt[q % (kPipe ? kU : 1)];
        } else {
#pragma unroll
            for (int q = 0; q < kU; ++q) {
                const int64_t t = t0 + (kU + q) * stride;
                v[q] = t < nthreads ? __ldcs(reinterpret_cast<const uint4*>(x) + t) : make_uint4(0, 0, 0, 0);
            }
        }
    }
    if (LAYOUT == LAYOUT_MMA) write_mma_padding(scales, rows, nb);
}

template <typename InT, int FMT, int LAYOUT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) quantize_kernel(const InT* __restrict__ x, int64_t nblocks, int64_t nb,
                                                            int64_t rows, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales) {
    // 64 bytes of input in flight per thread: 4 items of bf16, 2 of f32 (2 when
    // the tensor-core scale layout's index arithmetic needs the registers)
    constexpr int kU = (sizeof(InT) == 2 && LAYOUT == LAYOUT_ROWMAJOR) ? kUnroll : kUnroll / 2;
    const int lane = threadIdx.x & 31;
    const int part = lane & 3;  // which 8 of the block's 32 elements
    const int64_t nthreads = nblocks * 4;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t nb4 = round_up(nb, 4);

    for (int64_t t0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; t0 - lane < nthreads;
         t0 += stride * kU) {
        uint32_t u[kU][8];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t t = t0 + q * stride;
            if (t < nthreads) {
                Load8<InT>::run(x + t * 8, u[q]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) u[q][i] = 0;
            }
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t t = t0 + q * stride;
            if (t - lane >= nthreads) break;  // warp-uniform: whole warp past the end
            uint32_t m = 0, mn = 0xFFFFFFFFu;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t a = u[q][i] & 0x7FFFFFFFu;
                m = max(m, a);
                mn = min(mn, a);
            }
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            uint32_t c[8];
            const uint32_t sbyte = quantize8<FMT>(u[q], m, mn, c);
            const bool valid = t < nthreads;
            const int64_t b = t >> 2;  // block index
            if (valid) {
                if (FMT == FMT_E2M1) {
                    uint32_t w = c[7];
#pragma unroll
                    for (int i = 6; i >= 0; --i) w = w * 16u + c[i];  // element 0 in the low nibble
                    __stcs(reinterpret_cast<uint32_t*>(codes) + t, w);
                } else {
                    uint2 w;
                    w.x = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
                    w.y = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
                    __stcs(reinterpret_cast<uint2*>(codes) + t, w);
                }
            }
            // Scales.  The warp's first block index is a multiple of 8.  When
            // nb % 4 == 0 every aligned group of 4 blocks lies in one row and
            // is wholly valid or wholly past the end, so lanes 0 and 16 store
            // one 32-bit word each; otherwise each block's lane 0 stores a byte.
            const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 4);
            const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 8);
            const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sbyte, 12);
            const bool words = (nb & 3) == 0;
            if (valid && (words ? (lane & 15) == 0 : part == 0)) {
                int64_t off;
                if (LAYOUT == LAYOUT_ROWMAJOR) {
                    off = b;
                } else {
                    const int64_t r = b / nb, j = b - r * nb;
                    off = mma_scale_offset(r, j, nb4);
                }
                if (words)
                    *reinterpret_cast<uint32_t*>(scales + off) = sbyte | (s1 << 8) | (s2 << 16) | (s3 << 24);
                else
                    scales[off] = (uint8_t)sbyte;
            }
        }
    }

    if (LAYOUT == LAYOUT_MMA) write_mma_padding(scales, rows, nb);
}

// --------------------------------------------------------------- dequantize

// Decoding assembles binary32 bits directly.
//  E4M3FN normal (exponent field E >= 1): 2^(E-7) (1 + M/8) has the bits
//    (E + 120) << 23 | M << 20 = (code7 << 20) + (120 << 23).
//  E4M3FN subnormal (E = 0): M * 2^-9, exact in binary32.  Code 0x7F is NaN.
//  E2M1 (E >= 1): 2^(E-1) (1 + M/2) has the bits (code3 << 22) + (126 << 23);
//    for E = 0 the same assembly with exponent 127 gives 1 + M/2, and 1.0 is
//    subtracted afterwards (0 and 0.5).
__device__ __forceinline__ float e4m3_decode_slow(uint32_t c) {
    const uint32_t c7 = c & 0x7Fu;
    float m;
    if (c7 == 0x7Fu) m = __uint_as_float(0x7FC00000u);
    else if (c7 < 8u) m = (float)c7 * 0.001953125f;
    else m = __uint_as_float((c7 << 20) + 0x3C000000u);
    return (c & 0x80u) ? -m : m;
}

// Decode four codes (one E4M3FN word, or the low 16 bits of an E2M1 word)
// and scale them by `scale` (2^(s-127), or NaN for the poison scale).
template <int FMT>
__device__ __forceinline__ float4 decode4(uint32_t w, float scale) {
    float v[4];
    if (FMT == FMT_E2M1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t c = (w >> (4 * i)) & 0xFu;
            const uint32_t m22 = (c & 7u) << 22;
            const bool sub = m22 < (2u << 22);
            const uint32_t mag = m22 + (sub ? 0x3F800000u : 0x3F000000u);
            // exact: the true magnitude is representable and the fma rounds
            // once; the sign bit goes in afterwards so code 0x8 gives -0.0
            const float m = __fmaf_rn(__uint_as_float(mag), scale, sub ? -scale : 0.0f);
            v[i] = __uint_as_float(__float_as_uint(m) | ((c & 8u) << 28));
        }
    } else {
        // fast path unless some code is subnormal (exponent field 0) or NaN
        if ((__vcmpeq4(w & 0x78787878u, 0u) | __vcmpeq4(w & 0x7F7F7F7Fu, 0x7F7F7F7Fu)) == 0u) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t c = (w >> (8 * i)) & 0xFFu;
                const uint32_t bits = ((c & 0x7Fu) << 20) + 0x3C000000u + ((c & 0x80u) << 24);
                v[i] = __fmul_rn(__uint_as_float(bits), scale);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) v[i] = __fmul_rn(e4m3_decode_slow((w >> (8 * i)) & 0xFFu), scale);
        }
    }
    return make_float4(v[0], v[1], v[2], v[3]);
}

__device__ __forceinline__ float scale_value(uint32_t s) {
    // 2^(s-127) as binary32 (s = 0 is the subnormal 2^-127); the NaN scale 0xFF
    // becomes a NaN multiplier, which poisons the whole block.
    return s == 0xFFu ? __uint_as_float(0x7FC00000u) : (s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u));
}

// A warp owns windows of 8 consecutive blocks (256 elements).  Lane t decodes
// elements [4t, 4t+4) and [128+4t, 128+4t+4) of the window, so each of the
// warp's two 16-byte store instructions writes 512 contiguous bytes (whole
// sectors) and each code load reads 128 (E4M3) or 64 (E2M1) contiguous bytes.
template <int FMT, int LAYOUT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                                          const uint8_t* __restrict__ scales,
                                                                          int64_t nblocks, int64_t nb,
                                                                          float* __restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int64_t nwin = (nblocks + 7) / 8;
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t nb4 = round_up(nb, 4);
    for (int64_t w0 = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); w0 < nwin; w0 += warps * kUnroll) {
        uint32_t cw[kUnroll][2];
        uint32_t sc[kUnroll][2];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int64_t win = w0 + q * warps;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t b = win * 8 + 4 * h + (lane >> 3);  // block of this half
                cw[q][h] = 0;
                sc[q][h] = 0;
                if (win < nwin && b < nblocks) {
                    int64_t soff;
                    if (LAYOUT == LAYOUT_ROWMAJOR) {
                        soff = b;
                    } else {
                        const int64_t r = b / nb, j = b - r * nb;
                        soff = mma_scale_offset(r, j, nb4);
                    }
                    sc[q][h] = __ldg(scales + soff);
                    const int64_t e = win * 256 + 128 * h + 4 * lane;  // first element
                    if (FMT == FMT_E2M1)
                        cw[q][h] = __ldcs(reinterpret_cast<const uint16_t*>(codes) + e / 4);
                    else
                        cw[q][h] = __ldcs(reinterpret_cast<const uint32_t*>(codes) + e / 4);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int64_t win = w0 + q * warps;
            if (win >= nwin) break;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t b = win * 8 + 4 * h + (lane >> 3);
                if (b < nblocks) {
                    const int64_t e = win * 256 + 128 * h + 4 * lane;
                    __stcs(reinterpret_cast<float4*>(y + e), decode4<FMT>(cw[q][h], scale_value(sc[q][h])));
                }
            }
        }
    }
}

// ------------------------------------------------------------------ relayout

__global__ void relayout_kernel(const uint8_t* __restrict__ src, int src_layout, int64_t rows, int64_t nb,
                                uint8_t* __restrict__ dst, int dst_layout) {
    const int64_t nb4 = round_up(nb, 4);
    const int64_t r128 = round_up(rows, 128);
    const int64_t total = dst_layout == LAYOUT_MMA ? r128 * nb4 : rows * nb;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        int64_t r, j;
        if (dst_layout == LAYOUT_MMA) {
            r = i / nb4;
            j = i - r * nb4;
        } else {
            r = i / nb;
            j = i - r * nb;
        }
        const bool real = r < rows && j < nb;
        uint8_t v = 0;
        if (real) v = src[src_layout == LAYOUT_MMA ? mma_scale_offset(r, j, nb4) : r * nb + j];
        const int64_t o = dst_layout == LAYOUT_MMA ? mma_scale_offset(r, j, nb4) : r * nb + j;
        dst[o] = v;
    }
}

int64_t grid_for(int64_t work_threads, int per_sm) {
    int64_t g = (work_threads + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)sm_count() * per_sm;
    if (g > cap) g = cap;
    return g < 1 ? 1 : g;
}

template <typename InT, int FMT>
cudaError_t quant_dispatch_layout(const InT* x, int64_t nblocks, int64_t nb, int64_t rows, uint8_t* codes,
                                  uint8_t* scales, int layout, cudaStream_t st) {
    const int64_t work = nblocks * 4;
    int64_t grid = grid_for((work + 1) / 2, kMinBlocks);
    if constexpr (sizeof(InT) == 2 && FMT == FMT_E4M3) {
        if (layout == LAYOUT_MMA) {
            const int64_t pad = (round_up(rows, 128) - rows) * round_up(nb, 4) + rows * (round_up(nb, 4) - nb);
            const int64_t g2 = grid_for(pad, kMinBlocks);
            grid = grid > g2 ? grid : g2;
            quantize_bf16_e4m3_kernel<LAYOUT_MMA, 2, kMinBlocks, 1><<<(unsigned)grid, kThreads, 0, st>>>(x, nblocks, nb, rows, codes, scales);
        } else {
            // two items per thread per round, the next round's loads issued before
            // this round's work (measured fastest of the unroll / occupancy choices)
            const unsigned g = (unsigned)grid_for((work + 1) / 2, kMinBlocks);
            quantize_bf16_e4m3_kernel<LAYOUT_ROWMAJOR, 2, kMinBlocks, 1><<<g, kThreads, 0, st>>>(x, nblocks, nb, rows,
                                                                                                codes, scales);
        }
        return cudaGetLastError();
    }
    if (layout == LAYOUT_MMA) {
        const int64_t pad = (round_up(rows, 128) - rows) * round_up(nb, 4) + rows * (round_up(nb, 4) - nb);
        const int64_t g2 = grid_for(pad, 8);
        grid = grid > g2 ? grid : g2;
        quantize_kernel<InT, FMT, LAYOUT_MMA><<<(unsigned)grid, kThreads, 0, st>>>(x, nblocks, nb, rows, codes, scales);
    } else {
        quantize_kernel<InT, FMT, LAYOUT_ROWMAJOR><<<(unsigned)grid, kThreads, 0, st>>>(x, nblocks, nb, rows, codes,
                                                                                      scales);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const void* x, int dtype, int64_t rows, int64_t cols, int fmt, void* codes,
                            uint8_t* scales, int layout, cudaStream_t st) {
    const int64_t nb = cols / 32;
    const int64_t nblocks = rows * nb;
    uint8_t* c = static_cast<uint8_t*>(codes);
    if (dtype == DT_F32) {
        const float* p = static_cast<const float*>(x);
        return fmt == FMT_E2M1 ? quant_dispatch_layout<float, FMT_E2M1>(p, nblocks, nb, rows, c, scales, layout, st)
                               : quant_dispatch_layout<float, FMT_E4M3>(p, nblocks, nb, rows, c, scales, layout, st);
    }
    const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(x);
    return fmt == FMT_E2M1
               ? quant_dispatch_layout<__nv_bfloat16, FMT_E2M1>(p, nblocks, nb, rows, c, scales, layout, st)
               : quant_dispatch_layout<__nv_bfloat16, FMT_E4M3>(p, nblocks, nb, rows, c, scales, layout, st);
}

cudaError_t launch_dequantize(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols, int fmt,
                              int layout, float* y, cudaStream_t st) {
    const int64_t nb = cols / 32;
    const int64_t nblocks = rows * nb;
    // one warp per window of 8 blocks, kUnroll windows per warp per round
    const int64_t nwin = (nblocks + 7) / 8;
    const unsigned grid = (unsigned)grid_for((nwin * 32 + kUnroll - 1) / kUnroll, kMinBlocks);
    const uint8_t* c = static_cast<const uint8_t*>(codes);
    if (fmt == FMT_E2M1) {
        if (layout == LAYOUT_MMA)
            dequantize_kernel<FMT_E2M1, LAYOUT_MMA><<<grid, kThreads, 0, st>>>(c, scales, nblocks, nb, y);
        else
            dequantize_kernel<FMT_E2M1, LAYOUT_ROWMAJOR><<<grid, kThreads, 0, st>>>(c, scales, nblocks, nb, y);
    } else {
        if (layout == LAYOUT_MMA)
            dequantize_kernel<FMT_E4M3, LAYOUT_MMA><<<grid, kThreads, 0, st>>>(c, scales, nblocks, nb, y);
        else
            dequantize_kernel<FMT_E4M3, LAYOUT_ROWMAJOR><<<grid, kThreads, 0, st>>>(c, scales, nblocks, nb, y);
    }
    return cudaGetLastError();
}

cudaError_t launch_relayout(const uint8_t* src, int src_layout, int64_t rows, int64_t cols, uint8_t* dst,
                            int dst_layout, cudaStream_t st) {
    const int64_t nb = cols / 32;
    const int64_t total = dst_layout == LAYOUT_MMA ? round_up(rows, 128) * round_up(nb, 4) : rows * nb;
    if (total == 0) return cudaSuccess;
    relayout_kernel<<<(unsigned)grid_for(total, 8), kThreads, 0, st>>>(src, src_layout, rows, nb, dst, dst_layout);
    return cudaGetLastError();
}

}  // namespace mx
