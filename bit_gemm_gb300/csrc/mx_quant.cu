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
// directly.  bf16 input (32-byte aligned): one thread owns one block (two
// 256-bit loads, one 256- or 128-bit store of codes), so the per-block work --
// amax, scale, its store -- is done once, and elements are rounded by the
// hardware E4M3 / E2M1 conversions after an exact pre-scaling that turns
// their ties-to-even into ties-to-lower.  f32 input (and bf16 that is only
// 16-byte aligned): four threads own one block (8 elements each), a warp owns
// 8 consecutive blocks (fully coalesced), the block maximum is two
// xor-shuffles, and rounding is integer and compare logic on the binary32
// bits.  No math library calls; the file is built without flush-to-zero so
// subnormal inputs and outputs are exact.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mx_quant_block.cuh"

namespace mx {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;   // independent items per thread in flight (memory-level parallelism)
constexpr int kMinBlocks = 4; // 4 x 256 threads per SM: at most 64 registers per thread
// elements per lane of the dequantize kernels (measured on GB300, 4096^2
// MXFP8: f32 out 15.0 us with 8, 14.0 with 16, 16.8-18.1 with 32; bf16 out
// 9.6 us with 8, 9.0 with 16, 8.0 with 32)
constexpr int kDeqF32Lane = 16;
constexpr int kDeqBf16Lane = 32;

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

// Grid-strided over blocks, kU blocks per thread in flight.  x and codes are
// 32-byte aligned.  For the tensor-core scale layout the block's (row, block
// column) is carried incrementally across the stride.
template <int FMT, int LAYOUT, int kU>
__global__ void __launch_bounds__(kThreads, kMinBlocks)
    quantize_bf16_block_kernel(const __nv_bfloat16* __restrict__ x, int64_t nblocks, int64_t nb, int64_t rows,
                               uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    pdl_launch_dependents();  // the next kernel may set up while this one runs
    pdl_wait();               // the previous kernel's writes are visible
    constexpr int kCodeWords = FMT == FMT_E2M1 ? 4 : 8;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t nb4 = round_up(nb, 4);
    int64_t b0 = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    // (row, column) of block b0 and of the stride, for the tensor-core layout
    int32_t r = 0, j = 0, sr = 0, sj = 0;  // rows, blocks per row and the stride are below 2^31
    if (LAYOUT == LAYOUT_MMA) {
        r = (int32_t)(b0 / nb);
        j = (int32_t)(b0 - (int64_t)r * nb);
        sr = (int32_t)(stride / nb);
        sj = (int32_t)(stride - (int64_t)sr * nb);
    }
    for (; b0 < nblocks; b0 += stride * kU) {
        uint32_t w[kU][16];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t b = b0 + q * stride;
            if (b < nblocks) load_block_bf16(x + 32 * b, w[q]);
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int64_t b = b0 + q * stride;
            if (b >= nblocks) break;
            uint32_t out[kCodeWords];
            const uint32_t sbyte = quantize_block_bf16<FMT>(w[q], out);
            if (FMT == FMT_E2M1) {
                __stcs(reinterpret_cast<uint4*>(codes) + b, make_uint4(out[0], out[1], out[2], out[3]));
            } else {
                asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(codes + 32 * b),
                             "r"(out[0]), "r"(out[1]), "r"(out[2]), "r"(out[3]), "r"(out[4]), "r"(out[5]),
                             "r"(out[6]), "r"(out[7])
                             : "memory");
            }
            if (LAYOUT == LAYOUT_MMA) {
                scales[mma_scale_offset(r, j, nb4)] = (uint8_t)sbyte;
                r += sr;
                j += sj;
                if (j >= nb) {
                    j -= nb;
                    ++r;
                }
            } else {
                scales[b] = (uint8_t)sbyte;
            }
        }
    }
    if (LAYOUT == LAYOUT_MMA) write_mma_padding(scales, rows, nb);
}

template <typename InT, int FMT, int LAYOUT>
__global__ void __launch_bounds__(kThreads, kMinBlocks) quantize_kernel(const InT* __restrict__ x, int64_t nblocks, int64_t nb,
                                                            int64_t rows, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales) {
    pdl_launch_dependents();  // the next kernel may set up while this one runs
    pdl_wait();               // the previous kernel's writes are visible
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

// Decoding uses the hardware conversions E4M3FN / E2M1 -> f16 (exact: every
// element value, and the E4M3FN NaN code, is representable in f16), then
// f16 -> f32 (exact) and one multiply by the block's scale 2^(s-127), which
// is exact too: the smallest product, 2^-9 * 2^-127, is a binary32
// subnormal, and a product above the binary32 range is infinite, as the
// exact value rounded to binary32 is.  A NaN scale makes every product NaN.

// eight E4M3FN codes (byte i = element i) -> eight f32, times `mult`
__device__ __forceinline__ void decode8_e4m3(uint32_t lo, uint32_t hi, float mult, float (&v)[8]) {
    asm("{\n\t.reg .b16 c0, c1, c2, c3, h0, h1, h2, h3, h4, h5, h6, h7;\n\t"
        ".reg .b32 p0, p1, p2, p3;\n\t.reg .f32 f0, f1, f2, f3, f4, f5, f6, f7;\n\t"
        "mov.b32 {c0, c1}, %8;\n\tmov.b32 {c2, c3}, %9;\n\t"
        "cvt.rn.f16x2.e4m3x2 p0, c0;\n\tcvt.rn.f16x2.e4m3x2 p1, c1;\n\t"
        "cvt.rn.f16x2.e4m3x2 p2, c2;\n\tcvt.rn.f16x2.e4m3x2 p3, c3;\n\t"
        "mov.b32 {h0, h1}, p0;\n\tmov.b32 {h2, h3}, p1;\n\tmov.b32 {h4, h5}, p2;\n\tmov.b32 {h6, h7}, p3;\n\t"
        "cvt.f32.f16 f0, h0;\n\tcvt.f32.f16 f1, h1;\n\tcvt.f32.f16 f2, h2;\n\tcvt.f32.f16 f3, h3;\n\t"
        "cvt.f32.f16 f4, h4;\n\tcvt.f32.f16 f5, h5;\n\tcvt.f32.f16 f6, h6;\n\tcvt.f32.f16 f7, h7;\n\t"
        "mul.rn.f32 %0, f0, %10;\n\tmul.rn.f32 %1, f1, %10;\n\tmul.rn.f32 %2, f2, %10;\n\tmul.rn.f32 %3, f3, %10;\n\t"
        "mul.rn.f32 %4, f4, %10;\n\tmul.rn.f32 %5, f5, %10;\n\tmul.rn.f32 %6, f6, %10;\n\tmul.rn.f32 %7, f7, %10;\n\t}"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
        : "r"(lo), "r"(hi), "f"(mult));
}

// eight E2M1 codes (element i in nibble i, low nibble first) -> eight f32, times `mult`
__device__ __forceinline__ void decode8_e2m1(uint32_t w, float mult, float (&v)[8]) {
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t.reg .b16 h0, h1, h2, h3, h4, h5, h6, h7;\n\t"
        ".reg .b32 p0, p1, p2, p3;\n\t.reg .f32 f0, f1, f2, f3, f4, f5, f6, f7;\n\t"
        "mov.b32 {c0, c1, c2, c3}, %8;\n\t"
        "cvt.rn.f16x2.e2m1x2 p0, c0;\n\tcvt.rn.f16x2.e2m1x2 p1, c1;\n\t"
        "cvt.rn.f16x2.e2m1x2 p2, c2;\n\tcvt.rn.f16x2.e2m1x2 p3, c3;\n\t"
        "mov.b32 {h0, h1}, p0;\n\tmov.b32 {h2, h3}, p1;\n\tmov.b32 {h4, h5}, p2;\n\tmov.b32 {h6, h7}, p3;\n\t"
        "cvt.f32.f16 f0, h0;\n\tcvt.f32.f16 f1, h1;\n\tcvt.f32.f16 f2, h2;\n\tcvt.f32.f16 f3, h3;\n\t"
        "cvt.f32.f16 f4, h4;\n\tcvt.f32.f16 f5, h5;\n\tcvt.f32.f16 f6, h6;\n\tcvt.f32.f16 f7, h7;\n\t"
        "mul.rn.f32 %0, f0, %9;\n\tmul.rn.f32 %1, f1, %9;\n\tmul.rn.f32 %2, f2, %9;\n\tmul.rn.f32 %3, f3, %9;\n\t"
        "mul.rn.f32 %4, f4, %9;\n\tmul.rn.f32 %5, f5, %9;\n\tmul.rn.f32 %6, f6, %9;\n\tmul.rn.f32 %7, f7, %9;\n\t}"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]), "=f"(v[7])
        : "r"(w), "f"(mult));
}

__device__ __forceinline__ float scale_value(uint32_t s) {
    // 2^(s-127) as binary32 (s = 0 is the subnormal 2^-127); the NaN scale 0xFF
    // becomes a NaN multiplier, which poisons the whole block.
    return s == 0xFFu ? __uint_as_float(0x7FC00000u) : (s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u));
}

// A warp owns windows of EL consecutive blocks (32 EL elements).  Lane t
// decodes elements [EL t, EL t + EL) of the window (block t / (32 / EL)), so
// one code load per lane reads EL (E4M3) or EL / 2 (E2M1) contiguous bytes,
// and the warp's stores write 128 EL bytes of contiguous f32 (256-bit stores
// per lane when y is 32-byte aligned, else 128-bit ones) or 64 EL bytes of
// bf16.  EL = 16 halves the per-element index and scale work of EL = 8.
template <int FMT, int LAYOUT, bool kV8, bool kBF16 = false, int EL = 8, int kUnroll = kUnroll>
__global__ void __launch_bounds__(kThreads, kMinBlocks) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                                          const uint8_t* __restrict__ scales,
                                                                          int64_t nblocks, int64_t nb,
                                                                          void* __restrict__ yv) {
    static_assert(EL == 8 || EL == 16 || EL == 32, "elements per lane");
    constexpr int kLPB = 32 / EL;  // lanes per block
    constexpr int kCW = FMT == FMT_E2M1 ? EL / 8 : EL / 4;  // 32-bit code words per lane
    pdl_launch_dependents();  // the next kernel may set up while this one runs
    pdl_wait();               // the previous kernel's writes are visible
    float* __restrict__ y = static_cast<float*>(yv);
    const int lane = threadIdx.x & 31;
    const int64_t nwin = (nblocks + EL - 1) / EL;
    const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
    const int64_t nb4 = round_up(nb, 4);
    for (int64_t w0 = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); w0 < nwin; w0 += warps * kUnroll) {
        uint32_t cw[kUnroll][kCW];
        uint32_t sc[kUnroll];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int64_t win = w0 + q * warps;
            const int64_t b = win * EL + lane / kLPB;  // this lane's block
#pragma unroll
            for (int k = 0; k < kCW; ++k) cw[q][k] = 0;
            sc[q] = 0;
            if (win < nwin && b < nblocks) {
                int64_t soff;
                if (LAYOUT == LAYOUT_ROWMAJOR) {
                    soff = b;
                } else {
                    const int64_t r = b / nb, j = b - r * nb;
                    soff = mma_scale_offset(r, j, nb4);
                }
                sc[q] = __ldg(scales + soff);
                const int64_t e = win * 32 * EL + EL * lane;  // first element
                if (kCW == 1) {
                    cw[q][0] = __ldcs(reinterpret_cast<const uint32_t*>(codes) + e / 8);
                } else if (kCW == 2) {
                    const uint2 c2 = __ldcs(reinterpret_cast<const uint2*>(codes + (FMT == FMT_E2M1 ? e / 2 : e)));
                    cw[q][0] = c2.x;
                    cw[q][1] = c2.y;
                } else {
#pragma unroll
                    for (int k = 0; k < kCW / 4; ++k) {
                        const uint4 c4 = __ldcs(reinterpret_cast<const uint4*>(codes + (FMT == FMT_E2M1 ? e / 2 : e)) + k);
                        cw[q][4 * k] = c4.x;
                        cw[q][4 * k + 1] = c4.y;
                        cw[q][4 * k + 2] = c4.z;
                        cw[q][4 * k + 3] = c4.w;
                    }
                }
            }
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int64_t win = w0 + q * warps;
            if (win >= nwin) break;
            const int64_t b = win * EL + lane / kLPB;
            if (b < nblocks) {
                float v[EL];
                const float mult = scale_value(sc[q]);
#pragma unroll
                for (int h = 0; h < EL / 8; ++h) {
                    float* vh = v + 8 * h;
                    float (&v8)[8] = *reinterpret_cast<float (*)[8]>(vh);
                    if (FMT == FMT_E2M1) decode8_e2m1(cw[q][h], mult, v8);
                    else decode8_e4m3(cw[q][2 * h], cw[q][2 * h + 1], mult, v8);
                }
                const int64_t e = win * 32 * EL + EL * lane;
                if (kBF16) {
                    // bfloat16 output: the exact value rounded to nearest, ties to
                    // even (cvt.rn.bf16x2.f32); 2 EL bytes per lane
                    uint32_t o[EL / 2];
#pragma unroll
                    for (int i = 0; i < EL / 2; ++i) {
                        const __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                        o[i] = *reinterpret_cast<const uint32_t*>(&pr);
                    }
                    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(yv) + e;
                    if (EL >= 16 && kV8) {
#pragma unroll
                        for (int i = 0; i < EL / 16; ++i)
                            asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 16 * i),
                                         "r"(o[8 * i]), "r"(o[8 * i + 1]), "r"(o[8 * i + 2]), "r"(o[8 * i + 3]),
                                         "r"(o[8 * i + (EL > 8 ? 4 : 0)]), "r"(o[8 * i + (EL > 8 ? 5 : 0)]),
                                         "r"(o[8 * i + (EL > 8 ? 6 : 0)]), "r"(o[8 * i + (EL > 8 ? 7 : 0)])
                                         : "memory");
                    } else {
#pragma unroll
                        for (int i = 0; i < EL / 8; ++i)
                            __stcs(reinterpret_cast<uint4*>(dst) + i, make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]));
                    }
                    continue;
                }
                float* dst = y + e;
#pragma unroll
                for (int h = 0; h < EL / 8; ++h) {
                    const float* vh = v + 8 * h;
                    if (kV8) {
                        asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 8 * h),
                                     "f"(vh[0]), "f"(vh[1]), "f"(vh[2]), "f"(vh[3]), "f"(vh[4]), "f"(vh[5]), "f"(vh[6]),
                                     "f"(vh[7])
                                     : "memory");
                    } else {
                        __stcs(reinterpret_cast<float4*>(dst + 8 * h), make_float4(vh[0], vh[1], vh[2], vh[3]));
                        __stcs(reinterpret_cast<float4*>(dst + 8 * h) + 1, make_float4(vh[4], vh[5], vh[6], vh[7]));
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------- fold_scale
//
// Multiply an MX tensor by 2^j: every real scale byte b != 0xFF becomes
// clamp(b + j, 0, 254); 0xFF (NaN) and the tensor-core layout's padding stay.
__global__ void fold_scale_kernel(uint8_t* __restrict__ scales, int64_t rows, int64_t nb, int layout, int j) {
    const int64_t total = rows * nb;
    const int64_t nb4 = round_up(nb, 4);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
        int64_t off = i;
        if (layout == LAYOUT_MMA) {
            const int64_t r = i / nb;
            off = mma_scale_offset(r, i - r * nb, nb4);
        }
        const int b = scales[off];
        if (b == 0xFF) continue;
        int v = b + j;
        v = v < 0 ? 0 : (v > 254 ? 254 : v);
        scales[off] = (uint8_t)v;
    }
}

// ---------------------------------------------------------- block axis 0
//
// Quantize x [rows][cols] in blocks of 32 consecutive ROWS of one column (the
// reduction axis of a K x N right-hand operand) and write codes and scales in
// the layout of the transposed tensor: codes [cols][rows] (packed as usual),
// scales [cols][rows/32] (either layout, with cols as its rows).  A thread
// owns kC adjacent columns and up to 4 consecutive blocks of them (128 rows);
// a warp's loads of one input row are 32 * kC contiguous elements, and each
// column's codes for its 4 blocks leave as contiguous 16- or 32-byte stores.
// Rounding is the same as along the last axis: bf16 blocks go through
// quantize_block_bf16, f32 blocks through quantize8.
template <typename InT, int kC>
struct Axis0Load;
template <>
struct Axis0Load<__nv_bfloat16, 2> {  // two columns per 32-bit load
    static __device__ __forceinline__ void row(const __nv_bfloat16* p, uint32_t (&u)[2]) {
        const uint32_t w = __ldcs(reinterpret_cast<const unsigned int*>(p));
        u[0] = w << 16;
        u[1] = w & 0xFFFF0000u;
    }
};
template <>
struct Axis0Load<__nv_bfloat16, 1> {
    static __device__ __forceinline__ void row(const __nv_bfloat16* p, uint32_t (&u)[1]) {
        u[0] = (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(p)) << 16;
    }
};
template <>
struct Axis0Load<float, 1> {
    static __device__ __forceinline__ void row(const float* p, uint32_t (&u)[1]) {
        u[0] = __float_as_uint(__ldcs(p));
    }
};

template <typename InT, int kC, int FMT, int LAYOUT>
__global__ void __launch_bounds__(kThreads) quantize_axis0_kernel(const InT* __restrict__ x, int64_t rows,
                                                                  int64_t cols, uint8_t* __restrict__ codes,
                                                                  uint8_t* __restrict__ scales) {
    constexpr int kCodeWords = FMT == FMT_E2M1 ? 4 : 8;
    const int64_t nb = rows / 32;
    const int64_t nb4 = round_up(nb, 4);
    const int64_t ncg = (cols + kC - 1) / kC;  // column groups
    const int64_t nrg = (nb + 3) / 4;           // groups of 4 blocks
    const int64_t tasks = ncg * nrg;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t code_row = FMT == FMT_E2M1 ? rows / 2 : rows;  // bytes of one output row
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < tasks; t += stride) {
        const int64_t cg = t % ncg, rg = t / ncg;
        const int64_t c0 = cg * kC;
        const int64_t b0 = rg * 4;
        const int nblk = (int)min((int64_t)4, nb - b0);
        for (int bi = 0; bi < nblk; ++bi) {
            const int64_t r0 = (b0 + bi) * 32;
            uint32_t u[kC][32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                uint32_t v[kC];
                Axis0Load<InT, kC>::row(x + (r0 + i) * cols + c0, v);
#pragma unroll
                for (int c = 0; c < kC; ++c) u[c][i] = v[c];
            }
#pragma unroll
            for (int c = 0; c < kC; ++c) {
                const int64_t col = c0 + c;
                if (col >= cols) break;
                uint32_t out[kCodeWords];
                const uint32_t sbyte = quantize_column_block<FMT>(u[c], sizeof(InT) == 2, out);
                uint8_t* dst = codes + col * code_row + (FMT == FMT_E2M1 ? r0 / 2 : r0);
                // write-back stores: the rest of each line comes from the next blocks
                reinterpret_cast<uint4*>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
                if (FMT == FMT_E4M3) reinterpret_cast<uint4*>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
                const int64_t off = LAYOUT == LAYOUT_MMA ? mma_scale_offset(col, b0 + bi, nb4) : col * nb + b0 + bi;
                scales[off] = (uint8_t)sbyte;
            }
        }
    }
    if (LAYOUT == LAYOUT_MMA) write_mma_padding(scales, cols, nb);
}

// ------------------------------------------------------------------ relayout

// Row-major scales [rows][nb] (nb % 4 == 0) -> the tensor-core layout, as
// 32-bit words: row r's word g (blocks 4g .. 4g+3) goes to word
// 4 (r % 32) + (r / 32) % 4 of tile (r / 128, g).  Both operands of a product
// in one launch: a CTA takes 128 rows and kRmGroups words of them of one
// operand through shared memory, reading whole rows (16-byte loads when rows
// are 16-byte multiples) and writing whole 512-byte tiles (16-byte stores);
// rows past the end are written as zero padding.
constexpr int kRmGroups = 32;

struct RmOperand {
    const uint32_t* src;
    uint32_t* dst;
    int64_t rows;
    int64_t ctas;  // tiles x group chunks
};

__global__ void __launch_bounds__(256) scales_to_mma_kernel(RmOperand a, RmOperand b, int64_t ng, int64_t gchunks) {
    __shared__ uint32_t tile[128][kRmGroups + 1];
    pdl_launch_dependents();
    int64_t cta = blockIdx.x;
    const bool is_a = cta < a.ctas;
    if (!is_a) cta -= a.ctas;
    const uint32_t* __restrict__ src = is_a ? a.src : b.src;
    uint32_t* __restrict__ dst = is_a ? a.dst : b.dst;
    const int64_t rows = is_a ? a.rows : b.rows;
    const int64_t t = cta / gchunks;
    const int64_t r0 = t * 128, g0 = (cta - t * gchunks) * kRmGroups;
    const int gn = (int)(ng - g0 < kRmGroups ? ng - g0 : kRmGroups);
    pdl_wait();
    if ((ng & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        // gn is a multiple of 4 here: whole 16-byte quads of each row
        for (int i = threadIdx.x; i < 128 * (kRmGroups / 4); i += blockDim.x) {
            const int r = i / (kRmGroups / 4), q = i % (kRmGroups / 4);
            uint4 v = make_uint4(0, 0, 0, 0);
            if (4 * q < gn && r0 + r < rows)
                v = *reinterpret_cast<const uint4*>(src + (r0 + r) * ng + g0 + 4 * q);
            tile[r][4 * q] = v.x;
            tile[r][4 * q + 1] = v.y;
            tile[r][4 * q + 2] = v.z;
            tile[r][4 * q + 3] = v.w;
        }
    } else {
        for (int i = threadIdx.x; i < 128 * kRmGroups; i += blockDim.x) {
            const int r = i / kRmGroups, g = i % kRmGroups;
            uint32_t v = 0;
            if (g < gn && r0 + r < rows) v = src[(r0 + r) * ng + g0 + g];
            tile[r][g] = v;
        }
    }
    __syncthreads();
    // output word 4k + j of a tile holds row 32 j + k
    for (int i = threadIdx.x; i < 32 * gn; i += blockDim.x) {
        const int g = i / 32, k = i % 32;
        *reinterpret_cast<uint4*>(dst + (t * ng + g0 + g) * 128 + 4 * k) =
            make_uint4(tile[k][g], tile[32 + k][g], tile[64 + k][g], tile[96 + k][g]);
    }
}

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
    const bool al32 = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(codes)) & 31) == 0;
    if constexpr (sizeof(InT) == 2) {
        if (al32) {
            constexpr int kU = 2;
            int64_t g = grid_for((nblocks + kU - 1) / kU, kMinBlocks);
            if (layout == LAYOUT_MMA) {
                const int64_t pad = (round_up(rows, 128) - rows) * round_up(nb, 4) + rows * (round_up(nb, 4) - nb);
                const int64_t g2 = grid_for(pad, kMinBlocks);
                g = g > g2 ? g : g2;
                (void)launch_pdl(quantize_bf16_block_kernel<FMT, LAYOUT_MMA, kU>, dim3((unsigned)g), dim3(kThreads), 0, st, x, nblocks, nb, rows, codes, scales);
            } else {
                (void)launch_pdl(quantize_bf16_block_kernel<FMT, LAYOUT_ROWMAJOR, kU>, dim3((unsigned)g), dim3(kThreads), 0, st, x, nblocks, nb, rows, codes, scales);
            }
            return cudaGetLastError();
        }
    }
    if (layout == LAYOUT_MMA) {
        const int64_t pad = (round_up(rows, 128) - rows) * round_up(nb, 4) + rows * (round_up(nb, 4) - nb);
        const int64_t g2 = grid_for(pad, 8);
        grid = grid > g2 ? grid : g2;
        (void)launch_pdl(quantize_kernel<InT, FMT, LAYOUT_MMA>, dim3((unsigned)grid), dim3(kThreads), 0, st, x, nblocks, nb, rows, codes, scales);
    } else {
        (void)launch_pdl(quantize_kernel<InT, FMT, LAYOUT_ROWMAJOR>, dim3((unsigned)grid), dim3(kThreads), 0, st, x, nblocks, nb, rows, codes, scales);
    }
    return cudaGetLastError();
}

template <bool kV8>
cudaError_t deq_dispatch(const uint8_t* c, const uint8_t* scales, int64_t nblocks, int64_t nb, int fmt, int layout,
                         float* y, unsigned grid, cudaStream_t st) {
    if (fmt == FMT_E2M1) {
        if (layout == LAYOUT_MMA)
            (void)launch_pdl(dequantize_kernel<FMT_E2M1, LAYOUT_MMA, kV8, false, kDeqF32Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
        else
            (void)launch_pdl(dequantize_kernel<FMT_E2M1, LAYOUT_ROWMAJOR, kV8, false, kDeqF32Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
    } else {
        if (layout == LAYOUT_MMA)
            (void)launch_pdl(dequantize_kernel<FMT_E4M3, LAYOUT_MMA, kV8, false, kDeqF32Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
        else
            (void)launch_pdl(dequantize_kernel<FMT_E4M3, LAYOUT_ROWMAJOR, kV8, false, kDeqF32Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
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
    // one warp per window of kDeqF32Lane blocks, kUnroll windows per warp per round
    const int64_t nwin = (nblocks + kDeqF32Lane - 1) / kDeqF32Lane;
    const unsigned grid = (unsigned)grid_for((nwin * 32 + kUnroll - 1) / kUnroll, kMinBlocks);
    const uint8_t* c = static_cast<const uint8_t*>(codes);
    if ((reinterpret_cast<uintptr_t>(y) & 31) == 0)
        return deq_dispatch<true>(c, scales, nblocks, nb, fmt, layout, y, grid, st);
    return deq_dispatch<false>(c, scales, nblocks, nb, fmt, layout, y, grid, st);
}


template <bool kV8>
void deq_bf16_dispatch(const uint8_t* c, const uint8_t* scales, int64_t nblocks, int64_t nb, int fmt, int layout,
                       void* y, unsigned grid, cudaStream_t st) {
    if (fmt == FMT_E2M1) {
        if (layout == LAYOUT_MMA)
            (void)launch_pdl(dequantize_kernel<FMT_E2M1, LAYOUT_MMA, kV8, true, kDeqBf16Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
        else
            (void)launch_pdl(dequantize_kernel<FMT_E2M1, LAYOUT_ROWMAJOR, kV8, true, kDeqBf16Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
    } else {
        if (layout == LAYOUT_MMA)
            (void)launch_pdl(dequantize_kernel<FMT_E4M3, LAYOUT_MMA, kV8, true, kDeqBf16Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
        else
            (void)launch_pdl(dequantize_kernel<FMT_E4M3, LAYOUT_ROWMAJOR, kV8, true, kDeqBf16Lane>, dim3(grid), dim3(kThreads), 0, st, c, scales, nblocks, nb, y);
    }
}

cudaError_t launch_dequantize_bf16(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols, int fmt,
                                   int layout, void* y, cudaStream_t st) {
    const int64_t nb = cols / 32;
    const int64_t nblocks = rows * nb;
    const int64_t nwin = (nblocks + kDeqBf16Lane - 1) / kDeqBf16Lane;
    const unsigned grid = (unsigned)grid_for((nwin * 32 + kUnroll - 1) / kUnroll, kMinBlocks);
    const uint8_t* c = static_cast<const uint8_t*>(codes);
    if ((reinterpret_cast<uintptr_t>(y) & 31) == 0) deq_bf16_dispatch<true>(c, scales, nblocks, nb, fmt, layout, y, grid, st);
    else deq_bf16_dispatch<false>(c, scales, nblocks, nb, fmt, layout, y, grid, st);
    return cudaGetLastError();
}

cudaError_t launch_fold_scale(uint8_t* scales, int64_t rows, int64_t cols, int layout, int j, cudaStream_t st) {
    const int64_t nb = cols / 32;
    if (rows * nb == 0) return cudaSuccess;
    fold_scale_kernel<<<(unsigned)grid_for(rows * nb, 8), kThreads, 0, st>>>(scales, rows, nb, layout, j);
    return cudaGetLastError();
}

namespace {
template <typename InT, int kC, int FMT>
cudaError_t axis0_layout(const InT* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales, int layout,
                         cudaStream_t st) {
    const int64_t nb = rows / 32;
    const int64_t tasks = ((cols + kC - 1) / kC) * ((nb + 3) / 4);
    int64_t grid = grid_for(tasks, 4);
    if (layout == LAYOUT_MMA) {
        const int64_t pad = (round_up(cols, 128) - cols) * round_up(nb, 4) + cols * (round_up(nb, 4) - nb);
        const int64_t g2 = grid_for(pad, 4);
        grid = grid > g2 ? grid : g2;
        quantize_axis0_kernel<InT, kC, FMT, LAYOUT_MMA><<<(unsigned)grid, kThreads, 0, st>>>(x, rows, cols, codes, scales);
    } else {
        quantize_axis0_kernel<InT, kC, FMT, LAYOUT_ROWMAJOR><<<(unsigned)grid, kThreads, 0, st>>>(x, rows, cols, codes,
                                                                                            scales);
    }
    return cudaGetLastError();
}
template <typename InT, int kC>
cudaError_t axis0_fmt(const InT* x, int64_t rows, int64_t cols, int fmt, uint8_t* codes, uint8_t* scales, int layout,
                      cudaStream_t st) {
    return fmt == FMT_E2M1 ? axis0_layout<InT, kC, FMT_E2M1>(x, rows, cols, codes, scales, layout, st)
                           : axis0_layout<InT, kC, FMT_E4M3>(x, rows, cols, codes, scales, layout, st);
}
}  // namespace

cudaError_t launch_quantize_axis0(const void* x, int dtype, int64_t rows, int64_t cols, int fmt, void* codes,
                                  uint8_t* scales, int layout, cudaStream_t st) {
    if (quantize_axis0_direct_applies(x, dtype, cols, codes))
        return launch_quantize_axis0_direct(x, rows, cols, fmt, codes, scales, layout, st);
    if (quantize_axis0_tiled_applies(x, dtype, cols))
        return launch_quantize_axis0_tiled(x, dtype, rows, cols, fmt, codes, scales, layout, st);
    uint8_t* c = static_cast<uint8_t*>(codes);
    if (dtype == DT_F32) return axis0_fmt<float, 1>(static_cast<const float*>(x), rows, cols, fmt, c, scales, layout, st);
    const __nv_bfloat16* p = static_cast<const __nv_bfloat16*>(x);
    // two columns per 32-bit load when every row starts on a 4-byte boundary
    if ((cols & 1) == 0) return axis0_fmt<__nv_bfloat16, 2>(p, rows, cols, fmt, c, scales, layout, st);
    return axis0_fmt<__nv_bfloat16, 1>(p, rows, cols, fmt, c, scales, layout, st);
}

cudaError_t launch_scales_to_mma(const uint8_t* a_src, int64_t a_rows, const uint8_t* b_src, int64_t b_rows,
                                 int64_t cols, uint8_t* a_dst, uint8_t* b_dst, cudaStream_t st) {
    const int64_t ng = cols / 128;  // 4-block words per row
    if (ng == 0 || (a_rows == 0 && b_rows == 0)) return cudaSuccess;
    const int64_t gchunks = (ng + kRmGroups - 1) / kRmGroups;
    RmOperand a{reinterpret_cast<const uint32_t*>(a_src), reinterpret_cast<uint32_t*>(a_dst), a_rows,
                (a_rows + 127) / 128 * gchunks};
    RmOperand b{reinterpret_cast<const uint32_t*>(b_src), reinterpret_cast<uint32_t*>(b_dst), b_rows,
                (b_rows + 127) / 128 * gchunks};
    return launch_pdl(scales_to_mma_kernel, dim3((unsigned)(a.ctas + b.ctas)), dim3(256), 0, st, a, b, ng, gchunks);
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
