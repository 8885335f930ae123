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
constexpr int kUnroll = 2;

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

// E2M1: nearest of {0, .5, 1, 1.5, 2, 3, 4, 6} to y >= 0, ties to the lower
// magnitude, saturating at 6.  The index is the number of midpoints strictly
// below y.
__device__ __forceinline__ uint32_t round_e2m1(float y) {
    return (uint32_t)(y > 0.25f) + (uint32_t)(y > 0.75f) + (uint32_t)(y > 1.25f) + (uint32_t)(y > 1.75f) +
           (uint32_t)(y > 2.5f) + (uint32_t)(y > 3.5f) + (uint32_t)(y > 5.0f);
}

// E4M3FN: nearest finite magnitude to y in [0, 512), ties to the lower
// magnitude, saturating at 448.
//  * y < 2^-6 (subnormal range, quantum 2^-9): k = ceil(512 y - 1/2) is the
//    nearest multiple with ties down; k = 8 is the first normal 2^-6, whose
//    code is also 8.
//  * otherwise: keep 3 mantissa bits of the binary32 pattern, rounding the 20
//    dropped bits half-down (add 2^19 - 1, truncate); a carry moves into the
//    exponent as it should.  Then clamp to 448 and re-bias 127 -> 7.
__device__ __forceinline__ uint32_t round_e4m3(float y) {
    if (y < 0.015625f) {
        const float q = __fsub_rn(__fmul_rn(y, 512.0f), 0.5f);
        return (uint32_t)__float2int_ru(q) & 0xFu;
    }
    uint32_t b = (__float_as_uint(y) + 0x7FFFFu) & 0xFFF00000u;
    b = b > 0x43E00000u ? 0x43E00000u : b;  // 448 = 1.75 * 2^8
    return ((((b >> 23) - 120u) << 3) | ((b >> 20) & 7u)) & 0x7Fu;
}

// Quantize the 8 elements a thread owns, given the block's max |bits|.
// Returns the scale byte; fills 8 codes (sign included).
template <int FMT>
__device__ __forceinline__ uint32_t quantize8(const uint32_t (&u)[8], uint32_t amax_bits, uint32_t (&code)[8]) {
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
    // 2^-e; e <= 125 here, so the pattern is a normal binary32.
    const float inv = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t mag = u[i] & 0x7FFFFFFFu;
        const float y = __fmul_rn(__uint_as_float(mag), inv);  // exact where it matters
        uint32_t c = FMT == FMT_E2M1 ? round_e2m1(y) : round_e4m3(y);
        if ((u[i] >> 31) && mag) c |= kSign;  // x < 0 (not -0.0)
        code[i] = c;
    }
    return (uint32_t)(e + 127);
}

template <typename InT, int FMT, int LAYOUT>
__global__ void __launch_bounds__(kThreads) quantize_kernel(const InT* __restrict__ x, int64_t nblocks, int64_t nb,
                                                            int64_t rows, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int part = lane & 3;  // which 8 of the block's 32 elements
    const int64_t nthreads = nblocks * 4;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t nb4 = round_up(nb, 4);

    for (int64_t t0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; t0 - lane < nthreads;
         t0 += stride * kUnroll) {
        uint32_t u[kUnroll][8];
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int64_t t = t0 + q * stride;
            if (t < nthreads) {
                Load8<InT>::run(x + t * 8, u[q]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) u[q][i] = 0;
            }
        }
#pragma unroll
        for (int q = 0; q < kUnroll; ++q) {
            const int64_t t = t0 + q * stride;
            if (t - lane >= nthreads) break;  // warp-uniform: whole warp past the end
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) m = max(m, u[q][i] & 0x7FFFFFFFu);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            uint32_t c[8];
            const uint32_t sbyte = quantize8<FMT>(u[q], m, c);
            const bool valid = t < nthreads;
            const int64_t b = t >> 2;  // block index
            if (valid) {
                if (FMT == FMT_E2M1) {
                    uint32_t w = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) w |= c[i] << (4 * i);  // element 0 in the low nibble
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

    if (LAYOUT == LAYOUT_MMA) {
        // Padding of the tensor-core layout: rows up to a multiple of 128 and
        // blocks per row up to a multiple of 4 are written as 0 (scale 2^-127,
        // finite, so zero-filled operand padding contributes exactly 0).
        const int64_t r128 = round_up(rows, 128);
        const int64_t pad_rows = (r128 - rows) * nb4;
        const int64_t pad_cols = rows * (nb4 - nb);
        for (int64_t p = (int64_t)blockIdx.x * kThreads + threadIdx.x; p < pad_rows + pad_cols; p += stride) {
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
}

// --------------------------------------------------------------- dequantize

// E2M1 magnitude index (3 bits) -> binary32 bits of the magnitude.
__device__ __forceinline__ uint32_t e2m1_bits(uint32_t c) {
    const uint32_t E = (c >> 1) & 3u, M = c & 1u;
    if (E == 0) return M ? 0x3F000000u : 0u;  // 0.5 * M
    return ((E + 126u) << 23) | (M << 22);    // 2^(E-1) * (1 + M/2)
}

// E4M3FN code (7 bits) -> binary32 bits of the magnitude; 0x7F is NaN.
__device__ __forceinline__ uint32_t e4m3_bits(uint32_t c) {
    const uint32_t E = c >> 3, M = c & 7u;
    if (c == 0x7Fu) return 0x7FC00000u;
    if (E == 0) return __float_as_uint((float)M * 0.001953125f);  // M * 2^-9
    return ((E + 120u) << 23) | (M << 20);                        // 2^(E-7) * (1 + M/8)
}

template <int FMT, int LAYOUT>
__global__ void __launch_bounds__(kThreads) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                              const uint8_t* __restrict__ scales, int64_t nblocks,
                                                              int64_t nb, float* __restrict__ y) {
    const int64_t nthreads = nblocks * 4;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t nb4 = round_up(nb, 4);
    for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < nthreads; t += stride) {
        const int64_t b = t >> 2;
        int64_t soff;
        if (LAYOUT == LAYOUT_ROWMAJOR) {
            soff = b;
        } else {
            const int64_t r = b / nb, j = b - r * nb;
            soff = mma_scale_offset(r, j, nb4);
        }
        const uint32_t s = __ldg(scales + soff);
        uint32_t c[8];
        if (FMT == FMT_E2M1) {
            const uint32_t w = __ldcs(reinterpret_cast<const uint32_t*>(codes) + t);
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = (w >> (4 * i)) & 0xFu;
        } else {
            const uint2 w = __ldcs(reinterpret_cast<const uint2*>(codes) + t);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                c[i] = (w.x >> (8 * i)) & 0xFFu;
                c[4 + i] = (w.y >> (8 * i)) & 0xFFu;
            }
        }
        // 2^(s-127) as binary32 (s = 0 is the subnormal 2^-127).
        const float scale = s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t mbits, sign;
            if (FMT == FMT_E2M1) {
                mbits = e2m1_bits(c[i] & 7u);
                sign = (c[i] & 8u) << 28;
            } else {
                mbits = e4m3_bits(c[i] & 0x7Fu);
                sign = (c[i] & 0x80u) << 24;
            }
            // Exact: at most 4 significant bits times a power of two (or an
            // IEEE overflow to infinity, as the definition gives).
            v[i] = __fmul_rn(__uint_as_float(mbits | sign), scale);
            if (s == 0xFFu) v[i] = __uint_as_float(0x7FC00000u);  // NaN scale poisons the block
        }
        float4* out = reinterpret_cast<float4*>(y) + t * 2;
        __stcs(out, make_float4(v[0], v[1], v[2], v[3]));
        __stcs(out + 1, make_float4(v[4], v[5], v[6], v[7]));
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
    int64_t grid = grid_for((work + kUnroll - 1) / kUnroll, 8);
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
    const unsigned grid = (unsigned)grid_for(nblocks * 4, 8);
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
