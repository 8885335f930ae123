// mx_abi.cu -- the extern "C" boundary declared in include/mx.h.
//
// Host-side argument checks (the type verifier of "A Dialect Is a Set of
// Co-Designed Decisions: Designing for MX Quantization in MLIR", "The type:
// !mx.tensor": block size 32 dividing the last dimension), device checks, and
// dispatch to the kernel launchers.  Every check runs before anything is
// launched; a failed check launches nothing and returns an mx_status_t with a
// thread-local detail string.
#include <cuda_runtime.h>

#include <cstdint>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mx.h"
#include "mx_internal.h"

namespace mx {
cudaError_t read_clear_device_error(unsigned* out, cudaStream_t st);  // mx_gemm.cu
}

namespace {

thread_local char g_detail[256] = "";

mx_status_t fail(mx_status_t s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
mx_status_t fail(mx_status_t s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return s;
}

mx_status_t ok() {
    g_detail[0] = 0;
    return MX_OK;
}

mx_status_t cuda_fail(cudaError_t e, const char* where) {
    return fail(MX_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_fmt(int f) { return f == MX_E2M1 || f == MX_E4M3FN; }
bool valid_layout(int l) { return l == MX_SCALES_ROWMAJOR || l == MX_SCALES_MMA; }

// Device must be an sm_103 part (GB300).  Cached per device ordinal.
mx_status_t check_device() {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(MX_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    static std::mutex mu;
    static int cached[64] = {0};  // 0 unknown, 1 ok, 2 wrong arch
    if (dev < 0 || dev >= 64) return fail(MX_ERR_NO_DEVICE, "device ordinal %d out of range", dev);
    {
        std::lock_guard<std::mutex> lk(mu);
        if (cached[dev] == 0) {
            int major = 0, minor = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
                cudaGetLastError();
                return fail(MX_ERR_NO_DEVICE, "cannot query device %d", dev);
            }
            cached[dev] = (major == 10 && minor == 3) ? 1 : 2;
        }
        if (cached[dev] == 2)
            return fail(MX_ERR_NO_DEVICE, "device %d is not sm_103 (this library is built for sm_103a only)", dev);
    }
    return MX_OK;
}

mx_status_t check_common(int block_size, int scale_type) {
    if (block_size != 32) return fail(MX_ERR_UNSUPPORTED, "block_size %d (only 32 is supported)", block_size);
    if (scale_type != MX_SCALE_E8M0) return fail(MX_ERR_UNSUPPORTED, "scale_type %d (only E8M0)", scale_type);
    return MX_OK;
}

mx_status_t check_shape(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return fail(MX_ERR_SHAPE, "negative dimension (%lld x %lld)", (long long)rows,
                                          (long long)cols);
    if (cols % 32 != 0)
        return fail(MX_ERR_SHAPE, "cols %lld is not a multiple of the block size 32", (long long)cols);
    if (rows > (int64_t(1) << 40) || cols > (int64_t(1) << 40)) return fail(MX_ERR_SHAPE, "dimension too large");
    return MX_OK;
}

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

}  // namespace

namespace mx {
// For entry points defined in other files: a failure with its detail text.
mx_status_t record_failure(mx_status_t s, const char* detail) { return fail(s, "%s", detail); }
}  // namespace mx

extern "C" {

int64_t mx_codes_bytes(mx_format_t fmt, int64_t rows, int64_t cols) {
    if (!valid_fmt(fmt) || rows < 0 || cols < 0 || cols % 32) return -1;
    return fmt == MX_E2M1 ? rows * cols / 2 : rows * cols;
}

int64_t mx_scales_bytes(mx_scale_layout_t layout, int64_t rows, int64_t cols) {
    if (!valid_layout(layout) || rows < 0 || cols < 0 || cols % 32) return -1;
    const int64_t nb = cols / 32;
    if (layout == MX_SCALES_ROWMAJOR) return rows * nb;
    if (rows == 0 || nb == 0) return 0;
    return mx::round_up(rows, 128) / 128 * (mx::round_up(nb, 4) / 4) * 512;
}

mx_status_t mx_quantize(const void* x, mx_dtype_t x_dtype, int64_t rows, int64_t cols, mx_format_t fmt,
                        int block_size, mx_scale_type_t scale_type, void* codes, uint8_t* scales,
                        mx_scale_layout_t scale_layout, void* stream) {
    mx_status_t s;
    if ((s = check_common(block_size, scale_type)) != MX_OK) return s;
    if (!valid_fmt(fmt)) return fail(MX_ERR_UNSUPPORTED, "element format %d", (int)fmt);
    if (x_dtype != MX_F32 && x_dtype != MX_BF16) return fail(MX_ERR_UNSUPPORTED, "input dtype %d", (int)x_dtype);
    if (!valid_layout(scale_layout)) return fail(MX_ERR_UNSUPPORTED, "scale layout %d", (int)scale_layout);
    if ((s = check_shape(rows, cols)) != MX_OK) return s;
    if (rows == 0 || cols == 0) return ok();
    if (!x || !codes || !scales) return fail(MX_ERR_NULL, "x, codes and scales must be non-NULL");
    if (!aligned(x, 16) || !aligned(codes, 16))
        return fail(MX_ERR_ALIGN, "x and codes must be 16-byte aligned");
    if (!aligned(scales, scale_layout == MX_SCALES_MMA ? 16 : 4))
        return fail(MX_ERR_ALIGN, "scales must be %d-byte aligned", scale_layout == MX_SCALES_MMA ? 16 : 4);
    const int64_t xb = rows * cols * (x_dtype == MX_F32 ? 4 : 2);
    if (overlaps(x, xb, codes, mx_codes_bytes(fmt, rows, cols)) ||
        overlaps(x, xb, scales, mx_scales_bytes(scale_layout, rows, cols)) ||
        overlaps(codes, mx_codes_bytes(fmt, rows, cols), scales, mx_scales_bytes(scale_layout, rows, cols)))
        return fail(MX_ERR_UNSUPPORTED, "input and outputs overlap");
    if ((s = check_device()) != MX_OK) return s;
    cudaError_t e = mx::launch_quantize(x, x_dtype, rows, cols, fmt, codes, scales, scale_layout,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    return ok();
}

mx_status_t mx_dequantize(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols, mx_format_t fmt,
                          int block_size, mx_scale_type_t scale_type, mx_scale_layout_t scale_layout, float* y,
                          void* stream) {
    mx_status_t s;
    if ((s = check_common(block_size, scale_type)) != MX_OK) return s;
    if (!valid_fmt(fmt)) return fail(MX_ERR_UNSUPPORTED, "element format %d", (int)fmt);
    if (!valid_layout(scale_layout)) return fail(MX_ERR_UNSUPPORTED, "scale layout %d", (int)scale_layout);
    if ((s = check_shape(rows, cols)) != MX_OK) return s;
    if (rows == 0 || cols == 0) return ok();
    if (!codes || !scales || !y) return fail(MX_ERR_NULL, "codes, scales and y must be non-NULL");
    if (!aligned(codes, 16) || !aligned(y, 16)) return fail(MX_ERR_ALIGN, "codes and y must be 16-byte aligned");
    if (overlaps(y, rows * cols * 4, codes, mx_codes_bytes(fmt, rows, cols)) ||
        overlaps(y, rows * cols * 4, scales, mx_scales_bytes(scale_layout, rows, cols)))
        return fail(MX_ERR_UNSUPPORTED, "output overlaps an input");
    if ((s = check_device()) != MX_OK) return s;
    cudaError_t e = mx::launch_dequantize(codes, scales, rows, cols, fmt, scale_layout, y,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dequantize launch");
    return ok();
}

mx_status_t mx_quantize_axis(const void* x, mx_dtype_t x_dtype, int64_t rows, int64_t cols, int axis,
                             mx_format_t fmt, int block_size, mx_scale_type_t scale_type, void* codes,
                             uint8_t* scales, mx_scale_layout_t scale_layout, void* stream) {
    if (axis == 1)
        return mx_quantize(x, x_dtype, rows, cols, fmt, block_size, scale_type, codes, scales, scale_layout, stream);
    if (axis != 0) return fail(MX_ERR_UNSUPPORTED, "block axis %d (0 or 1)", axis);
    mx_status_t s;
    if ((s = check_common(block_size, scale_type)) != MX_OK) return s;
    if (!valid_fmt(fmt)) return fail(MX_ERR_UNSUPPORTED, "element format %d", (int)fmt);
    if (x_dtype != MX_F32 && x_dtype != MX_BF16) return fail(MX_ERR_UNSUPPORTED, "input dtype %d", (int)x_dtype);
    if (!valid_layout(scale_layout)) return fail(MX_ERR_UNSUPPORTED, "scale layout %d", (int)scale_layout);
    if ((s = check_shape(cols, rows)) != MX_OK) return s;  // blocks run along rows
    if (rows == 0 || cols == 0) return ok();
    if (!x || !codes || !scales) return fail(MX_ERR_NULL, "x, codes and scales must be non-NULL");
    if (!aligned(x, 16) || !aligned(codes, 16))
        return fail(MX_ERR_ALIGN, "x and codes must be 16-byte aligned");
    if (!aligned(scales, scale_layout == MX_SCALES_MMA ? 16 : 4))
        return fail(MX_ERR_ALIGN, "scales must be %d-byte aligned", scale_layout == MX_SCALES_MMA ? 16 : 4);
    const int64_t xb = rows * cols * (x_dtype == MX_F32 ? 4 : 2);
    const int64_t cb = mx_codes_bytes(fmt, cols, rows), sb = mx_scales_bytes(scale_layout, cols, rows);
    if (overlaps(x, xb, codes, cb) || overlaps(x, xb, scales, sb) || overlaps(codes, cb, scales, sb))
        return fail(MX_ERR_UNSUPPORTED, "input and outputs overlap");
    if ((s = check_device()) != MX_OK) return s;
    cudaError_t e = mx::launch_quantize_axis0(x, x_dtype, rows, cols, fmt, codes, scales, scale_layout,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "axis-0 quantize launch");
    return ok();
}

mx_status_t mx_dequantize_bf16(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                               mx_format_t fmt, int block_size, mx_scale_type_t scale_type,
                               mx_scale_layout_t scale_layout, void* y, void* stream) {
    mx_status_t s;
    if ((s = check_common(block_size, scale_type)) != MX_OK) return s;
    if (!valid_fmt(fmt)) return fail(MX_ERR_UNSUPPORTED, "element format %d", (int)fmt);
    if (!valid_layout(scale_layout)) return fail(MX_ERR_UNSUPPORTED, "scale layout %d", (int)scale_layout);
    if ((s = check_shape(rows, cols)) != MX_OK) return s;
    if (rows == 0 || cols == 0) return ok();
    if (!codes || !scales || !y) return fail(MX_ERR_NULL, "codes, scales and y must be non-NULL");
    if (!aligned(codes, 16) || !aligned(y, 16)) return fail(MX_ERR_ALIGN, "codes and y must be 16-byte aligned");
    if (overlaps(y, rows * cols * 2, codes, mx_codes_bytes(fmt, rows, cols)) ||
        overlaps(y, rows * cols * 2, scales, mx_scales_bytes(scale_layout, rows, cols)))
        return fail(MX_ERR_UNSUPPORTED, "output overlaps an input");
    if ((s = check_device()) != MX_OK) return s;
    cudaError_t e = mx::launch_dequantize_bf16(codes, scales, rows, cols, fmt, scale_layout, y,
                                               static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "bf16 dequantize launch");
    return ok();
}

mx_status_t mx_fold_scale(uint8_t* scales, int64_t rows, int64_t cols, mx_scale_layout_t scale_layout,
                          double scalar, void* stream) {
    if (!valid_layout(scale_layout)) return fail(MX_ERR_UNSUPPORTED, "scale layout %d", (int)scale_layout);
    mx_status_t s;
    if ((s = check_shape(rows, cols)) != MX_OK) return s;
    // foldable: a positive finite power of two (frexp mantissa exactly 1/2)
    int ex = 0;
    if (!(scalar > 0.0) || !std::isfinite(scalar) || std::frexp(scalar, &ex) != 0.5)
        return fail(MX_ERR_UNSUPPORTED, "scalar %g is not a positive power of two", scalar);
    const int j = ex - 1;
    if (rows == 0 || cols == 0) return ok();
    if (!scales) return fail(MX_ERR_NULL, "scales must be non-NULL");
    if ((s = check_device()) != MX_OK) return s;
    // beyond +-254 every byte saturates the same way
    const int jc = j > 255 ? 255 : (j < -255 ? -255 : j);
    cudaError_t e = mx::launch_fold_scale(scales, rows, cols, scale_layout, jc, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fold_scale launch");
    return ok();
}

mx_status_t mx_block_matmul_act(const void* a, mx_dtype_t a_dtype, mx_format_t a_fmt, const void* b_codes,
                                const uint8_t* b_scales, mx_format_t b_fmt, mx_scale_layout_t b_scale_layout,
                                int block_size, mx_scale_type_t scale_type, int64_t M, int64_t N, int64_t K, float* C,
                                void* stream) {
    mx_status_t s;
    if ((s = check_common(block_size, scale_type)) != MX_OK) return s;
    if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt)) return fail(MX_ERR_UNSUPPORTED, "element formats %d, %d",
                                                            (int)a_fmt, (int)b_fmt);
    if (a_dtype != MX_F32 && a_dtype != MX_BF16) return fail(MX_ERR_UNSUPPORTED, "activation dtype %d", (int)a_dtype);
    if (a_fmt == MX_E2M1 && b_fmt == MX_E4M3FN)
        return fail(MX_ERR_UNSUPPORTED, "E2M1 activations need E2M1 weights here (quantize with mx_quantize instead)");
    if (b_scale_layout != MX_SCALES_MMA)
        return fail(MX_ERR_UNSUPPORTED, "the weights' scales must be in MX_SCALES_MMA");
    if (M < 0 || N < 0 || K < 0) return fail(MX_ERR_SHAPE, "negative dimension");
    if (M > 64)
        return fail(MX_ERR_UNSUPPORTED,
                    "M = %lld > 64: quantize A once with mx_quantize and use mx_block_matmul (a larger A would be "
                    "quantized again for every column tile)", (long long)M);
    if (K % 32) return fail(MX_ERR_SHAPE, "K %lld is not a multiple of the block size 32", (long long)K);
    if (N > (1ll << 31) - 256 || K > (1ll << 31) - 256) return fail(MX_ERR_SHAPE, "dimension too large");
    const bool mixed = a_fmt != b_fmt;
    if (mixed && K % 128)
        return fail(MX_ERR_SHAPE, "mixed E2M1/E4M3FN operands need K %% 128 == 0 (K = %lld)", (long long)K);
    if (M == 0 || N == 0 || K == 0) return ok();
    if (!a || !b_codes || !b_scales || !C) return fail(MX_ERR_NULL, "operand pointers must be non-NULL");
    if (!aligned(a, 32)) return fail(MX_ERR_ALIGN, "the activations must be 32-byte aligned");
    if (!aligned(b_codes, mixed ? 32 : 16) || !aligned(b_scales, 16) || !aligned(C, 16))
        return fail(MX_ERR_ALIGN, "weight codes (32 B when E2M1 in a mixed product), scales and C must be 16-byte aligned");
    const int64_t cb = M * N * 4;
    if (overlaps(C, cb, a, M * K * (a_dtype == MX_F32 ? 4 : 2)) || overlaps(C, cb, b_codes, mx_codes_bytes(b_fmt, N, K)) ||
        overlaps(C, cb, b_scales, mx_scales_bytes(MX_SCALES_MMA, N, K)))
        return fail(MX_ERR_UNSUPPORTED, "C overlaps an input");
    if ((s = check_device()) != MX_OK) return s;
    mx::GemmActArgs g{a, a_dtype, a_fmt, b_codes, b_scales, b_fmt, M, N, K, C};
    const char* detail = nullptr;
    cudaError_t e = mx::launch_block_matmul_act(g, static_cast<cudaStream_t>(stream), &detail);
    if (e != cudaSuccess) return detail ? fail(MX_ERR_CUDA, "%s", detail) : cuda_fail(e, "block_matmul_act launch");
    return ok();
}

mx_status_t mx_block_matmul_f32b(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt,
                                 mx_scale_layout_t a_scale_layout, int block_size, mx_scale_type_t scale_type,
                                 const float* B, int64_t M, int64_t N, int64_t K, float* C, void* stream) {
    mx_status_t s;
    if ((s = check_common(block_size, scale_type)) != MX_OK) return s;
    if (!valid_fmt(a_fmt)) return fail(MX_ERR_UNSUPPORTED, "element format %d", (int)a_fmt);
    if (!valid_layout(a_scale_layout)) return fail(MX_ERR_UNSUPPORTED, "scale layout %d", (int)a_scale_layout);
    if (M < 0 || N < 0 || K < 0) return fail(MX_ERR_SHAPE, "negative dimension");
    if (K % 32) return fail(MX_ERR_SHAPE, "K %lld is not a multiple of the block size 32", (long long)K);
    if (M > (1ll << 40) || N > (1ll << 31) - 1024 || K > (1ll << 31) - 1024)
        return fail(MX_ERR_SHAPE, "dimension too large");
    if (M == 0 || N == 0 || K == 0) return ok();  // C += (empty sum) is C
    if (N % 4) return fail(MX_ERR_ALIGN, "N %lld: rows of B and C must be whole 16-byte units (N %% 4 == 0)",
                           (long long)N);
    if (!a_codes || !a_scales || !B || !C) return fail(MX_ERR_NULL, "operand pointers must be non-NULL");
    if (!aligned(a_codes, 16) || !aligned(a_scales, 16) || !aligned(B, 16) || !aligned(C, 16))
        return fail(MX_ERR_ALIGN, "A codes, A scales, B and C must be 16-byte aligned");
    const int64_t cb = M * N * 4;
    if (overlaps(C, cb, a_codes, mx_codes_bytes(a_fmt, M, K)) ||
        overlaps(C, cb, a_scales, mx_scales_bytes(a_scale_layout, M, K)) || overlaps(C, cb, B, K * N * 4))
        return fail(MX_ERR_UNSUPPORTED, "C overlaps an input");
    if ((s = check_device()) != MX_OK) return s;
    mx::GemmF32bArgs g{a_codes, a_scales, a_fmt, a_scale_layout, B, M, N, K, C};
    const char* detail = nullptr;
    cudaError_t e = mx::launch_block_matmul_f32b(g, static_cast<cudaStream_t>(stream), &detail);
    if (e != cudaSuccess) return detail ? fail(MX_ERR_CUDA, "%s", detail) : cuda_fail(e, "block_matmul_f32b launch");
    return ok();
}

mx_status_t mx_measure_mma_rate(mx_format_t fmt, int iters, double* tflops, void* stream) {
    if (!valid_fmt(fmt)) return fail(MX_ERR_UNSUPPORTED, "element format %d", (int)fmt);
    if (iters < 1 || iters > 1000000) return fail(MX_ERR_SHAPE, "iters %d outside 1..1000000", iters);
    if (!tflops) return fail(MX_ERR_NULL, "tflops must be non-NULL");
    mx_status_t s;
    if ((s = check_device()) != MX_OK) return s;
    cudaError_t e = mx::measure_mma_rate(fmt == MX_E2M1 ? 1 : 0, iters, tflops, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorLaunchTimeout) return fail(MX_ERR_TIMEOUT, "an MMA-rate CTA gave up waiting for its commit");
    if (e != cudaSuccess) return cuda_fail(e, "MMA-rate measurement");
    return ok();
}

}  // extern "C"

namespace {

// The argument checks of block_matmul (shared by mx_block_matmul and
// mx_block_matmul_ws).  MX_OK with *empty set: nothing to compute.
mx_status_t check_block_matmul(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt, const void* b_codes,
                               const uint8_t* b_scales, mx_format_t b_fmt, mx_scale_layout_t scale_layout,
                               int block_size, mx_scale_type_t scale_type, int64_t M, int64_t N, int64_t K,
                               const float* C, bool* empty) {
    *empty = false;
    mx_status_t s;
    if ((s = check_common(block_size, scale_type)) != MX_OK) return s;
    if (!valid_fmt(a_fmt) || !valid_fmt(b_fmt)) return fail(MX_ERR_UNSUPPORTED, "element formats %d, %d",
                                                            (int)a_fmt, (int)b_fmt);
    if (!valid_layout(scale_layout)) return fail(MX_ERR_UNSUPPORTED, "scale layout %d", (int)scale_layout);
    if (M < 0 || N < 0 || K < 0) return fail(MX_ERR_SHAPE, "negative dimension");
    if (K % 32) return fail(MX_ERR_SHAPE, "K %lld is not a multiple of the block size 32", (long long)K);
    if (M > (1ll << 31) - 256 || N > (1ll << 31) - 256 || K > (1ll << 31) - 256)
        return fail(MX_ERR_SHAPE, "dimension too large");
    const bool mixed = a_fmt != b_fmt;
    if (mixed && K % 128)
        return fail(MX_ERR_SHAPE, "mixed E2M1/E4M3FN operands need K %% 128 == 0 (K = %lld)", (long long)K);
    if (scale_layout == MX_SCALES_ROWMAJOR && K % 128)
        return fail(MX_ERR_SHAPE, "row-major scales need K %% 128 == 0 (K = %lld); use MX_SCALES_MMA",
                    (long long)K);
    if (M == 0 || N == 0 || K == 0) {  // C += (empty sum) is C
        *empty = true;
        return MX_OK;
    }
    if (!a_codes || !a_scales || !b_codes || !b_scales || !C)
        return fail(MX_ERR_NULL, "operand pointers must be non-NULL");
    if (!aligned(a_codes, 16) || !aligned(b_codes, 16) || !aligned(C, 16) || !aligned(a_scales, 16) ||
        !aligned(b_scales, 16))
        return fail(MX_ERR_ALIGN, "codes, scales and C must be 16-byte aligned");
    if (mixed && !aligned(a_fmt == MX_E2M1 ? a_codes : b_codes, 32))
        return fail(MX_ERR_ALIGN, "the E2M1 operand of a mixed product must be 32-byte aligned");
    const int64_t cb = M * N * 4;
    if (overlaps(C, cb, a_codes, mx_codes_bytes(a_fmt, M, K)) ||
        overlaps(C, cb, b_codes, mx_codes_bytes(b_fmt, N, K)) ||
        overlaps(C, cb, a_scales, mx_scales_bytes(scale_layout, M, K)) ||
        overlaps(C, cb, b_scales, mx_scales_bytes(scale_layout, N, K)))
        return fail(MX_ERR_UNSUPPORTED, "C overlaps an input");
    return MX_OK;
}

mx_status_t run_block_matmul(const mx::GemmArgs& g, void* stream) {
    const char* detail = nullptr;
    cudaError_t e = mx::launch_block_matmul(g, static_cast<cudaStream_t>(stream), &detail);
    if (e != cudaSuccess) return fail(MX_ERR_CUDA, "block_matmul: %s%s%s", cudaGetErrorString(e),
                                      detail ? ": " : "", detail ? detail : "");
    return ok();
}

// Where the tensor-core-layout copy of B's scales starts in a workspace.
int64_t ws_b_offset(int64_t M, int64_t K) { return mx::round_up(mx_scales_bytes(MX_SCALES_MMA, M, K), 256); }

}  // namespace

extern "C" {

mx_status_t mx_block_matmul(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt, const void* b_codes,
                            const uint8_t* b_scales, mx_format_t b_fmt, mx_scale_layout_t scale_layout,
                            int block_size, mx_scale_type_t scale_type, int64_t M, int64_t N, int64_t K, float* C,
                            void* stream) {
    bool empty;
    mx_status_t s = check_block_matmul(a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, scale_layout, block_size,
                                       scale_type, M, N, K, C, &empty);
    if (s != MX_OK) return s;
    if (empty) return ok();
    if ((s = check_device()) != MX_OK) return s;
    return run_block_matmul({a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, scale_layout, M, N, K, C}, stream);
}

int64_t mx_block_matmul_workspace_bytes(mx_scale_layout_t scale_layout, int64_t M, int64_t N, int64_t K) {
    if (!valid_layout(scale_layout) || M < 0 || N < 0 || K < 0 || K % 32) return -1;
    if (scale_layout == MX_SCALES_MMA || M == 0 || N == 0 || K == 0) return 0;
    return ws_b_offset(M, K) + mx::round_up(mx_scales_bytes(MX_SCALES_MMA, N, K), 256);
}

mx_status_t mx_block_matmul_ws(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt, const void* b_codes,
                               const uint8_t* b_scales, mx_format_t b_fmt, mx_scale_layout_t scale_layout,
                               int block_size, mx_scale_type_t scale_type, int64_t M, int64_t N, int64_t K,
                               float* C, void* workspace, int64_t workspace_bytes, void* stream) {
    bool empty;
    mx_status_t s = check_block_matmul(a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, scale_layout, block_size,
                                       scale_type, M, N, K, C, &empty);
    if (s != MX_OK) return s;
    if (empty) return ok();
    if (scale_layout == MX_SCALES_MMA) {
        if ((s = check_device()) != MX_OK) return s;
        return run_block_matmul({a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, scale_layout, M, N, K, C},
                                stream);
    }
    const int64_t need = mx_block_matmul_workspace_bytes(scale_layout, M, N, K);
    if (!workspace) return fail(MX_ERR_NULL, "workspace must be non-NULL for row-major scales");
    if (workspace_bytes < need)
        return fail(MX_ERR_SHAPE, "workspace of %lld bytes; these shapes need %lld (mx_block_matmul_workspace_bytes)",
                    (long long)workspace_bytes, (long long)need);
    if (!aligned(workspace, 256)) return fail(MX_ERR_ALIGN, "workspace must be 256-byte aligned");
    if (overlaps(workspace, need, C, M * N * 4) || overlaps(workspace, need, a_codes, mx_codes_bytes(a_fmt, M, K)) ||
        overlaps(workspace, need, b_codes, mx_codes_bytes(b_fmt, N, K)) ||
        overlaps(workspace, need, a_scales, mx_scales_bytes(scale_layout, M, K)) ||
        overlaps(workspace, need, b_scales, mx_scales_bytes(scale_layout, N, K)))
        return fail(MX_ERR_UNSUPPORTED, "workspace overlaps C or an input");
    if ((s = check_device()) != MX_OK) return s;
    if (mx::block_matmul_gathers_scales_fast(a_fmt, b_fmt, M, N, K))
        // decode shapes: the product reads the row-major scales itself, one launch
        return run_block_matmul({a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, scale_layout, M, N, K, C},
                                stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint8_t* a_sf = ws;
    uint8_t* b_sf = ws + ws_b_offset(M, K);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = mx::launch_scales_to_mma(a_scales, M, b_scales, N, K, a_sf, b_sf, st);
    if (e != cudaSuccess) return cuda_fail(e, "scale relayout launch");
    return run_block_matmul({a_codes, a_sf, a_fmt, b_codes, b_sf, b_fmt, MX_SCALES_MMA, M, N, K, C}, stream);
}

mx_status_t mx_scales_relayout(const uint8_t* src, mx_scale_layout_t src_layout, int64_t rows, int64_t cols,
                               uint8_t* dst, mx_scale_layout_t dst_layout, void* stream) {
    mx_status_t s;
    if (!valid_layout(src_layout) || !valid_layout(dst_layout))
        return fail(MX_ERR_UNSUPPORTED, "scale layouts %d -> %d", (int)src_layout, (int)dst_layout);
    if ((s = check_shape(rows, cols)) != MX_OK) return s;
    if (rows == 0 || cols == 0) return ok();
    if (!src || !dst) return fail(MX_ERR_NULL, "src and dst must be non-NULL");
    if (overlaps(src, mx_scales_bytes(src_layout, rows, cols), dst, mx_scales_bytes(dst_layout, rows, cols)))
        return fail(MX_ERR_UNSUPPORTED, "src and dst overlap");
    if ((s = check_device()) != MX_OK) return s;
    cudaError_t e = mx::launch_relayout(src, src_layout, rows, cols, dst, dst_layout,
                                        static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "relayout launch");
    return ok();
}

mx_status_t mx_device_status(void* stream) {
    mx_status_t s;
    if ((s = check_device()) != MX_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    unsigned word = 0;
    e = mx::read_clear_device_error(&word, st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word & 1u) return fail(MX_ERR_TIMEOUT, "a kernel gave up waiting on a barrier (device error word 0x%x)", word);
    return ok();
}

mx_status_t mx_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
    if (limit_ns < 1000ull || limit_ns > 10000000000ull)
        return fail(MX_ERR_UNSUPPORTED, "limit_ns must be in [1e3, 1e10]");
    mx_status_t s;
    if ((s = check_device()) != MX_OK) return s;
    cudaError_t e = mx::launch_wait_selftest(limit_ns, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
    return ok();
}

const char* mx_status_string(mx_status_t status) {
    switch (status) {
        case MX_OK: return "MX_OK";
        case MX_ERR_NULL: return "MX_ERR_NULL: a required pointer is NULL";
        case MX_ERR_SHAPE: return "MX_ERR_SHAPE: shape not accepted";
        case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED: parameter value not supported";
        case MX_ERR_ALIGN: return "MX_ERR_ALIGN: pointer misaligned";
        case MX_ERR_TIMEOUT: return "MX_ERR_TIMEOUT: a kernel gave up waiting";
        case MX_ERR_CUDA: return "MX_ERR_CUDA: CUDA call failed";
        case MX_ERR_NO_DEVICE: return "MX_ERR_NO_DEVICE: no sm_103 device";
    }
    return "unknown mx_status_t";
}

const char* mx_last_error_detail(void) { return g_detail; }

}  // extern "C"

namespace mx {

uint64_t wait_limit_ns() {
    static uint64_t v = [] {
        const char* s = std::getenv("MX_WAIT_LIMIT_NS");
        if (s) {
            unsigned long long x = std::strtoull(s, nullptr, 10);
            if (x >= 1000ull && x <= 60000000000ull) return (uint64_t)x;
        }
        return (uint64_t)4000000000ull;  // 4 s
    }();
    return v;
}

int sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    static int cached[64] = {0};
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        n = 148;
    }
    if (dev >= 0 && dev < 64) cached[dev] = n;
    return n;
}

}  // namespace mx
