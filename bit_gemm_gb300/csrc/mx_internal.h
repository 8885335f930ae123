// mx_internal.h -- launchers shared between the C-ABI layer and the kernels.
// Arguments are already validated by the caller (mx_abi.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "mx.h"

#include <mutex>
#include <set>
#include <utility>

namespace mx {

// Raise a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device, size).
inline cudaError_t ensure_smem_limit(const void* kern, int bytes) {
    static std::mutex mu;
    static std::set<std::pair<std::pair<const void*, int>, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(std::make_pair(kern, dev), bytes);
    if (done.count(key)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert(key);
    return e;
}

// Launch with programmatic stream serialization (see pdl_wait in
// mx_device.cuh): the kernel may be scheduled while its predecessor in the
// stream drains, and must call pdl_wait() before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

enum Fmt : int { FMT_E2M1 = 1, FMT_E4M3 = 2 };
enum Layout : int { LAYOUT_ROWMAJOR = 0, LAYOUT_MMA = 1 };
enum DType : int { DT_F32 = 1, DT_BF16 = 2 };

// Offset of scale (r, j) in the tensor-core scale layout; nb4 = blocks per
// row rounded up to a multiple of 4.
__host__ __device__ inline int64_t mma_scale_offset(int64_t r, int64_t j, int64_t nb4) {
    return ((r >> 7) * (nb4 >> 2) + (j >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3);
}

__host__ __device__ inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

cudaError_t launch_quantize(const void* x, int dtype, int64_t rows, int64_t cols, int fmt, void* codes,
                            uint8_t* scales, int layout, cudaStream_t stream);
cudaError_t launch_dequantize(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols, int fmt,
                              int layout, float* y, cudaStream_t stream);
// Sets the detail text mx_last_error_detail() returns and returns s (for
// entry points defined outside mx_abi.cu).
mx_status_t record_failure(mx_status_t s, const char* detail);

// Row-major scales of two operands (a_rows and b_rows rows of cols elements,
// cols % 128 == 0, sources 4-byte aligned) rewritten in the tensor-core
// layout at a_dst and b_dst (16-byte aligned; padding included), one launch.
cudaError_t launch_scales_to_mma(const uint8_t* a_src, int64_t a_rows, const uint8_t* b_src, int64_t b_rows,
                                 int64_t cols, uint8_t* a_dst, uint8_t* b_dst, cudaStream_t st);
cudaError_t launch_relayout(const uint8_t* src, int src_layout, int64_t rows, int64_t cols, uint8_t* dst,
                            int dst_layout, cudaStream_t stream);
cudaError_t launch_dequantize_bf16(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols, int fmt,
                                   int layout, void* y, cudaStream_t stream);
cudaError_t launch_fold_scale(uint8_t* scales, int64_t rows, int64_t cols, int layout, int j, cudaStream_t stream);
// x [rows][cols] blocked along rows; codes/scales in the layout of the [cols][rows] transpose.
// The same through shared-memory tiles (TMA); applies when x and its rows start on 16-byte boundaries.
bool quantize_axis0_direct_applies(const void* x, int dtype, int64_t cols, const void* codes);
cudaError_t launch_quantize_axis0_direct(const void* x, int64_t rows, int64_t cols, int fmt, void* codes,
                                         uint8_t* scales, int layout, cudaStream_t st);
bool quantize_axis0_tiled_applies(const void* x, int dtype, int64_t cols);
cudaError_t launch_quantize_axis0_tiled(const void* x, int dtype, int64_t rows, int64_t cols, int fmt, void* codes,
                                        uint8_t* scales, int layout, cudaStream_t stream);
cudaError_t launch_quantize_axis0(const void* x, int dtype, int64_t rows, int64_t cols, int fmt, void* codes,
                                  uint8_t* scales, int layout, cudaStream_t stream);

struct GemmArgs {
    const void* a_codes;
    const uint8_t* a_scales;
    int a_fmt;
    const void* b_codes;
    const uint8_t* b_scales;
    int b_fmt;
    int scale_layout;
    int64_t M, N, K;
    float* C;
};
// Returns cudaSuccess or an error; *detail gets a static explanation on failure.
cudaError_t launch_block_matmul(const GemmArgs& a, cudaStream_t stream, const char** detail);
// True when block_matmul on row-major scales runs at about the speed of the
// tensor-core layout (decode shapes: at most 32 rows of A, K a whole number of
// two-atom stages), so a scale relayout in front of it would only add a launch.
bool block_matmul_gathers_scales_fast(int a_fmt, int b_fmt, int64_t M, int64_t N, int64_t K);

struct GemmActArgs {
    const void* act;  // [M][K] f32 or bf16
    int act_dtype;
    int act_fmt;
    const void* w_codes;  // [N][K], scales in the tensor-core layout
    const uint8_t* w_scales;
    int w_fmt;
    int64_t M, N, K;
    float* C;
};
// C += quantize(act) * W^T with the activations quantized inside the kernel (M <= 64).
cudaError_t launch_block_matmul_act(const GemmActArgs& a, cudaStream_t stream, const char** detail);

struct GemmF32bArgs {
    const void* a_codes;  // [M][K] in a_fmt
    const uint8_t* a_scales;
    int a_fmt;
    int a_layout;
    const float* B;  // [K][N] row-major, N % 4 == 0
    int64_t M, N, K;
    float* C;
};
// C += dequantize(A) * B on the CUDA cores (B has no MX encoding).
cudaError_t launch_block_matmul_f32b(const GemmF32bArgs& a, cudaStream_t stream, const char** detail);

// The library's device error word (raised by bounded waits that give up).
unsigned* device_error_word();

// cuTensorMapEncodeTiled through the runtime's driver entry point; false if
// the entry point is missing or the encoder rejects the arguments.
bool encode_tiled_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle);

// Measured rate (TFLOP/s over all SMs) of the block-scaled MMA, kind 0 =
// kind::mxf8f6f4 (E4M3), 1 = kind::mxf4 (E2M1); synchronous on `stream`.
cudaError_t measure_mma_rate(int kind, int iters, double* tflops, cudaStream_t stream);

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t stream);

// Limit (ns) for every bounded wait inside the library's kernels.
uint64_t wait_limit_ns();

int sm_count();

}  // namespace mx
