// mx_static_ws.cu -- block_matmul on row-major scales without any allocation.
//
// mx_block_matmul_ws needs a workspace for the tensor-core-layout copy of the
// operands' scales, and the caller allocates it.  Some callers cannot: a host
// framework or plugin runtime that owns every device buffer and hands a
// library only its inputs and outputs, a process running under a fixed device
// memory budget set at start-up, or a latency-critical path where an
// allocation (which may synchronize the device) is not acceptable.  For them,
// mx_block_matmul_static_ws runs the same product with its scratch in a
// file-scope device array of kStaticWsBytes, which every GPU that loads the
// library holds until the process exits.  Nothing here calls cudaMalloc,
// cudaFree or any other allocating routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "mx.h"
#include "mx_internal.h"

namespace {

// The scratch: the tensor-core-layout scales of A and of B (each rounded up
// to 256 bytes).  16 MiB covers, for example, M = N = K = 8192 (4 MiB) and
// M = 8192, N = 28672, K = 8192 (9 MiB).
constexpr int64_t kStaticWsBytes = int64_t(16) << 20;
static __device__ __align__(256) uint8_t g_static_ws[kStaticWsBytes];

// The array's device address, looked up once per device with that device
// current.  In host code g_static_ws names a host-side stand-in, not device
// memory, so only this address may be handed to a kernel.
void* static_ws_address(mx_status_t* status) {
    static std::mutex mu;
    static void* addr[64];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        *status = mx::record_failure(MX_ERR_NO_DEVICE, "no usable CUDA device for the static workspace");
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_ws);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            char msg[160];
            snprintf(msg, sizeof(msg), "static workspace address lookup on device %d: %s", dev,
                     cudaGetErrorString(e));
            *status = mx::record_failure(MX_ERR_CUDA, msg);
            return nullptr;
        }
        addr[dev] = p;
    }
    *status = MX_OK;
    return addr[dev];
}

}  // namespace

extern "C" {

mx_status_t mx_block_matmul_static_ws(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt,
                                      const void* b_codes, const uint8_t* b_scales, mx_format_t b_fmt,
                                      mx_scale_layout_t scale_layout, int block_size, mx_scale_type_t scale_type,
                                      int64_t M, int64_t N, int64_t K, float* C, void* stream) {
    const int64_t need = mx_block_matmul_workspace_bytes(scale_layout, M, N, K);
    if (need > kStaticWsBytes) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "M = %lld, N = %lld, K = %lld need %lld bytes of scale workspace; the static workspace holds %lld "
                 "(use mx_block_matmul_ws with a larger caller-owned workspace)",
                 (long long)M, (long long)N, (long long)K, (long long)need, (long long)kStaticWsBytes);
        return mx::record_failure(MX_ERR_SHAPE, msg);
    }
    void* ws = nullptr;
    if (need > 0) {
        mx_status_t s;
        ws = static_ws_address(&s);
        if (!ws) return s;
    }
    // the checks, the relayout into the workspace and the product are those
    // of mx_block_matmul_ws
    return mx_block_matmul_ws(a_codes, a_scales, a_fmt, b_codes, b_scales, b_fmt, scale_layout, block_size,
                              scale_type, M, N, K, C, ws, ws ? kStaticWsBytes : 0, stream);
}

}  // extern "C"
