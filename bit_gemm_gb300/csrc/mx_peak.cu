// mx_peak.cu -- measured rate of the block-scaled MMA instruction.
//
// A measurement helper with no counterpart in the method: the denominator
// for the block_matmul roofline, taken on this GPU rather than from a data
// sheet.  One CTA per SM issues back-to-back tcgen05.mma (M = 128, N = 256,
// one 128-byte K atom per group of four MMAs) on operands that stay in shared
// memory, accumulating in TMEM, with the scale factors already in TMEM: no
// HBM or L2 traffic, nothing but the tensor pipe.  Each CTA times its loop
// with %globaltimer from the first issue to the commit's completion, and the
// rate is the whole grid's flops over the span from the earliest start to the
// latest end (a CTA that ran in a second wave lengthens the span instead of
// being counted as concurrent).
//
// The per-CTA times go through one file-scope device array of at most
// kP_MaxCtas CTAs, shared by every call: calls must not overlap (two streams
// or two host threads measuring at once would read each other's times).
// The kernel allocates all 512 TMEM columns of its SM; tcgen05.alloc waits
// without a time limit while another resident kernel holds TMEM there, so it
// is meant for an otherwise idle GPU.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kP_Threads = 128;
constexpr int kP_MaxCtas = 1024;
constexpr int kP_OffB = 16384;     // A: 128 rows x 128 B (one swizzle-128 atom column)
constexpr int kP_OffSfa = 49152;   // B: 256 rows x 128 B
constexpr int kP_OffSfb = 49664;   // scale tiles: A 512 B, B 1 KB
constexpr int kP_OffBar = 50688;
// far more shared memory than used, so that one CTA (and its full TMEM
// allocation) is resident per SM
constexpr int kP_Smem = 120 * 1024;

// [2 i]: CTA i's start, [2 i + 1]: its end (%globaltimer, ns); end 0 = its wait gave up
__device__ unsigned long long g_mma_rate_ns[2 * kP_MaxCtas];

template <int KIND>  // 0: kind::mxf8f6f4 (E4M3 x E4M3), 1: kind::mxf4 (E2M1 x E2M1)
__global__ void __launch_bounds__(kP_Threads, 1) mma_rate_kernel(int iters, uint64_t limit_ns, unsigned* err) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kP_OffBar);
    uint32_t* slot = reinterpret_cast<uint32_t*>(smem + kP_OffBar + 8);
    // operands: codes 0x22 (E4M3 0.15625, E2M1 pairs of 1.0), scales 2^0
    for (int i = threadIdx.x; i < kP_OffSfa / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(smem)[i] = 0x22222222u;
    for (int i = threadIdx.x; i < (kP_OffBar - kP_OffSfa) / 4; i += blockDim.x)
        reinterpret_cast<uint32_t*>(smem + kP_OffSfa)[i] = 0x7F7F7F7Fu;
    fence_proxy_async_smem();
    if (threadIdx.x < 32) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbarrier_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    if (threadIdx.x == 0) {
        const uint32_t sfa = tmem + 256, sfb = tmem + 260;  // accumulator in columns 0..255
        tc_cp_32x128b_warpx4(sfa, smem_desc(smem_u32(smem + kP_OffSfa), 0, 128, 0));
        tc_cp_32x128b_warpx4(sfb, smem_desc(smem_u32(smem + kP_OffSfb), 0, 128, 0));
        tc_cp_32x128b_warpx4(sfb + 4, smem_desc(smem_u32(smem + kP_OffSfb + 512), 0, 128, 0));
        // instruction descriptor: formats, N = 256, K-major operands, M = 128
        const uint32_t code = KIND == 1 ? 1u : 0u;
        const uint32_t idesc = (code << 7) | (code << 10) | ((256u >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24);
        const uint64_t t0 = globaltimer_ns();
        for (int it = 0; it < iters; ++it) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint64_t ad = smem_desc(smem_u32(smem) + i * 32, 0, 1024, 2);
                const uint64_t bd = smem_desc(smem_u32(smem + kP_OffB) + i * 32, 0, 1024, 2);
                const int sf_id = KIND == 1 ? (i & 1) * 2 : i;  // which scale of the 4-block word
                const uint32_t id = idesc | ((uint32_t)sf_id << 4) | ((uint32_t)sf_id << 29);
                if (KIND == 1) mma_mxf4(tmem, ad, bd, id, sfa, sfb, 1);
                else mma_mxf8f6f4(tmem, ad, bd, id, sfa, sfb, 1);
            }
        }
        tc_commit(bar);
        const bool ok = mbar_wait(bar, 0, limit_ns, err);
        g_mma_rate_ns[2 * blockIdx.x] = t0;
        g_mma_rate_ns[2 * blockIdx.x + 1] = ok ? globaltimer_ns() : 0ull;
        if (!ok) mbar_wait(bar, 0, limit_ns, err);  // give the MMAs a second bound before TMEM is freed
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t measure_mma_rate(int kind, int iters, double* tflops, cudaStream_t st) {
    const int grid = std::min(sm_count(), kP_MaxCtas);
    unsigned* err = device_error_word();
    if (!err) return cudaErrorInvalidValue;
    auto kern = kind == 1 ? mma_rate_kernel<1> : mma_rate_kernel<0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kP_Smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kP_Threads, kP_Smem, st>>>(iters, wait_limit_ns(), err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    unsigned long long ns[2 * kP_MaxCtas];
    if ((e = cudaMemcpyFromSymbolAsync(ns, g_mma_rate_ns, sizeof(unsigned long long) * 2 * grid, 0,
                                       cudaMemcpyDeviceToHost, st)) != cudaSuccess)
        return e;
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return e;
    unsigned long long first = ~0ull, last = 0;
    for (int i = 0; i < grid; ++i) {
        if (ns[2 * i + 1] == 0) return cudaErrorLaunchTimeout;  // a CTA's wait gave up
        first = std::min(first, ns[2 * i]);
        last = std::max(last, ns[2 * i + 1]);
    }
    if (last <= first) return cudaErrorUnknown;
    const double k_per_mma = kind == 1 ? 64.0 : 32.0;
    const double flops = (double)grid * iters * 4 * 2.0 * 128 * 256 * k_per_mma;
    *tflops = flops / (double)(last - first) / 1e3;
    return cudaSuccess;
}

}  // namespace mx
