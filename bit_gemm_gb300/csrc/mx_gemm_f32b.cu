// mx_gemm_f32b.cu -- block_matmul with an MX left operand and a plain f32
// right operand: C[M][N] += dequantize(A)[M][K] * B[K][N].
//
// The op of "Block-scaled matmul in MLIR" ([Dialect] "The four ops", the
// first block_matmul: quantized A, unquantized f32 B).  B carries no scales,
// so the product cannot run on the block-scaled tensor cores, and an f32 B
// cannot feed the tf32/bf16 ones without rounding it; the kernel uses the
// CUDA cores (FFMA) instead.  For decode-shaped products (a few rows of A
// against a large B) the cost is streaming B from HBM once, which this kernel
// is built around.
//
// Work split.  C is cut into tiles of 16 rows x 512 columns and K into steps
// of 32 (one MX block of A).  The units (column tile, row tile, K step), K
// step fastest, are dealt to one persistent CTA per SM as contiguous ranges
// of equal length, so every SM streams the same share of B whatever the
// shape; a CTA whose range crosses a tile boundary adds its partial sums into
// C with vector reductions (red.global.add.v4.f32) at that boundary.  Row
// tiles of the same column tile are adjacent in the order, so for M > 16 the
// 8 MB (K = 4096) column strip of B is re-read from L2, not HBM.
//
// Per CTA: warp 0 streams B by TMA, one K step (32 rows x 512 f32 = 64 KB,
// two 256-column boxes) per stage through a ring of stages; warps 1..8
// compute.  Each compute warp also decodes its share of A's block for the
// step (16 rows x 32 codes, unscaled values) into shared memory, with the
// scale kept aside: a thread sums the 32 products of a block in f32 first and
// multiplies by the block's scale 2^(s-127) once (exact unless it leaves the
// binary32 range), folding the block sum into its running sum with one FMA.
// That keeps the f32 rounding error of an output near (32 + number of blocks)
// units in the last place of sum |a*b| instead of K of them.
//
// Thread (warp w = 1..8, lane l): columns 4g..4g+3 of the tile with
// g = 32*((w-1) % 4) + l, rows 8*((w-1) / 4) .. +7; 32 sums and 32 block sums
// in registers.  Per K row it reads one float4 of B (a warp reads 512
// contiguous bytes: no bank conflicts) and two broadcast float4 of A.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kF_Rows = 16;                        // rows of C per tile
constexpr int kF_Cols = 512;                       // columns of C per tile
constexpr int kF_Half = 256;                       // columns per TMA box
constexpr int kF_KStep = 32;                       // rows of B per stage (one MX block of A)
constexpr int kF_Stages = 3;
constexpr int kF_RowGroups = 2;                    // compute warps split the 16 rows in two
constexpr int kF_TM = kF_Rows / kF_RowGroups;      // rows per thread
constexpr int kF_Workers = 4 * kF_RowGroups;       // compute warps
constexpr int kF_Threads = 32 * (kF_Workers + 1);  // + the TMA warp
constexpr int kF_HalfBytes = kF_KStep * kF_Half * 4;
constexpr int kF_StageBytes = 2 * kF_HalfBytes;    // 64 KB
constexpr int kF_OffA = kF_Stages * kF_StageBytes;               // decoded A: [2][32 k][16 rows] f32
constexpr int kF_OffS = kF_OffA + 2 * kF_KStep * kF_Rows * 4;   // block scales: [2][16] f32
constexpr int kF_OffBar = kF_OffS + 2 * kF_Rows * 4;
constexpr int kF_Smem = kF_OffBar + 2 * kF_Stages * 8 + 1024;     // + alignment slack
static_assert(kF_Rows * kF_KStep / 2 == 32 * kF_Workers, "one pair of A codes per compute thread");
static_assert(kF_Smem <= 227 * 1024, "shared memory");

struct F32bParams {
    const uint8_t* a_codes;
    const uint8_t* a_scales;
    int64_t M, N, K;
    int64_t a_row_bytes;  // bytes of codes per row of A
    int64_t nb, nb4;      // blocks per row; rounded up to 4 (tensor-core scale layout)
    int a_layout;
    int MT, NT, KB;       // row tiles, column tiles, K steps
    int64_t total;        // MT * NT * KB units
    float* C;
    uint64_t wait_limit_ns;
    unsigned* err;
};

// two E4M3FN codes (low byte = first element) -> their exact values
__device__ __forceinline__ float2 decode2_e4m3(uint32_t pair) {
    uint32_t h;
    asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}" : "=r"(h) : "r"(pair));
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// two E2M1 codes packed in a byte (low nibble = first element) -> their exact values
__device__ __forceinline__ float2 decode2_e2m1(uint32_t byte) {
    uint32_t h;
    asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}" : "=r"(h) : "r"(byte));
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

__device__ __forceinline__ float block_scale(uint32_t s) {
    // 2^(s-127) in binary32 (s = 0 is the subnormal 2^-127); 0xFF is NaN and
    // poisons every product of its block.
    return s == 0xFFu ? __uint_as_float(0x7FC00000u) : (s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u));
}

struct Unit {
    int kb, mt, nt;
    __device__ __forceinline__ void next(const F32bParams& p) {
        if (++kb == p.KB) {
            kb = 0;
            if (++mt == p.MT) {
                mt = 0;
                ++nt;
            }
        }
    }
    __device__ __forceinline__ bool same_tile(const Unit& o) const { return mt == o.mt && nt == o.nt; }
};

__device__ __forceinline__ Unit unit_at(const F32bParams& p, int64_t u) {
    Unit w;
    w.kb = (int)(u % p.KB);
    const int64_t t = u / p.KB;
    w.mt = (int)(t % p.MT);
    w.nt = (int)(t / p.MT);
    return w;
}

// The two codes and (for j == 0) the scale byte of row m of the tile, K step kb.
template <int FMT>
__device__ __forceinline__ void load_a_raw(const F32bParams& p, const Unit& w, int m, int j, uint32_t& codes,
                                           uint32_t& sbyte) {
    const int64_t row = (int64_t)w.mt * kF_Rows + m;
    codes = 0;
    sbyte = 127;
    if (row < p.M) {
        const uint8_t* rp = p.a_codes + row * p.a_row_bytes;
        if constexpr (FMT == FMT_E4M3) codes = __ldg(reinterpret_cast<const uint16_t*>(rp + (int64_t)w.kb * 32) + j);
        else codes = __ldg(rp + (int64_t)w.kb * 16 + j);
        if (j == 0)
            sbyte = __ldg(p.a_scales + (p.a_layout == LAYOUT_MMA ? mma_scale_offset(row, w.kb, p.nb4)
                                                                 : row * p.nb + w.kb));
    }
}

template <int FMT>
__global__ void __launch_bounds__(kF_Threads, 1) gemm_f32b_kernel(const __grid_constant__ CUtensorMap tm_b,
                                                                  const F32bParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    float* a_dec = reinterpret_cast<float*>(smem + kF_OffA);
    float* a_scl = reinterpret_cast<float*>(smem + kF_OffS);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kF_OffBar);
    uint64_t* empty = full + kF_Stages;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t u0 = p.total * blockIdx.x / gridDim.x, u1 = p.total * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_b);
        for (int s = 0; s < kF_Stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kF_Workers);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    if (u0 >= u1) return;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA
        if (lane == 0) {
            Unit w = unit_at(p, u0);
            bool ok = true;
            int64_t i = 0;
            for (int64_t u = u0; u < u1; ++u, ++i, w.next(p)) {
                const int stage = (int)(i % kF_Stages);
                const uint32_t phase = (uint32_t)(i / kF_Stages) & 1u;
                if (ok) ok = mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns, p.err);
                if (!ok) break;  // the compute warps time out on `full` and skip the rest
                const int32_t x = w.nt * kF_Cols, y = w.kb * kF_KStep;
                const bool second = (int64_t)x + kF_Half < p.N;  // a box wholly past N is not loaded
                uint8_t* dst = smem + stage * kF_StageBytes;
                mbar_arrive_expect_tx(&full[stage], second ? kF_StageBytes : kF_HalfBytes);
                tma_load_2d(dst, &tm_b, x, y, &full[stage]);
                if (second) tma_load_2d(dst + kF_HalfBytes, &tm_b, x + kF_Half, y, &full[stage]);
            }
            // every issued copy has landed before the CTA exits (normally long
            // since: the compute warps waited for each of them)
            const int64_t n = i;
            for (int64_t q = n > kF_Stages ? n - kF_Stages : 0; q < n; ++q)
                if (!mbar_wait(&full[q % kF_Stages], (uint32_t)(q / kF_Stages) & 1u, p.wait_limit_ns, p.err)) break;
        }
        return;
    }

    // -------------------------------------------------------------- compute
    const int t = threadIdx.x - 32;         // 0 .. 255
    const int g = t & 127;                  // column group: columns 4g .. 4g+3 of the tile
    const int rg = t >> 7;                  // row group: rows kF_TM*rg ..
    const int am = t & 15, aj = t >> 4;     // this thread decodes codes 2aj, 2aj+1 of tile row am
    const uint32_t b_off = (uint32_t)((g >> 6) * kF_HalfBytes + (g & 63) * 16);

    float acc[kF_TM][4];
#pragma unroll
    for (int r = 0; r < kF_TM; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;

    Unit w = unit_at(p, u0);
    uint32_t raw_c, raw_s;
    load_a_raw<FMT>(p, w, am, aj, raw_c, raw_s);
    bool live = true;  // false after a timed-out wait: the remaining units are skipped
    int64_t i = 0;
    for (int64_t u = u0; u < u1; ++u, ++i) {
        const int buf = (int)(i & 1);
        const int stage = (int)(i % kF_Stages);
        const uint32_t phase = (uint32_t)(i / kF_Stages) & 1u;
        // decoded codes of this step into a_dec[buf] (k-major: [k][row]), scale into a_scl[buf]
        {
            const float2 v = FMT == FMT_E4M3 ? decode2_e4m3(raw_c) : decode2_e2m1(raw_c);
            float* d = a_dec + buf * (kF_KStep * kF_Rows);
            d[(2 * aj) * kF_Rows + am] = v.x;
            d[(2 * aj + 1) * kF_Rows + am] = v.y;
            if (aj == 0) a_scl[buf * kF_Rows + am] = block_scale(raw_s);
        }
        Unit nx = w;
        nx.next(p);
        if (u + 1 < u1) load_a_raw<FMT>(p, nx, am, aj, raw_c, raw_s);  // used one step later
        // a_dec[buf] complete; every thread is also past its reads of a_dec[buf]
        // from two steps ago (it reached this barrier one step ago)
        named_bar_sync(1, 32 * kF_Workers);
        if (live) live = mbar_wait(&full[stage], phase, p.wait_limit_ns, p.err);
        if (live) {
            const uint8_t* bs = smem + stage * kF_StageBytes + b_off;
            const float* as = a_dec + buf * (kF_KStep * kF_Rows) + rg * kF_TM;
            float blk[kF_TM][4];
#pragma unroll
            for (int k = 0; k < kF_KStep; ++k) {
                const float4 b = *reinterpret_cast<const float4*>(bs + k * (kF_Half * 4));
                float a[kF_TM];
#pragma unroll
                for (int r = 0; r < kF_TM; r += 4) {
                    const float4 q = *reinterpret_cast<const float4*>(as + k * kF_Rows + r);
                    a[r] = q.x;
                    a[r + 1] = q.y;
                    a[r + 2] = q.z;
                    a[r + 3] = q.w;
                }
#pragma unroll
                for (int r = 0; r < kF_TM; ++r) {
                    if (k == 0) {
                        blk[r][0] = a[r] * b.x;
                        blk[r][1] = a[r] * b.y;
                        blk[r][2] = a[r] * b.z;
                        blk[r][3] = a[r] * b.w;
                    } else {
                        blk[r][0] = fmaf(a[r], b.x, blk[r][0]);
                        blk[r][1] = fmaf(a[r], b.y, blk[r][1]);
                        blk[r][2] = fmaf(a[r], b.z, blk[r][2]);
                        blk[r][3] = fmaf(a[r], b.w, blk[r][3]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
#pragma unroll
            for (int r = 0; r < kF_TM; ++r) {
                const float sc = a_scl[buf * kF_Rows + rg * kF_TM + r];
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(blk[r][c], sc, acc[r][c]);
            }
        }
        if (u + 1 == u1 || !nx.same_tile(w)) {
            // end of this CTA's share of the tile: add the partial sums into C
            const int64_t col = (int64_t)w.nt * kF_Cols + 4 * g;
            if (live && col < p.N) {
#pragma unroll
                for (int r = 0; r < kF_TM; ++r) {
                    const int64_t row = (int64_t)w.mt * kF_Rows + rg * kF_TM + r;
                    if (row < p.M) red_add_v4(p.C + row * p.N + col, acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
                }
            }
#pragma unroll
            for (int r = 0; r < kF_TM; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
        }
        w = nx;
    }
}

template <int FMT>
cudaError_t run_f32b(const CUtensorMap& tm, const F32bParams& p, int grid, cudaStream_t st) {
    auto kern = gemm_f32b_kernel<FMT>;
    static bool configured = false;  // per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kF_Smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, kF_Threads, kF_Smem, st>>>(tm, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_block_matmul_f32b(const GemmF32bArgs& a, cudaStream_t stream, const char** detail) {
    F32bParams p{};
    p.a_codes = static_cast<const uint8_t*>(a.a_codes);
    p.a_scales = a.a_scales;
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.a_row_bytes = a.a_fmt == FMT_E2M1 ? a.K / 2 : a.K;
    p.nb = a.K / 32;
    p.nb4 = round_up(p.nb, 4);
    p.a_layout = a.a_layout;
    p.MT = (int)((a.M + kF_Rows - 1) / kF_Rows);
    p.NT = (int)((a.N + kF_Cols - 1) / kF_Cols);
    p.KB = (int)(a.K / kF_KStep);
    p.total = (int64_t)p.MT * p.NT * p.KB;
    p.C = a.C;
    p.wait_limit_ns = wait_limit_ns();
    p.err = device_error_word();
    if (!p.err) {
        *detail = "the device error word is not addressable";
        return cudaErrorInvalidValue;
    }
    CUtensorMap tm;
    const uint64_t dims[2] = {(uint64_t)a.N, (uint64_t)a.K};
    const uint64_t strides[1] = {(uint64_t)a.N * 4};
    const uint32_t box[2] = {(uint32_t)kF_Half, (uint32_t)kF_KStep};
    if (!encode_tiled_map(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.B, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) {
        *detail = "cuTensorMapEncodeTiled rejected B";
        return cudaErrorInvalidValue;
    }
    const int grid = (int)(p.total < sm_count() ? p.total : sm_count());
    return a.a_fmt == FMT_E2M1 ? run_f32b<FMT_E2M1>(tm, p, grid, stream) : run_f32b<FMT_E4M3>(tm, p, grid, stream);
}

}  // namespace mx
