// mx_quant_axis0.cu -- quantize with the blocks along the first axis.
//
// "Block-scaled matmul in MLIR" ([Dialect] "The block axis"): the blocks of a
// K x N right-hand operand run down its columns (along K), and its codes and
// scales are stored in the layout of the N x K transpose, ready to be the
// block_matmul operand.  Two kernels:
//
// * bf16 input (even column count): loads straight to registers.  A CTA of
//   four warps takes 128 (or 64) columns x 4 blocks; a lane loads its 32 rows
//   of four (or two) neighbouring columns as 64-bit (or 32-bit) words, one
//   row segment per warp load, rounds each column's block with the row-wise
//   bf16 routine's arithmetic, and writes each column's codes of the block
//   with one 32-byte (E4M3FN) or 16-byte (E2M1) store; the scale words meet
//   in shared memory.  Many small CTAs per SM keep the loads in flight.
//
// * f32 input: units of [128 rows x 128 columns] through shared memory.  TMA
//   brings the tile in, thread c quantizes column c (four blocks, with the
//   rounding of the last-axis quantize), the 128 columns' codes -- one whole
//   128-byte (E4M3FN) or 64-byte (E2M1) run of each output row -- are staged
//   in shared memory and leave with one TMA tensor store, and the scales leave
//   as one 32-bit word per column (in the tensor-core layout a unit's scales
//   are one contiguous 512-byte tile, padding included).  Persistent CTAs:
//   warp 0 streams input tiles through a ring of stages; warps 1..4
//   quantize; units (column tile, row group), row group fastest, are dealt to
//   CTAs as contiguous ranges.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mx_quant_block.cuh"

namespace mx {
namespace {

constexpr int kX_Cols = 128;                  // columns per unit: one per quantizing thread
constexpr int kX_Blocks = 4;                  // blocks per unit along the rows (128 rows)
constexpr int kX_Rows = 32 * kX_Blocks;
constexpr int kX_Workers = kX_Cols / 32;      // quantizing warps
constexpr int kX_Threads = 32 * (kX_Workers + 1);

template <typename InT, int FMT>
struct AxisCfg {
    static constexpr int kTileBytes = kX_Rows * kX_Cols * (int)sizeof(InT);  // 32 KB bf16, 64 KB f32
    static constexpr int kCodeRun = FMT == FMT_E2M1 ? 16 * kX_Blocks : 32 * kX_Blocks;  // bytes per column per unit
    static constexpr int kStageOut = kX_Cols * kCodeRun;                     // staged codes of a unit
    static constexpr int kCtas = sizeof(InT) == 2 ? 2 : 1;                   // resident CTAs per SM
    static constexpr int kStages = 2;
    static constexpr int kOffOut = kStages * kTileBytes;
    static constexpr int kOffBar = kOffOut + 2 * kStageOut;
    static constexpr int kSmem = kOffBar + 2 * kStages * 8 + 1024;
    static_assert(kSmem * kCtas <= 227 * 1024, "shared memory");
    static_assert(kCodeRun == 128 || kCodeRun == 64, "staged rows use the 128- or 64-byte swizzle");
};

struct Axis0Params {
    int64_t rows, cols;
    int64_t nb, nb4;      // blocks per column; rounded up to 4
    int64_t nrg;          // row groups (units along the rows)
    int64_t total;        // column tiles x row groups
    uint8_t* scales;
    uint64_t wait_limit_ns;
    unsigned* err;
};

// Byte offset of 16-byte chunk j of staged row r (the swizzle the code map uses).
template <int RUN>
__device__ __forceinline__ uint32_t staged_chunk(int r, int j) {
    if constexpr (RUN == 128) return (uint32_t)(r * 128 + ((j ^ (r & 7)) << 4));
    else return (uint32_t)(r * 64 + ((j ^ ((r >> 1) & 3)) << 4));
}

template <typename InT, int FMT, int LAYOUT>
__global__ void __launch_bounds__(kX_Threads, (AxisCfg<InT, FMT>::kCtas))
    quantize_axis0_tiled_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_codes,
                                const Axis0Params p) {
    using Cf = AxisCfg<InT, FMT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + Cf::kOffBar);
    uint64_t* empty = full + Cf::kStages;

    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t u0 = p.total * blockIdx.x / gridDim.x, u1 = p.total * (blockIdx.x + 1) / gridDim.x;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_x);
        prefetch_tensormap(&tm_codes);
        for (int s = 0; s < Cf::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kX_Workers);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    pdl_wait();  // set-up above overlaps the previous kernel's tail

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA
        if (lane == 0) {
            int64_t i = 0;
            for (int64_t u = u0; u < u1; ++u, ++i) {
                const int stage = (int)(i % Cf::kStages);
                const uint32_t phase = (uint32_t)(i / Cf::kStages) & 1u;
                if (!mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns, p.err)) break;
                const int64_t ct = u / p.nrg, rg = u - ct * p.nrg;
                mbar_arrive_expect_tx(&full[stage], Cf::kTileBytes);
                tma_load_2d(smem + stage * Cf::kTileBytes, &tm_x, (int32_t)(ct * kX_Cols), (int32_t)(rg * kX_Rows),
                            &full[stage]);
            }
            // every issued copy has landed before the CTA exits
            const int64_t n = i;
            for (int64_t q = n > Cf::kStages ? n - Cf::kStages : 0; q < n; ++q)
                if (!mbar_wait(&full[q % Cf::kStages], (uint32_t)(q / Cf::kStages) & 1u, p.wait_limit_ns, p.err))
                    break;
        }
        return;
    }

    // -------------------------------------------------------------- quantize
    constexpr int kWords = FMT == FMT_E2M1 ? 4 : 8;  // code words per block
    const int t = threadIdx.x - 32;                  // column of the unit
    bool live = true;
    int64_t i = 0;
    for (int64_t u = u0; u < u1; ++u, ++i) {
        const int stage = (int)(i % Cf::kStages);
        const uint32_t phase = (uint32_t)(i / Cf::kStages) & 1u;
        const int64_t ct = u / p.nrg, rg = u - ct * p.nrg;
        const int nblk = (int)min((int64_t)kX_Blocks, p.nb - rg * kX_Blocks);
        if (live) live = mbar_wait(&full[stage], phase, p.wait_limit_ns, p.err);
        uint32_t codes[kX_Blocks][kWords];
        uint32_t sword = 0;  // scale bytes of the unit's blocks, block b in byte b (zero past nb)
#pragma unroll
        for (int b = 0; b < kX_Blocks; ++b)
#pragma unroll
            for (int q = 0; q < kWords; ++q) codes[b][q] = 0;
        if (live) {
            const InT* col = reinterpret_cast<const InT*>(smem + stage * Cf::kTileBytes) + t;
#pragma unroll
            for (int b = 0; b < kX_Blocks; ++b) {
                uint32_t v[32];
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    if constexpr (sizeof(InT) == 2)
                        v[r] = (uint32_t)reinterpret_cast<const uint16_t*>(col)[(32 * b + r) * kX_Cols] << 16;
                    else
                        v[r] = reinterpret_cast<const uint32_t*>(col)[(32 * b + r) * kX_Cols];
                }
                if (b == kX_Blocks - 1) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[stage]);  // the tile is read
                }
                const uint32_t s = quantize_column_block<FMT>(v, sizeof(InT) == 2, codes[b]);
                if (b < nblk) sword |= s << (8 * b);
            }
        }
        // stage the codes: row t of buffer (i & 1), in the swizzle of the code map.
        // That buffer was last read by the store issued two units ago, which had
        // finished reading before the barrier of the previous unit.
        uint8_t* out = smem + Cf::kOffOut + (i & 1) * Cf::kStageOut;
#pragma unroll
        for (int b = 0; b < kX_Blocks; ++b)
#pragma unroll
            for (int q = 0; q < kWords / 4; ++q)
                *reinterpret_cast<uint4*>(out + staged_chunk<Cf::kCodeRun>(t, b * (kWords / 4) + q)) =
                    make_uint4(codes[b][4 * q], codes[b][4 * q + 1], codes[b][4 * q + 2], codes[b][4 * q + 3]);
        fence_proxy_async_smem();
        if (t == 0) bulk_wait_group_read<0>();  // last unit's store is done reading the other buffer
        named_bar_sync(1, 32 * kX_Workers);
        if (t == 0 && live) {
            // rows past `cols` and bytes past the column's codes are clipped by the map
            tma_store_2d(&tm_codes, out, (int32_t)(rg * Cf::kCodeRun), (int32_t)(ct * kX_Cols));
            bulk_commit_group();
        }
        // scales
        const int64_t c = ct * kX_Cols + t;
        if (LAYOUT == LAYOUT_MMA) {
            // the unit's 128 rows x 4 blocks are one 512-byte tile; columns past
            // `cols` and blocks past nb are the layout's zero padding
            uint32_t* tile = reinterpret_cast<uint32_t*>(p.scales + (ct * (p.nb4 >> 2) + rg) * 512);
            tile[(t & 31) * 4 + ((t >> 5) & 3)] = c < p.cols ? sword : 0u;
        } else if (c < p.cols) {
            uint8_t* dst = p.scales + c * p.nb + rg * kX_Blocks;
            if (nblk == kX_Blocks && (p.nb & 3) == 0) {
                *reinterpret_cast<uint32_t*>(dst) = sword;
            } else {
                for (int b = 0; b < nblk; ++b) dst[b] = (uint8_t)(sword >> (8 * b));
            }
        }
    }
    if (t == 0) bulk_wait_group<0>();  // staged codes stay in place until stored
}

template <typename InT, int FMT, int LAYOUT>
cudaError_t run_axis0(const CUtensorMap& tx, const CUtensorMap& tc, const Axis0Params& p, cudaStream_t st) {
    using Cf = AxisCfg<InT, FMT>;
    auto kern = quantize_axis0_tiled_kernel<InT, FMT, LAYOUT>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), Cf::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t slots = (int64_t)Cf::kCtas * sm_count();
    const int grid = (int)(p.total < slots ? p.total : slots);
    return launch_pdl(kern, dim3(grid), dim3(kX_Threads), Cf::kSmem, st, tx, tc, p);
}

template <typename InT>
cudaError_t axis0_dispatch(const CUtensorMap& tx, const CUtensorMap& tc, const Axis0Params& p, int fmt, int layout,
                           cudaStream_t st) {
    if (fmt == FMT_E2M1)
        return layout == LAYOUT_MMA ? run_axis0<InT, FMT_E2M1, LAYOUT_MMA>(tx, tc, p, st)
                                    : run_axis0<InT, FMT_E2M1, LAYOUT_ROWMAJOR>(tx, tc, p, st);
    return layout == LAYOUT_MMA ? run_axis0<InT, FMT_E4M3, LAYOUT_MMA>(tx, tc, p, st)
                                : run_axis0<InT, FMT_E4M3, LAYOUT_ROWMAJOR>(tx, tc, p, st);
}

// ------------------------------------------------- bf16: loads straight to registers
//
// For bf16 input the units above leave an SM with eight quantizing warps (the
// staged tiles fill its shared memory), too few to cover the latency of their
// column walks.  Here nothing is staged and an SM holds many small CTAs: a CTA
// of four warps takes 64 columns x 4 blocks (128 rows), warp w block w and
// lane l columns 2l and 2l + 1.  A lane loads its 32 rows as 32-bit words (a
// warp's load is one 128-byte row segment), rounds both columns from those
// words with the scale and rounding of the row-wise bf16 path, and writes
// each column's codes of the block with one 32-byte (E4M3) or 16-byte (E2M1)
// store; the CTA's four warps together write whole 128- or 64-byte runs of
// each column.  The scale bytes meet in shared memory and leave as one 32-bit
// word per column (blocks 4 ry .. 4 ry + 3).
constexpr int kXD_Threads = 128;

// kP column pairs per lane (1: 32-bit loads; 2: 64-bit loads, cols % 4 == 0)
template <int FMT, int LAYOUT, int kP>
__global__ void __launch_bounds__(kXD_Threads, kP == 1 ? 8 : 5)
    quantize_axis0_direct_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols, int64_t nb,
                                 int64_t ncx, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
    constexpr int kOut = FMT == FMT_E2M1 ? 4 : 8;
    constexpr int kCols = 64 * kP;      // columns per CTA
    __shared__ uint32_t s_word[kCols];  // scale word of each of the CTA's columns, block w in byte w
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t ry = blockIdx.x / ncx, cx = blockIdx.x - ry * ncx;
    const int64_t blk = 4 * ry + warp;
    const int64_t c = kCols * cx + 2 * kP * lane;  // the lane's first column; cols % (2 kP) == 0
    pdl_wait();                                    // the previous kernel's writes are visible
    uint32_t sbytes[kP];                           // zero: padding past nb or cols
#pragma unroll
    for (int q = 0; q < kP; ++q) sbytes[q] = 0;
    if (blk < nb && c < cols) {
        const __nv_bfloat16* p = x + 32 * blk * cols + c;
        uint32_t w[kP][32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            if constexpr (kP == 1) {
                w[0][i] = __ldcs(reinterpret_cast<const unsigned int*>(p + i * cols));
            } else {
                const uint2 v = __ldcs(reinterpret_cast<const uint2*>(p + i * cols));
                w[0][i] = v.x;
                w[1][i] = v.y;
            }
        }
        const int64_t code_row = FMT == FMT_E2M1 ? rows / 2 : rows;
        uint8_t* dst = codes + c * code_row + (FMT == FMT_E2M1 ? 16 : 32) * blk;
#pragma unroll
        for (int q = 0; q < kP; ++q) {
            uint32_t out[2][kOut];
            sbytes[q] = quantize_column_pair_bf16<FMT>(w[q], out[0], out[1]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint8_t* d = dst + (2 * q + h) * code_row;
                if constexpr (FMT == FMT_E2M1) {
                    *reinterpret_cast<uint4*>(d) = make_uint4(out[h][0], out[h][1], out[h][2], out[h][3]);
                } else {
                    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(d), "r"(out[h][0]),
                                 "r"(out[h][1]), "r"(out[h][2]), "r"(out[h][3]), "r"(out[h][4]), "r"(out[h][5]),
                                 "r"(out[h][6]), "r"(out[h][7])
                                 : "memory");
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < kP; ++q) {
        reinterpret_cast<uint8_t*>(s_word)[(2 * kP * lane + 2 * q) * 4 + warp] = (uint8_t)sbytes[q];
        reinterpret_cast<uint8_t*>(s_word)[(2 * kP * lane + 2 * q + 1) * 4 + warp] = (uint8_t)(sbytes[q] >> 8);
    }
    __syncthreads();
    if (threadIdx.x < kCols) {
        const int64_t col = kCols * cx + threadIdx.x;
        const uint32_t word = s_word[threadIdx.x];
        if (LAYOUT == LAYOUT_MMA) {
            // the grid covers the layout's padding columns (to a multiple of 128)
            const int t = (int)(col & 127);
            uint32_t* tile = reinterpret_cast<uint32_t*>(scales + ((col >> 7) * (round_up(nb, 4) >> 2) + ry) * 512);
            tile[(t & 31) * 4 + (t >> 5)] = word;
        } else if (col < cols) {
            uint8_t* d = scales + col * nb + 4 * ry;
            const int nblk = (int)min((int64_t)4, nb - 4 * ry);
            if (nblk == 4 && (nb & 3) == 0) {
                *reinterpret_cast<uint32_t*>(d) = word;
            } else {
                for (int b = 0; b < nblk; ++b) d[b] = (uint8_t)(word >> (8 * b));
            }
        }
    }
}

template <int FMT, int kP>
cudaError_t run_axis0_direct(const __nv_bfloat16* x, int64_t rows, int64_t cols, uint8_t* codes, uint8_t* scales,
                             int layout, cudaStream_t st) {
    const int64_t nb = rows / 32;
    // the tensor-core layout's grid covers its padding columns, to a multiple of 128
    const int64_t ncx = layout == LAYOUT_MMA ? (128 / (64 * kP)) * ((cols + 127) / 128) : (cols + 64 * kP - 1) / (64 * kP);
    const int64_t ctas = ncx * ((nb + 3) / 4);
    if (ctas == 0) return cudaSuccess;
    const dim3 grid((unsigned)ctas), block(kXD_Threads);
    if (layout == LAYOUT_MMA)
        return launch_pdl(quantize_axis0_direct_kernel<FMT, LAYOUT_MMA, kP>, grid, block, 0, st, x, rows, cols, nb, ncx, codes, scales);
    return launch_pdl(quantize_axis0_direct_kernel<FMT, LAYOUT_ROWMAJOR, kP>, grid, block, 0, st, x, rows, cols, nb, ncx, codes, scales);
}

}  // namespace

bool quantize_axis0_direct_applies(const void* x, int dtype, int64_t cols, const void* codes) {
    return dtype != DT_F32 && (cols & 1) == 0 && (reinterpret_cast<uintptr_t>(x) & 3) == 0 &&
           (reinterpret_cast<uintptr_t>(codes) & 31) == 0;
}

cudaError_t launch_quantize_axis0_direct(const void* x, int64_t rows, int64_t cols, int fmt, void* codes,
                                         uint8_t* scales, int layout, cudaStream_t st) {
    const __nv_bfloat16* xp = static_cast<const __nv_bfloat16*>(x);
    uint8_t* cp = static_cast<uint8_t*>(codes);
    // 64-bit loads when every row starts on an 8-byte boundary
    const bool wide = (cols & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 7) == 0;
    if (fmt == FMT_E2M1)
        return wide ? run_axis0_direct<FMT_E2M1, 2>(xp, rows, cols, cp, scales, layout, st)
                    : run_axis0_direct<FMT_E2M1, 1>(xp, rows, cols, cp, scales, layout, st);
    return wide ? run_axis0_direct<FMT_E4M3, 2>(xp, rows, cols, cp, scales, layout, st)
                : run_axis0_direct<FMT_E4M3, 1>(xp, rows, cols, cp, scales, layout, st);
}

bool quantize_axis0_tiled_applies(const void* x, int dtype, int64_t cols) {
    const int64_t row_bytes = cols * (dtype == DT_F32 ? 4 : 2);
    return (reinterpret_cast<uintptr_t>(x) & 15) == 0 && row_bytes % 16 == 0 && device_error_word() != nullptr;
}

cudaError_t launch_quantize_axis0_tiled(const void* x, int dtype, int64_t rows, int64_t cols, int fmt, void* codes,
                                        uint8_t* scales, int layout, cudaStream_t st) {
    Axis0Params p{};
    p.rows = rows;
    p.cols = cols;
    p.nb = rows / 32;
    p.nb4 = round_up(p.nb, 4);
    p.nrg = (p.nb + kX_Blocks - 1) / kX_Blocks;
    p.total = (cols + kX_Cols - 1) / kX_Cols * p.nrg;
    p.scales = scales;
    p.wait_limit_ns = wait_limit_ns();
    p.err = device_error_word();
    const int esz = dtype == DT_F32 ? 4 : 2;
    CUtensorMap tx, tc;
    {
        const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
        const uint64_t strides[1] = {(uint64_t)cols * esz};
        const uint32_t box[2] = {(uint32_t)kX_Cols, (uint32_t)kX_Rows};
        if (!encode_tiled_map(&tx, dtype == DT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                              2, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    {
        // codes as bytes: [cols][code bytes per column]; a unit is a box of one
        // column tile x one run of codes
        const int64_t code_row = fmt == FMT_E2M1 ? rows / 2 : rows;
        const uint32_t run = fmt == FMT_E2M1 ? 16 * kX_Blocks : 32 * kX_Blocks;
        const uint64_t dims[2] = {(uint64_t)code_row, (uint64_t)cols};
        const uint64_t strides[1] = {(uint64_t)code_row};
        const uint32_t box[2] = {run, (uint32_t)kX_Cols};
        if (!encode_tiled_map(&tc, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, codes, dims, strides, box,
                              run == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
            return cudaErrorInvalidValue;
    }
    return dtype == DT_F32 ? axis0_dispatch<float>(tx, tc, p, fmt, layout, st)
                           : axis0_dispatch<__nv_bfloat16>(tx, tc, p, fmt, layout, st);
}

}  // namespace mx
