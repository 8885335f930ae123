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
// two 256-column boxes, issued by two lanes) per stage through a ring of
// stages, and decodes A's block for the step (16 rows x 32 codes, unscaled
// values, raw codes loaded two steps ahead) into the stage's slot; the stage
// is full when both the bytes and the decoded block have arrived.  Warps
// 1..8 compute and wait on nothing else, so they drift freely within the
// ring.  The block's scale is kept aside: a thread sums the 32 products of a
// block in f32 first and multiplies by the block's scale 2^(s-127) once
// (exact unless it leaves the binary32 range), folding the block sum into its
// running sum with one FMA.  That keeps the f32 rounding error of an output
// near (32 + number of blocks) units in the last place of sum |a*b| instead
// of K of them.
//
// Thread (warp w = 1..8, lane l): columns 4g..4g+3 of the tile with
// g = 32*((w-1) % 4) + l, rows 8*((w-1) / 4) .. +7; 32 sums and 32 block sums
// in registers, updated two rows at a time by packed f32x2 FMAs.  Per K row
// it reads one float4 of B (a warp reads 512 contiguous bytes: no bank
// conflicts) and two broadcast float4 of A.
//
// Measured on the decode shape (16 x 14336 x 4096, B 235 MB): the kernel
// runs within about 10% of the same pipeline with the arithmetic removed,
// i.e. it is bound by streaming B.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "mx_device.cuh"
#include "mx_internal.h"

namespace mx {
namespace {

constexpr int kF_Rows = 16;                                 // rows of C per tile
constexpr int kF_Cols = 512;                                // columns of C per tile
constexpr int kF_KStep = 32;                                // rows of B per stage (16: half an MX block)
constexpr int kF_Stages = 3;
constexpr int kF_CtasPerSm = 1;
constexpr int kF_RowGroups = 2;                             // the 16 rows are split over this many threads
constexpr int kF_Box = 256;                                 // columns per TMA box
constexpr int kF_Boxes = kF_Cols / kF_Box;
constexpr int kF_ColGroups = kF_Cols / 4;                   // a thread owns 4 columns
constexpr int kF_TM = kF_Rows / kF_RowGroups;               // rows per thread
constexpr int kF_Workers = kF_ColGroups * kF_RowGroups / 32;  // compute warps
constexpr int kF_Threads = 32 * (kF_Workers + 1);           // + the TMA warp
constexpr int kF_BoxBytes = kF_KStep * kF_Box * 4;
constexpr int kF_StageBytes = kF_Boxes * kF_BoxBytes;
constexpr int kF_OffA = kF_Stages * kF_StageBytes;                      // decoded A: [stage][k][16 rows] f32
constexpr int kF_OffS = kF_OffA + kF_Stages * kF_KStep * kF_Rows * 4;  // block scales: [stage][16] f32
constexpr int kF_OffBar = kF_OffS + kF_Stages * kF_Rows * 4;
constexpr int kF_Smem = kF_OffBar + 2 * kF_Stages * 8 + 1024;          // + alignment slack
static_assert(kF_Cols % kF_Box == 0 && kF_Boxes <= 32 && (kF_KStep == 16 || kF_KStep == 32), "tile shape");
static_assert(kF_TM % 4 == 0, "rows per thread are read as float4");
static_assert(kF_Smem * kF_CtasPerSm <= 227 * 1024, "shared memory");

struct F32bParams {
    const uint8_t* a_codes;
    const uint8_t* a_scales;
    int64_t M, N, K;
    int64_t a_row_bytes;  // bytes of codes per row of A
    int64_t nb, nb4;      // blocks per row; rounded up to 4 (tensor-core scale layout)
    int a_layout;
    int MT, NT, KS;       // row tiles, column tiles, K steps
    int64_t total;        // MT * NT * KS units
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

// Packed pairs of f32 (low word = first): fma.rn.f32x2 / mul.rn.f32x2 do two
// IEEE binary32 operations per instruction, each rounded as fmaf / a * b are,
// which halves the instructions the compute warps issue.
__device__ __forceinline__ unsigned long long pk2(float lo, float hi) {
    unsigned long long d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ void unpk2(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

struct Unit {
    int ks, mt, nt;  // K step, row tile, column tile
    __device__ __forceinline__ void next(const F32bParams& p) {
        if (++ks == p.KS) {
            ks = 0;
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
    w.ks = (int)(u % p.KS);
    const int64_t t = u / p.KS;
    w.mt = (int)(t % p.MT);
    w.nt = (int)(t / p.MT);
    return w;
}

// One lane's share of A for a K step: row (lane & 15) of the row tile, codes
// h*KStep/2 .. (h+1)*KStep/2 - 1 of the step with h = lane >> 4 (one load of
// 4 to 16 bytes), and the scale byte of the step's block (lanes 0..15).  Rows
// past M read as zero codes.
struct ARaw {
    uint4 c;
    uint32_t s;
};

template <int FMT>
__device__ __forceinline__ ARaw load_a_raw(const F32bParams& p, const Unit& w, int lane) {
    constexpr int kBytes = (FMT == FMT_E4M3 ? kF_KStep : kF_KStep / 2) / 2;  // code bytes per lane
    ARaw r{make_uint4(0, 0, 0, 0), 127};
    const int64_t row = (int64_t)w.mt * kF_Rows + (lane & 15);
    const int h = lane >> 4;
    if (row < p.M) {
        const uint8_t* src = p.a_codes + row * p.a_row_bytes + ((int64_t)w.ks * 2 + h) * kBytes;
        if constexpr (kBytes == 16) {
            r.c = __ldg(reinterpret_cast<const uint4*>(src));
        } else if constexpr (kBytes == 8) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
            r.c.x = v.x;
            r.c.y = v.y;
        } else {
            r.c.x = __ldg(reinterpret_cast<const uint32_t*>(src));
        }
        if (h == 0) {
            const int64_t kb = (int64_t)w.ks * kF_KStep / 32;
            r.s = __ldg(p.a_scales + (p.a_layout == LAYOUT_MMA ? mma_scale_offset(row, kb, p.nb4) : row * p.nb + kb));
        }
    }
    return r;
}

// The lane's codes as exact values into dec[k][row] (k-major), and its scale.
template <int FMT>
__device__ __forceinline__ void store_a(const ARaw& r, int lane, float* dec, float* scl) {
    const int row = lane & 15, k0 = (lane >> 4) * (kF_KStep / 2);
    const uint32_t wv[4] = {r.c.x, r.c.y, r.c.z, r.c.w};
#pragma unroll
    for (int i = 0; i < kF_KStep / 4; ++i) {
        // pair i: elements k0 + 2i, k0 + 2i + 1
        const float2 v = FMT == FMT_E4M3 ? decode2_e4m3(wv[i >> 1] >> (16 * (i & 1)))
                                         : decode2_e2m1(wv[i >> 2] >> (8 * (i & 3)));
        dec[(k0 + 2 * i) * kF_Rows + row] = v.x;
        dec[(k0 + 2 * i + 1) * kF_Rows + row] = v.y;
    }
    if (lane < 16) scl[row] = block_scale(r.s);
}

template <int FMT>
__global__ void __launch_bounds__(kF_Threads, kF_CtasPerSm) gemm_f32b_kernel(const __grid_constant__ CUtensorMap tm_b,
                                                                  const F32bParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // aligned by an offset from the array itself, so that the compiler keeps
    // the accesses below as shared-memory loads and stores
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    float* a_dec = reinterpret_cast<float*>(smem + kF_OffA);
    float* a_scl = reinterpret_cast<float*>(smem + kF_OffS);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kF_OffBar);
    uint64_t* empty = full + kF_Stages;

    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t u0 = p.total * blockIdx.x / gridDim.x, u1 = p.total * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_b);
        for (int s = 0; s < kF_Stages; ++s) {
            mbar_init(&full[s], 2);  // the TMA issue (with its bytes) and the decoded A
            mbar_init(&empty[s], kF_Workers);
        }
        fence_mbarrier_init();
    }
    __syncthreads();
    pdl_wait();  // set-up above overlaps the previous kernel's tail
    if (u0 >= u1) return;

    if (warp == 0) {
        // ------------------------------------------------ TMA and A decoding
        // Per stage: lane 0 issues B's loads; then the warp decodes A's block
        // into the stage's slot (raw codes loaded two steps ahead) and lane 0
        // arrives a second time.
        Unit w = unit_at(p, u0), w1 = w, w2 = w;
        w1.next(p);
        w2 = w1;
        w2.next(p);
        ARaw r0 = load_a_raw<FMT>(p, w, lane), r1{};
        if (u0 + 1 < u1) r1 = load_a_raw<FMT>(p, w1, lane);
        int64_t i = 0;
        for (int64_t u = u0; u < u1; ++u, ++i) {
            const int stage = (int)(i % kF_Stages);
            const uint32_t phase = (uint32_t)(i / kF_Stages) & 1u;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1u, p.wait_limit_ns, p.err);
            if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;  // the compute warps time out on `full`
            {
                // lane b loads box b (columns x + 256b ..); boxes wholly past N are not loaded
                const int32_t x = w.nt * kF_Cols, y = w.ks * kF_KStep;
                const int64_t left = p.N - x;
                const int nbox = left >= kF_Cols ? kF_Boxes : (int)((left + kF_Box - 1) / kF_Box);
                if (lane == 0) mbar_arrive_expect_tx(&full[stage], (uint32_t)(nbox * kF_BoxBytes));
                __syncwarp();
                if (lane < nbox)
                    tma_load_2d(smem + stage * kF_StageBytes + lane * kF_BoxBytes, &tm_b, x + lane * kF_Box, y,
                                &full[stage]);
            }
            store_a<FMT>(r0, lane, a_dec + stage * (kF_KStep * kF_Rows), a_scl + stage * kF_Rows);
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[stage]);
            r0 = r1;
            if (u + 2 < u1) r1 = load_a_raw<FMT>(p, w2, lane);
            w = w1;
            w1 = w2;
            w2.next(p);
        }
        // every issued copy has landed before the CTA exits (normally long
        // since: the compute warps waited for each of them)
        if (lane == 0) {
            const int64_t n = i;
            for (int64_t q = n > kF_Stages ? n - kF_Stages : 0; q < n; ++q)
                if (!mbar_wait(&full[q % kF_Stages], (uint32_t)(q / kF_Stages) & 1u, p.wait_limit_ns, p.err)) break;
        }
        return;
    }

    // -------------------------------------------------------------- compute
    const int t = threadIdx.x - 32;
    const int g = t % kF_ColGroups;         // column group: columns 4g .. 4g+3 of the tile
    const int rg = t / kF_ColGroups;        // row group: rows kF_TM*rg ..
    const uint32_t b_off = (uint32_t)((g >> 6) * kF_BoxBytes + (g & 63) * 16);

    float acc[kF_TM][4];
#pragma unroll
    for (int r = 0; r < kF_TM; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;

    Unit w = unit_at(p, u0);
    bool live = true;  // false after a timed-out wait: the remaining units are skipped
    int64_t i = 0;
    for (int64_t u = u0; u < u1; ++u, ++i) {
        const int stage = (int)(i % kF_Stages);
        const uint32_t phase = (uint32_t)(i / kF_Stages) & 1u;
        Unit nx = w;
        nx.next(p);
        if (live) live = mbar_wait(&full[stage], phase, p.wait_limit_ns, p.err);
        if (live) {
            const uint8_t* bs = smem + stage * kF_StageBytes + b_off;
            const float* as = a_dec + stage * (kF_KStep * kF_Rows) + rg * kF_TM;
            // packed pairs of rows (r, r+1): two f32 lanes per fma.rn.f32x2
            unsigned long long blk2[kF_TM / 2][4];
            float4 bn = *reinterpret_cast<const float4*>(bs);
            float4 an[kF_TM / 4];
#pragma unroll
            for (int r = 0; r < kF_TM / 4; ++r) an[r] = *reinterpret_cast<const float4*>(as + 4 * r);
#pragma unroll
            for (int k = 0; k < kF_KStep; ++k) {
                const float4 b = bn;
                unsigned long long ap[kF_TM / 2], bd[4];
#pragma unroll
                for (int r = 0; r < kF_TM / 4; ++r) {
                    ap[2 * r] = pk2(an[r].x, an[r].y);
                    ap[2 * r + 1] = pk2(an[r].z, an[r].w);
                }
                bd[0] = pk2(b.x, b.x);
                bd[1] = pk2(b.y, b.y);
                bd[2] = pk2(b.z, b.z);
                bd[3] = pk2(b.w, b.w);
                if (k + 1 < kF_KStep) {
                    bn = *reinterpret_cast<const float4*>(bs + (k + 1) * (kF_Box * 4));
#pragma unroll
                    for (int r = 0; r < kF_TM / 4; ++r)
                        an[r] = *reinterpret_cast<const float4*>(as + (k + 1) * kF_Rows + 4 * r);
                }
#pragma unroll
                for (int r = 0; r < kF_TM / 2; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) blk2[r][c] = k == 0 ? mul2(ap[r], bd[c]) : fma2(ap[r], bd[c], blk2[r][c]);
            }
            unsigned long long sc2[kF_TM / 2];
#pragma unroll
            for (int r = 0; r < kF_TM / 2; ++r)
                sc2[r] = pk2(a_scl[stage * kF_Rows + rg * kF_TM + 2 * r], a_scl[stage * kF_Rows + rg * kF_TM + 2 * r + 1]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);  // B stage and A slot both read
#pragma unroll
            for (int r = 0; r < kF_TM / 2; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    unsigned long long a2 = pk2(acc[2 * r][c], acc[2 * r + 1][c]);
                    a2 = fma2(blk2[r][c], sc2[r], a2);
                    unpk2(a2, acc[2 * r][c], acc[2 * r + 1][c]);
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
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), kF_Smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kF_Threads), kF_Smem, st, tm, p);
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
    p.KS = (int)(a.K / kF_KStep);
    p.total = (int64_t)p.MT * p.NT * p.KS;
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
    const uint32_t box[2] = {(uint32_t)kF_Box, (uint32_t)kF_KStep};
    if (!encode_tiled_map(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.B, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_NONE)) {
        *detail = "cuTensorMapEncodeTiled rejected B";
        return cudaErrorInvalidValue;
    }
    const int64_t slots = (int64_t)kF_CtasPerSm * sm_count();
    const int grid = (int)(p.total < slots ? p.total : slots);
    return a.a_fmt == FMT_E2M1 ? run_f32b<FMT_E2M1>(tm, p, grid, stream) : run_f32b<FMT_E4M3>(tm, p, grid, stream);
}

}  // namespace mx
