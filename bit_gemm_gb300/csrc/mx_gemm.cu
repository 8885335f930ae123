// mx_gemm.cu -- block_matmul on the sm_103a tensor cores (tcgen05, TMEM, TMA).
//
// block_matmul of "A Dialect Is a Set of Co-Designed Decisions: Designing for
// MX Quantization in MLIR" ("The four ops", "The block axis", "The
// accumulator operand"):  C <- C + A * B with A [M,K] and B given as Bt [N,K],
// both blocked along the reduction axis K, so each block's two E8M0 scales
// factor out of its partial sum -- exactly what the block-scaled MMA does in
// hardware (kind::mxf8f6f4: K = 32 per instruction, one scale per row;
// kind::mxf4: K = 64 per instruction, two scales per row).
//
// Two kernels, both persistent (one CTA, or one CTA pair, per SM or SM pair):
//   gemm_kernel       one CTA per 128 x BN tile: M or N <= 128, row-major
//                     scales, and the swapped decode shapes;
//   gemm_pair_kernel  256 x 256 tiles on a CTA pair (tcgen05 .cta_group::2).
// Roles in a CTA:
//   warp 0      TMA producer: A/B code tiles (128-byte swizzled, K-major) and
//               the 512-byte scale tiles into a STAGES-deep shared-memory ring.
//   warp 1      allocates TMEM; one lane copies the scale tiles to TMEM
//               (tcgen05.cp) and issues the MMAs into an f32 TMEM accumulator
//               (decode shapes: a second MMA warp takes every stage's second
//               K atom into a second accumulator).
//   gate warp   waits on each stage's barrier and passes it to the MMA warp(s)
//               through a named barrier, so the issuing thread never touches
//               shared memory between MMAs.
//   act warps   (decode shapes with bf16 activations quantized in the kernel)
//               quantize each stage's activations into the ring's B slot.
//   epilogue    4 or 8 warps: TMEM -> registers -> swizzled shared staging ->
//               TMA reduce-add into C (C += acc, performed at L2), so C is read
//               and written in place with no extra pass.
// The work schedule (whole tiles, or equal slices of the (tile, K stage)
// space, whose partial sums meet in C through the same reduce-add) is in
// mx_schedule.h.  For M <= 64 the operands are swapped (C^T = Bt * A^T) so the
// long N side fills the 128-row MMA dimension.
//
// Every mbarrier wait is bounded (see mx_device.cuh); a CTA that gives up sets
// the device error word, drains what it issued, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "mx_device.cuh"
#include "mx_internal.h"
#include "mx_quant_block.cuh"
#include "mx_schedule.h"

namespace mx {

__device__ unsigned int g_mx_device_error = 0;

cudaError_t read_clear_device_error(unsigned* out, cudaStream_t st) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_mx_device_error, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return e;
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return e;
    if (*out) {
        const unsigned zero = 0;
        e = cudaMemcpyToSymbolAsync(g_mx_device_error, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    return e;
}

namespace {

constexpr int KIND_F8F6F4 = 0;  // kind::mxf8f6f4 (E4M3 x E4M3, mixed E4M3 / E2M1)
constexpr int KIND_F4 = 1;      // kind::mxf4     (E2M1 x E2M1, packed)

constexpr int kBlockM = 128;
constexpr int kRowBytes = 128;        // bytes of K per tile row per stage (one 128-B swizzle atom)
constexpr int kMmaPerStage = 4;       // 4 MMAs of 32 bytes of K each
constexpr int kAccCol = 0;            // accumulator buffers at columns [0, ACC * BN)
constexpr uint32_t kTmemCols = 512;
constexpr int kActStreamed = -1;      // ACT_ATOMS value: activations quantized stage by stage

struct GemmParams {
    int32_t P, Q, K;       // rows of the MMA A operand, rows of the MMA B operand, reduction length
    int32_t tiles_p, tiles_q;
    int32_t k_stages;      // stages of 128 bytes of K
    int32_t sf_groups;     // 4-block scale groups per 128-row scale tile (NB4 / 4)
    int32_t mode;          // 0 = whole tiles round-robin, 1 = equal slices of (tile, stage),
                           // 2 = whole tiles for the full rounds, the remaining tiles as in 1
    int64_t total_units;   // tiles * k_stages
    uint64_t wait_limit_ns;
    uint32_t idesc;        // instruction descriptor without scale-factor ids
    int32_t swap;          // 1: C(q, p) += acc(p, q)  (operands swapped)
    int32_t use_tma_epi;   // 1: C map valid (TMA reduce-add epilogue), 0: per-element atomics
    int32_t epi_red_v4;    // 1: write C with vector reductions instead of TMA (BN = 256 path)
    float* C;
    int64_t ldc;
    const uint8_t* sfa;    // scales of the MMA A operand (tensor-core layout)
    const uint8_t* sfb;    // scales of the MMA B operand
    uint32_t tx_a, tx_b;   // bytes one stage's code load counts on its barrier
    int32_t sf_rowmajor;   // 1: scales are row-major [rows][K/32]; gathered by the producer lanes
    int32_t nb;            // K / 32 (row stride of row-major scales, a multiple of 4)
    int32_t group_p;       // whole-tile order: bands of this many row tiles sweep all column tiles
    int32_t op3d;          // 1: operand maps are 3-D [atoms][rows][128 B] (K a whole number of stages)
    int32_t k_atom0;       // first stage of K this launch covers (K split into launches)
    // activations quantized in the kernel (MMA B operand, swapped shapes):
    const void* act;       // [Q][act_ld] f32 or bf16, row-major
    int64_t act_ld;        // elements per activation row
    int32_t act_bf16;      // 1: bf16, 0: f32
};

// Waits that end a launch after an abort -- for loads and MMAs already
// issued, which always complete -- use at least this limit, whatever limit
// the caller set for the waits that can give up.
constexpr uint64_t kDrainLimitNs = 1000000000ull;

// Named barrier `id` over `count` threads that also ORs a predicate across
// them: returns whether any participant passed true (no shared-memory access).
__device__ __forceinline__ bool named_bar_red_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Count `bytes` as arrived on the current phase of a barrier of this CTA.
__device__ __forceinline__ void mbar_complete_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// A 32-bit store into the shared memory of another CTA of the cluster.
__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

template <int KIND, int BN, int STAGES, int SWAP, int NBUF_ = 0, int ACT_ATOMS = 0, int SA = 1>
struct Cfg {
    // SA: K atoms (128 bytes of K per operand row) per pipeline stage; a stage
    // of SA atoms is loaded with one 3-D box per operand and scale tensor, so
    // per-stage costs (barrier round trips, load issue) are paid once per SA
    // atoms.  SA > 1 needs K a whole number of stages and tensor-core scales.
    // ACT_ATOMS > 0: the activations (the MMA B operand of a swapped shape) are
    // quantized by the kernel into a resident region of that many K stages.
    // ACT_ATOMS == kActStreamed: they are quantized stage by stage into the
    // ring's B slots by ACT_WARPS warps of their own, as the weights stream.
    static constexpr bool ACT = ACT_ATOMS > 0;
    static constexpr bool SACT = ACT_ATOMS == kActStreamed;
    static constexpr int G = KIND == KIND_F4 ? 2 : 1;                 // scale groups per atom
    static constexpr int GS = SA * G;                                  // scale groups per stage
    // 128-row scale tiles covering the BN rows of a B tile (tiles start on
    // 128-row boundaries: scale-factor TMEM addresses must stay aligned)
    static constexpr int SFB_TILES = (BN + 127) / 128;
    // TMEM accumulator buffers: two 128-column buffers for BN = 128; for BN = 256
    // the single buffer is drained into the registers of eight epilogue warps
    // (two per TMEM lane quarter, 128 columns each) and released at once, so
    // the next tile's MMAs overlap the write-out of this one
    static constexpr int ACC = (!SWAP && 2 * BN <= 256) ? 2 : 1;
    static constexpr int EPI_WARPS = (!SWAP && BN == 256) ? 8 : 4;
    static constexpr int GATE_WARP = 2 + EPI_WARPS;  // waits on stage barriers for the MMA warp(s)
    // MMA-issuing warps: with several atoms per stage (decode shapes, where one
    // thread's issue rate sets the pace) each of MW warps takes SA / MW atoms
    // of every stage into its own accumulator; the epilogue adds them.  Warp 1
    // and, for MW = 2, the warp after the gate.
    static constexpr int MW = (SWAP && SA == 2) ? 2 : 1;
    static constexpr int PRO_WARPS = GATE_WARP + MW - 1;  // warps 1.. that quantize resident activations
    static constexpr int ACT_WARP0 = GATE_WARP + MW;      // streamed activations: the last ACT_WARPS warps
    static constexpr int ACT_WARPS = SACT ? 4 : 0;
    static constexpr int THREADS = 32 * (GATE_WARP + MW + ACT_WARPS);
    static constexpr int A_ATOM = kBlockM * kRowBytes;                // 16 KB
    static constexpr int B_ATOM = BN * kRowBytes;
    static constexpr int A_BYTES = SA * A_ATOM;
    static constexpr int B_BYTES = ACT ? 0 : SA * B_ATOM;
    static constexpr int SFA_BYTES = GS * 512;
    static constexpr int SFB_BYTES = ACT ? 0 : GS * SFB_TILES * 512;
    // full scale boxes of a stage that TMA loads (streamed activations: A's only)
    static constexpr uint32_t SF_TX = (uint32_t)(SFA_BYTES + (SACT ? 0 : SFB_BYTES));
    static constexpr int ACT_BYTES = BN * kRowBytes;  // one resident K stage of the activations
    static constexpr int ACT_SF_BYTES = G * 512;
    static constexpr int SF_COLS_A = 4 * GS;
    static constexpr int SF_COLS_B = 4 * GS * SFB_TILES;
    static constexpr int SF_COLS_STAGE = SF_COLS_A + SF_COLS_B;
    static constexpr int SF_COL0 = ACC * BN > 256 ? ACC * BN : 256;   // first scale column
    // scale slots in TMEM; a slot is rewritten by tcgen05.cp only after the
    // MMAs that read it were issued (tcgen05 operations of one thread execute
    // in issue order)
    static constexpr int SF_SLOTS_FIT = ((int)kTmemCols - SF_COL0) / SF_COLS_STAGE;
    static constexpr int SF_SLOTS = SF_SLOTS_FIT < STAGES ? SF_SLOTS_FIT : STAGES;
    // epilogue staging per warp: NBUF buffers of 32 rows x 32 f32 (non-swapped)
    // or BN rows x 32 f32 (swapped)
    static constexpr int NBUF = NBUF_ ? NBUF_ : (EPI_WARPS == 8 ? 1 : 2);
    static constexpr int EPI_COLS = SWAP ? 32 : (EPI_WARPS == 8 ? 16 : 32);   // C columns per staged box
    static constexpr int EPI_BUF = SWAP ? BN * 32 * 4 : 32 * EPI_COLS * 4;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_ACT = (OFF_SFB + STAGES * SFB_BYTES + 1023) / 1024 * 1024;
    static constexpr int RES_ATOMS = ACT ? ACT_ATOMS : 0;  // resident activation stages
    static constexpr int OFF_ACT_SF = OFF_ACT + RES_ATOMS * ACT_BYTES;
    static constexpr int OFF_EPI = (OFF_ACT_SF + RES_ATOMS * ACT_SF_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * NBUF * EPI_BUF;
    static constexpr int BAR_BYTES = (2 * STAGES + 2 * ACC + 1) * 8 + 16;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;           // + alignment slack
    static_assert(!ACT || (SWAP && ACT_BYTES % 1024 == 0), "resident activations: swapped shapes, whole swizzle atoms");
    static_assert(STAGES <= (ACT ? 14 : 15), "named barriers 1..STAGES (and 15 for the activation prologue)");
    static_assert(SF_SLOTS >= 2, "at least two scale slots in TMEM");
    static_assert(SF_COL0 + SF_SLOTS * SF_COLS_STAGE <= (int)kTmemCols, "TMEM columns");
    static_assert(ACC * MW * BN <= SF_COL0, "accumulator columns");
    static_assert(SA % MW == 0, "whole atoms per MMA warp");
    static_assert(!SACT || (SWAP && BN == 16), "streamed activations: swapped shapes, up to 16 rows");
    // An activation warp waits for fill n's slot by the parity of the slot's
    // empty barrier, which is unambiguous only while the barrier is at most
    // one phase behind: its previous wait (fill n - ACT_WARPS) guarantees fill
    // n - ACT_WARPS - STAGES was consumed, and fill n needs n - 2 STAGES, so
    // ACT_WARPS may not exceed STAGES.
    static_assert(ACT_WARPS <= STAGES, "activation warps at most one ring phase ahead");
    static_assert(32 * (PRO_WARPS + 1) <= THREADS, "warps 1..PRO_WARPS exist");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(SWAP || BN % 128 == 0, "B tiles start on 128-row boundaries");
    static_assert(SMEM <= 232448, "shared memory per CTA");
    static_assert(STAGES <= 15, "one named barrier per stage");
    static_assert(SA == 1 || SWAP, "several atoms per stage: swapped (decode) shapes");
};

// Write 32 rows x 128 columns of accumulator (this warp's lane quarter, in
// registers: r[c][j] = column 32c + j of row p0 + lane) into C at (p0, qc):
// TMA reduce-add of 32 x 16 boxes through one 2 KB 64-byte-swizzled staging
// buffer per warp, or vector / scalar reductions.  Columns past N and rows past
// M are clipped.
// EC: columns per TMA box, 16 (64-byte swizzled rows, 2 KB per warp) or 8
// (unswizzled 32-byte rows, 1 KB per warp, for kernels short of shared memory).
template <int EC = 16>
__device__ __forceinline__ void epilogue_write_128(const GemmParams& p, const CUtensorMap& tm_c, const uint32_t (&r)[4][32],
                                                   int32_t p0, int32_t qc, uint8_t* stage_buf, int& nbuf, int lane) {
    static_assert(EC == 16 || EC == 8, "epilogue box columns");
    const int32_t pr = p0 + lane;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (qc + 32 * c >= p.Q) break;
        if (p.epi_red_v4) {
            if (pr < p.P) {
                float* row = p.C + (int64_t)pr * p.ldc + qc + 32 * c;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (qc + 32 * c + 4 * j + 3 < p.Q) {
                        red_add_v4(row + 4 * j, __uint_as_float(r[c][4 * j]), __uint_as_float(r[c][4 * j + 1]),
                                   __uint_as_float(r[c][4 * j + 2]), __uint_as_float(r[c][4 * j + 3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (qc + 32 * c + 4 * j + e < p.Q) atomicAdd(row + 4 * j + e, __uint_as_float(r[c][4 * j + e]));
                    }
                }
            }
        } else if (p.use_tma_epi) {
#pragma unroll
            for (int hh = 0; hh < 32 / EC; ++hh) {
                if (qc + 32 * c + EC * hh >= p.Q) break;
                uint8_t* buf = stage_buf;  // one 32 x EC buffer per warp
                if (nbuf >= 1 && lane == 0) bulk_wait_group_read<0>();
                __syncwarp();
                if constexpr (EC == 16) {
                    // [32 rows][16 f32], 64-byte swizzle: 16-B chunk j of row i at j ^ ((i >> 1) & 3)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int js = j ^ ((lane >> 1) & 3);
                        const uint32_t* v = &r[c][16 * hh + 4 * j];
                        *reinterpret_cast<uint4*>(buf + lane * 64 + js * 16) = make_uint4(v[0], v[1], v[2], v[3]);
                    }
                } else {
                    // [32 rows][8 f32], no swizzle
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t* v = &r[c][8 * hh + 4 * j];
                        *reinterpret_cast<uint4*>(buf + lane * 32 + j * 16) = make_uint4(v[0], v[1], v[2], v[3]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_reduce_add_2d(&tm_c, buf, qc + 32 * c + EC * hh, p0);
                    bulk_commit_group();
                }
                ++nbuf;
            }
        } else if (pr < p.P) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (qc + 32 * c + j < p.Q) atomicAdd(p.C + (int64_t)pr * p.ldc + qc + 32 * c + j, __uint_as_float(r[c][j]));
        }
    }
}

template <int KIND, int BN, int STAGES, int SWAP, int NBUF_, int ACT_ATOMS = 0, int SA = 1>
__global__ void __launch_bounds__(Cfg<KIND, BN, STAGES, SWAP, NBUF_, ACT_ATOMS, SA>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                const __grid_constant__ CUtensorMap tm_c, const GemmParams p) {
    using C_ = Cfg<KIND, BN, STAGES, SWAP, NBUF_, ACT_ATOMS, SA>;
    constexpr int ACC = C_::ACC;
    extern __shared__ uint8_t smem_raw[];
    // aligned by an offset from the array itself: the compiler then keeps the
    // generic accesses below (epilogue staging, activation tiles) in the shared window
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C_::OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* tmem_full = empty + STAGES;   // [ACC]
    uint64_t* tmem_empty = tmem_full + ACC;  // [ACC]
    uint64_t* mma_done = tmem_empty + ACC;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    unsigned* err = &g_mx_device_error;
    // fills the producer issued (fill n goes to slot n % STAGES), for the
    // drain after the CTA's final barrier
    int n_issued = 0;
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // row-major scales: the 32 producer lanes' cp.async arrivals as well
            // + the activation warp that fills the stage's B slot, when streamed
            mbar_init(&full[s], p.sf_rowmajor ? 33 : (C_::SACT ? 2 : 1));
            mbar_init(&empty[s], C_::MW);  // one commit per MMA warp
        }
        for (int a = 0; a < ACC; ++a) {
            mbar_init(&tmem_full[a], C_::MW);
            mbar_init(&tmem_empty[a], C_::EPI_WARPS);
        }
        mbar_init(mma_done, C_::MW);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_a);
        if (!C_::ACT && !C_::SACT) prefetch_tensormap(&tm_b);  // activations quantized here: no B map
        if (!p.sf_rowmajor) {
            prefetch_tensormap(&tm_sfa);
            if (!C_::ACT && !C_::SACT) prefetch_tensormap(&tm_sfb);
        }
        if (p.use_tma_epi) prefetch_tensormap(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // The first two work units, computed before the wait (the integer
    // divisions of the schedule take a few hundred ns of one warp's time,
    // which then overlap the previous kernel's tail instead of delaying the
    // first load and the MMA warps' first tile change).
    Work wl0, wl1;
    const bool hl0 = get_work(p, blockIdx.x, gridDim.x, 0, wl0);
    const bool hl1 = hl0 && get_work(p, blockIdx.x, gridDim.x, 1, wl1);
    auto work_at = [&](int it, Work& w) -> bool {
        if (it == 0) {
            w = wl0;
            return hl0;
        }
        if (it == 1) {
            w = wl1;
            return hl1;
        }
        return get_work(p, blockIdx.x, gridDim.x, it, w);
    };
    // set-up above overlaps the previous kernel's tail; global memory from here on
    pdl_wait();

    // K stages this CTA touches (the hull of its work units), for the
    // resident activations
    int kb_lo = 0x7FFFFFFF, kb_hi = 0;
    if constexpr (C_::ACT) {
        Work w;
        for (int it = 0; work_at(it, w); ++it) {
            kb_lo = min(kb_lo, w.kb0);
            kb_hi = max(kb_hi, w.kb1);
        }
        if (kb_hi <= kb_lo) kb_lo = kb_hi = 0;
        if (warp >= 1 && warp <= C_::PRO_WARPS) {
            // ------------------------------------------------ activation prologue
            // The warps that are idle while the producer starts streaming the
            // weights quantize this CTA's K stages of the activations once, with
            // mx_quantize's rounding, into the MMA operand layout: per stage, BN
            // rows of 128 bytes with the 128-byte swizzle, and the scale tile(s).
            // Rows past M and elements past K become zero codes.
            constexpr int BPA = KIND == KIND_F4 ? 8 : 4;  // 32-element blocks per atom
            constexpr int AFMT = KIND == KIND_F4 ? FMT_E2M1 : FMT_E4M3;
            const int nthr = 32 * C_::PRO_WARPS;
            const int64_t items = (int64_t)SA * (kb_hi - kb_lo) * BN * BPA;
            // block i: atom a (of the CTA's range), row r, block j of the atom; its first element k
            auto item = [&](int64_t i, int& a, int& r, int& j, int64_t& k) {
                j = (int)(i % BPA);
                r = (int)((i / BPA) % BN);
                a = (int)(i / (BPA * BN));
                k = (((int64_t)SA * (p.k_atom0 + kb_lo) + a) * BPA + j) * 32;
            };
            auto emit = [&](const uint32_t (&u)[32], bool bf16, int a, int r, int j) {
                uint32_t out[AFMT == FMT_E2M1 ? 4 : 8];
                const uint32_t sbyte = quantize_column_block<AFMT>(u, bf16, out);
                uint8_t* rowp = smem + C_::OFF_ACT + a * C_::ACT_BYTES + r * kRowBytes;
                if constexpr (AFMT == FMT_E4M3) {  // a block is 32 bytes: chunks 2j, 2j+1
                    *reinterpret_cast<uint4*>(rowp + (((2 * j) ^ (r & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
                    *reinterpret_cast<uint4*>(rowp + (((2 * j + 1) ^ (r & 7)) << 4)) = make_uint4(out[4], out[5], out[6], out[7]);
                } else {  // packed E2M1: a block is 16 bytes, chunk j
                    *reinterpret_cast<uint4*>(rowp + ((j ^ (r & 7)) << 4)) = make_uint4(out[0], out[1], out[2], out[3]);
                }
                smem[C_::OFF_ACT_SF + (a * C_::G + j / 4) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (j & 3)] =
                    (uint8_t)sbyte;
            };
            // loads are issued a batch at a time before any of them is used, so
            // their latencies overlap
            if (p.act_bf16) {
                constexpr int kB = 4;
                const __nv_bfloat16* act = static_cast<const __nv_bfloat16*>(p.act);
                for (int64_t i0 = threadIdx.x - 32; i0 < items; i0 += (int64_t)nthr * kB) {
                    uint32_t w16[kB][16];
#pragma unroll
                    for (int q = 0; q < kB; ++q) {
                        int a, r, j;
                        int64_t k;
                        const int64_t i = i0 + (int64_t)q * nthr;
                        item(i, a, r, j, k);
                        if (i < items && r < p.Q && k < p.K) {
                            load_block_bf16(act + (int64_t)r * p.act_ld + k, w16[q]);
                        } else {
#pragma unroll
                            for (int t = 0; t < 16; ++t) w16[q][t] = 0;
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kB; ++q) {
                        int a, r, j;
                        int64_t k;
                        const int64_t i = i0 + (int64_t)q * nthr;
                        if (i >= items) break;
                        item(i, a, r, j, k);
                        uint32_t u[32];
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            u[2 * t] = w16[q][t] << 16;
                            u[2 * t + 1] = w16[q][t] & 0xFFFF0000u;
                        }
                        emit(u, true, a, r, j);
                    }
                }
            } else {
                constexpr int kB = 2;
                const float* act = static_cast<const float*>(p.act);
                for (int64_t i0 = threadIdx.x - 32; i0 < items; i0 += (int64_t)nthr * kB) {
                    uint32_t u[kB][32];
#pragma unroll
                    for (int q = 0; q < kB; ++q) {
                        int a, r, j;
                        int64_t k;
                        const int64_t i = i0 + (int64_t)q * nthr;
                        item(i, a, r, j, k);
                        if (i < items && r < p.Q && k < p.K) {
                            const uint4* src = reinterpret_cast<const uint4*>(act + (int64_t)r * p.act_ld + k);
#pragma unroll
                            for (int t = 0; t < 8; ++t) {
                                const uint4 v = __ldcs(src + t);
                                u[q][4 * t] = v.x;
                                u[q][4 * t + 1] = v.y;
                                u[q][4 * t + 2] = v.z;
                                u[q][4 * t + 3] = v.w;
                            }
                        } else {
#pragma unroll
                            for (int t = 0; t < 32; ++t) u[q][t] = 0;
                        }
                    }
#pragma unroll
                    for (int q = 0; q < kB; ++q) {
                        int a, r, j;
                        int64_t k;
                        const int64_t i = i0 + (int64_t)q * nthr;
                        if (i >= items) break;
                        item(i, a, r, j, k);
                        emit(u[q], false, a, r, j);
                    }
                }
            }
            fence_proxy_async_smem();  // generic writes, read by the tensor core
            __syncwarp();
            named_bar_sync(15, 32 * C_::PRO_WARPS);
        }
    }

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Lane 0 issues the TMA loads; with row-major scales every lane also
        // gathers 4-byte scale words of its rows straight into the tensor-core
        // tile layout (row r -> line r % 32, word (r / 32) % 4 of its tile).
        int stage = 0;
        uint32_t phase = 0;
        // load roles: 0 A, 1 B, 2 A's scales, 3 B's scales (resident activations: A and its scales only)
        constexpr bool kNoB = C_::ACT || C_::SACT;  // B is not loaded by TMA
        const int li = kNoB ? ((lane & 1) ? 2 : 0) : (lane & 3);
        const void* lmap = li == 0 ? (const void*)&tm_a : li == 1 ? (const void*)&tm_b
                                                    : li == 2 ? (const void*)&tm_sfa : (const void*)&tm_sfb;
        const uint32_t lbase = smem_u32(smem) + (li == 0 ? C_::OFF_A : li == 1 ? C_::OFF_B
                                                  : li == 2 ? C_::OFF_SFA : C_::OFF_SFB);
        const uint32_t lstep = li == 0 ? C_::A_BYTES : li == 1 ? C_::B_BYTES : li == 2 ? C_::SFA_BYTES : C_::SFB_BYTES;
        int fills = 0;
        // row-major scales: the lane's scale rows of the current tile, and their byte counts
        const uint8_t* rm_a[4];
        const uint8_t* rm_b[C_::SFB_TILES][4];
        uint32_t rm_na[4], rm_nb[C_::SFB_TILES][4];
        bool ok = true;
        Work w;
        for (int it = 0; ok && work_at(it, w); ++it) {
            const int32_t p0 = w.tp * kBlockM;
            const int32_t q0 = w.tq * BN;
            const int nk = w.kb1 - w.kb0;
            for (int j = 0; j < nk; ++j) {
                const int kb = w.kb0 + j;
                // (the abort flag is consulted only when a bounded wait gives up:
                // a shared-memory load and branch per stage would delay issue)
                int okw = 1;
                // (the first STAGES fills find their slots free: no wait).  The
                // slot's previous fill must also have landed: after the gate
                // gives up, the MMA warps may release a slot whose load is still
                // in flight, and a refill must not overlap it.  The parity is
                // unambiguous because every earlier fill of the slot was seen
                // landing here.  A fill lands before the MMAs release it, so
                // this wait comes first and ends while the release is still
                // pending: the refill is issued as soon as the release arrives.
                // (Not with streamed activations: there the MMA warps stop at
                // the stage the gate gave up on, so no slot is released before
                // its data has landed, and the check lengthened the decode step.)
                if (lane == 0 && fills >= STAGES)
                    okw = (C_::SACT || mbar_wait(&full[stage], phase ^ 1, p.wait_limit_ns, err)) &&
                          mbar_wait(&empty[stage], phase ^ 1, p.wait_limit_ns, err);
                ++fills;
                okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                if (!okw) {
                    if (lane == 0) *abort_flag = 1;
                    ok = false;
                    break;
                }
                // scale groups present for this stage (the last stage of a
                // ragged K may need only the first)
                const int g_first = (kb + p.k_atom0) * C_::GS;
                const int g_count = min(C_::GS, p.sf_groups - g_first);
                // A stage is A, B and (tensor-core scale layout) the scale boxes
                // of both, issued by lanes 0..3 with one instruction where the
                // operand maps are 3-D; boxes past the tensor's end read zeros
                // and count their full bytes.
                if (lane == 0)
                    mbar_arrive_expect_tx(&full[stage], p.tx_a + (kNoB ? 0u : p.tx_b) +
                                                            (p.sf_rowmajor ? 0u : C_::SF_TX));
                {
                    const int kbg = kb + p.k_atom0;  // stage of K in the whole tensor
                    const int nl = (kNoB || p.sf_rowmajor) ? 2 : 4;
                    const uint32_t dst = lbase + (uint32_t)stage * lstep;
                    const int32_t y = li == 0 ? p0 : li == 1 ? q0 : 4 * C_::GS * kbg;
                    const int32_t z = li < 2 ? SA * kbg : (li == 2 ? w.tp : q0 >> 7);
                    if (lane < nl) {
                        if (p.op3d || li >= 2) tma_load_3d_at(dst, lmap, 0, y, z, &full[stage]);
                        else tma_load_2d_at(dst, lmap, kbg * kRowBytes, y, &full[stage]);
                    }
                    __syncwarp();
                }
                if (p.sf_rowmajor) {
                    if (j == 0) {
                        // this lane's scale rows of the tile: A rows p0 + lane + 32 i, B rows
                        // q0 + 128 t + lane + 32 i (rows past the end read nothing, as zeros)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int32_t r = p0 + lane + 32 * i;
                            rm_a[i] = p.sfa + (int64_t)(r < p.P ? r : p.P - 1) * p.nb;
                            rm_na[i] = r < p.P ? 4u : 0u;
#pragma unroll
                            for (int t = 0; t < C_::SFB_TILES; ++t) {
                                const int32_t rb = q0 + 128 * t + lane + 32 * i;
                                rm_b[t][i] = p.sfb + (int64_t)(rb < p.Q ? rb : p.Q - 1) * p.nb;
                                rm_nb[t][i] = rb < p.Q ? 4u : 0u;
                            }
                        }
                    }
                    for (int g = 0; g < g_count; ++g) {
                        const int word = 4 * (g_first + g);  // byte offset of the group in a row
                        uint8_t* da = smem + C_::OFF_SFA + stage * C_::SFA_BYTES + g * 512 + lane * 16;
#pragma unroll
                        for (int i = 0; i < 4; ++i) cp_async_4(da + 4 * i, rm_a[i] + word, rm_na[i]);
#pragma unroll
                        for (int t = 0; t < C_::SFB_TILES; ++t) {
                            // group g of row tile t where the MMA side reads it
                            uint8_t* db = smem + C_::OFF_SFB + stage * C_::SFB_BYTES + (t * C_::GS + g) * 512 + lane * 16;
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                // the MMA reads the first BN rows of B's scale tiles only
                                if (128 * t + 32 * i < BN) cp_async_4(db + 4 * i, rm_b[t][i] + word, rm_nb[t][i]);
                            }
                        }
                    }
                    cp_async_arrive_noinc(&full[stage]);
                }
                ++n_issued;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // (loads still in flight after a give-up are awaited after the CTA's
        // final barrier)
    } else if (warp == 1 || (C_::MW > 1 && warp == C_::GATE_WARP + 1)) {
        // ---------------------------------------------------------- MMA issue
        // The whole warp walks the schedule and syncs on stage s's named
        // barrier (1 + s) with the gate warp, which has seen the stage's data
        // land; lane 0 issues.  MMA warp m (of MW) issues atoms
        // [m SA / MW, (m + 1) SA / MW) of every stage into accumulator m.  The
        // warp learns of an abort at its next tile (the abort flag, or its own
        // wait giving up); until then it may issue on stages the gate gave up
        // on.  After that it keeps walking (and syncing) without issuing, so
        // its syncs and the gate's always pair up.
        // Everything that does not depend on the stage is built once: the
        // shared-memory descriptors of stage 0 (a stage's descriptors differ
        // only in the start-address field, which is advanced by adds) and the
        // four instruction descriptors carrying the scale-factor ids.
        const uint64_t a_desc0 = smem_desc(smem_u32(smem + C_::OFF_A), 0, 1024, 2);
        const uint64_t b_desc0 = smem_desc(smem_u32(smem + (C_::ACT ? C_::OFF_ACT : C_::OFF_B)), 0, 1024, 2);
        const uint64_t sfa_desc0 = smem_desc(smem_u32(smem + C_::OFF_SFA), 0, 128, 0);
        const uint64_t sfb_desc0 = smem_desc(smem_u32(smem + (C_::ACT ? C_::OFF_ACT_SF : C_::OFF_SFB)), 0, 128, 0);
        uint32_t idesc[kMmaPerStage];
#pragma unroll
        for (int i = 0; i < kMmaPerStage; ++i) {
            // kind::mxf4: MMA i covers blocks 2i, 2i+1 of the stage (scale bytes
            // 0-1 or 2-3 of its group); kind::mxf8f6f4: block i (byte i)
            const uint32_t sf_id = KIND == KIND_F4 ? (uint32_t)(i & 1) * 2u : (uint32_t)i;
            idesc[i] = p.idesc | (sf_id << 4) | (sf_id << 29);
        }
        constexpr int k_elem_per_stage = SA * (KIND == KIND_F4 ? 256 : 128);
        constexpr int k_elem_per_mma = KIND == KIND_F4 ? 64 : 32;
        constexpr int AW = SA / C_::MW;  // atoms per MMA warp
        const int m = warp == 1 ? 0 : 1;
        const int a_first = m * AW;
        int stage = 0;
        int sf_slot = 0;
        bool live = true;  // false after an abort: walk without issuing
        Work w;
        for (int it = 0; work_at(it, w); ++it) {
            const int acc = it % ACC;
            const uint32_t acc_phase = (uint32_t)(it / ACC) & 1u;
            int okt = 1;
            if (lane == 0 && live)
                okt = !*abort_flag && mbar_wait(&tmem_empty[acc], acc_phase ^ 1, p.wait_limit_ns, err);
            okt = __shfl_sync(0xFFFFFFFFu, okt, 0);
            if (live && !okt) {
                live = false;
                if (lane == 0) *abort_flag = 1;
            }
            const uint32_t d_tmem = tmem + kAccCol + (acc * C_::MW + m) * BN;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                // the gate saw this stage's data land, or gave up waiting for it
                // (the MMAs then read whatever the slot holds: the launch has
                // reported its timeout, and the producer refills no slot whose
                // load is in flight).  With streamed activations the warps stop
                // at that stage instead: releasing later slots would let an
                // activation warp run a phase ahead and arrive on a barrier
                // phase not its own.
                if constexpr (C_::SACT) {
                    if (named_bar_red_or(1 + stage, 32 * (1 + C_::MW), false)) live = false;
                } else {
                    named_bar_sync(1 + stage, 32 * (1 + C_::MW));
                }
                if (lane == 0 && live) {
                    tc_fence_after();
                    // scales gathered with cp.async (generic proxy) are read by tcgen05.cp
                    // through the async proxy
                    if (p.sf_rowmajor) fence_proxy_async_smem();
                    const uint32_t sf_col = tmem + C_::SF_COL0 + sf_slot * C_::SF_COLS_STAGE;
                    const uint64_t a_desc = a_desc0 + stage * (C_::A_BYTES >> 4);
                    // B and its scales: the stage's ring slot, or the resident stage kb
                    const uint64_t b_desc = C_::ACT ? b_desc0 + (kb - kb_lo) * SA * (C_::ACT_BYTES >> 4)
                                                    : b_desc0 + stage * (C_::B_BYTES >> 4);
                    const uint64_t sfa_desc = sfa_desc0 + stage * (C_::SFA_BYTES >> 4);
                    const uint64_t sfb_desc = C_::ACT ? sfb_desc0 + (kb - kb_lo) * SA * (C_::ACT_SF_BYTES >> 4)
                                                      : sfb_desc0 + stage * (C_::SFB_BYTES >> 4);
                    const int g_first = (kb + p.k_atom0) * C_::G;
                    // valid MMAs in this stage (ragged K): each consumes 32 bytes of K
                    const int rem = p.K - (kb + p.k_atom0) * k_elem_per_stage;
                    if (SA > 1 || rem >= k_elem_per_stage) {
                        // full stage: everything unrolled.
                        // scale tiles -> TMEM: SFA group g at sf_col + 4g;
                        // SFB group g, row-tile t at sf_col + SF_COLS_A + 4(g*SFB_TILES + t)
                        // (g counts the stage's groups: atom a holds groups a*G ..)
#pragma unroll
                        for (int gg = 0; gg < AW * C_::G; ++gg) {
                            const int g = a_first * C_::G + gg;  // this warp's atoms' groups
                            tc_cp_32x128b_warpx4(sf_col + 4 * g, sfa_desc + g * 32);
#pragma unroll
                            for (int t = 0; t < C_::SFB_TILES; ++t)
                                tc_cp_32x128b_warpx4(sf_col + C_::SF_COLS_A + 4 * (g * C_::SFB_TILES + t),
                                                     sfb_desc + (t * C_::GS + g) * 32);
                        }
#pragma unroll
                        for (int aa = 0; aa < AW; ++aa) {
                            const int a = a_first + aa;
                            // atom a of the stage: its A and B rows follow the previous atom's
                            const uint64_t ad = a_desc + a * (C_::A_ATOM >> 4);
                            const uint64_t bd = b_desc + a * (C_::B_ATOM >> 4);
#pragma unroll
                            for (int i = 0; i < kMmaPerStage; ++i) {
                                const int g = a * C_::G + (KIND == KIND_F4 ? (i >> 1) : 0);
                                const uint32_t accum = (kb > w.kb0 || aa > 0 || i > 0) ? 1u : 0u;
                                if (KIND == KIND_F4)
                                    mma_mxf4(d_tmem, ad + 2 * i, bd + 2 * i, idesc[i], sf_col + 4 * g,
                                             sf_col + C_::SF_COLS_A + 4 * g * C_::SFB_TILES, accum);
                                else
                                    mma_mxf8f6f4(d_tmem, ad + 2 * i, bd + 2 * i, idesc[i], sf_col + 4 * g,
                                                 sf_col + C_::SF_COLS_A + 4 * g * C_::SFB_TILES, accum);
                            }
                        }
                    } else {
                        // the ragged last stage of K
                        const int g_count = min(C_::G, p.sf_groups - g_first);
                        for (int g = 0; g < g_count; ++g) {
                            tc_cp_32x128b_warpx4(sf_col + 4 * g, sfa_desc + g * 32);
                            for (int t = 0; t < C_::SFB_TILES; ++t)
                                tc_cp_32x128b_warpx4(sf_col + C_::SF_COLS_A + 4 * (g * C_::SFB_TILES + t),
                                                     sfb_desc + (t * C_::G + g) * 32);
                        }
                        const int n_mma = (rem + k_elem_per_mma - 1) / k_elem_per_mma;
                        for (int i = 0; i < n_mma; ++i) {
                            const int g = KIND == KIND_F4 ? (i >> 1) : 0;
                            const uint32_t sf_id = KIND == KIND_F4 ? (uint32_t)(i & 1) * 2u : (uint32_t)i;
                            const uint32_t id = p.idesc | (sf_id << 4) | (sf_id << 29);
                            const uint32_t accum = (kb > w.kb0 || i > 0) ? 1u : 0u;
                            if (KIND == KIND_F4)
                                mma_mxf4(d_tmem, a_desc + 2 * i, b_desc + 2 * i, id, sf_col + 4 * g,
                                         sf_col + C_::SF_COLS_A + 4 * g * C_::SFB_TILES, accum);
                            else
                                mma_mxf8f6f4(d_tmem, a_desc + 2 * i, b_desc + 2 * i, id, sf_col + 4 * g,
                                             sf_col + C_::SF_COLS_A + 4 * g * C_::SFB_TILES, accum);
                        }
                    }
                    tc_commit(&empty[stage]);  // stage free once these MMAs have read it
                }
                __syncwarp();
                if (++sf_slot == C_::SF_SLOTS) sf_slot = 0;
                if (++stage == STAGES) stage = 0;
            }
            if (lane == 0 && live) tc_commit(&tmem_full[acc]);
            __syncwarp();
        }
        if (lane == 0) {
            // every tcgen05 op issued by this thread completes before TMEM is freed
            tc_commit(mma_done);
            mbar_wait(mma_done, 0, p.wait_limit_ns > kDrainLimitNs ? p.wait_limit_ns : kDrainLimitNs, err);
        }
        __syncwarp();
    } else if (warp == C_::GATE_WARP) {
        // ---------------------------------------------------------------- gate
        // For every stage of the schedule, wait (bounded) for its data, then
        // sync with the MMA warp on the stage's named barrier: once per stage,
        // in the same order, so neither warp can run a generation ahead; after
        // a timeout the gate stops waiting but keeps syncing.
        int stage = 0;
        uint32_t phase = 0;
        bool live = true;
        Work w;
        for (int it = 0; work_at(it, w); ++it) {
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                if (live) {
                    int okw = 1;
                    if (lane == 0) okw = mbar_wait(&full[stage], phase, p.wait_limit_ns, err);
                    okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                    if (!okw) {
                        live = false;
                        if (lane == 0) *abort_flag = 1;
                    }
                }
                if constexpr (C_::SACT) named_bar_red_or(1 + stage, 32 * (1 + C_::MW), !live);
                else named_bar_sync(1 + stage, 32 * (1 + C_::MW));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (C_::SACT && warp >= C_::ACT_WARP0) {
        if constexpr (C_::SACT) {
        // -------------------------------------------- streamed activations
        // Activation warp aw fills the B slot (codes and scale tile) of every
        // ACT_WARPS-th stage of the CTA's schedule, starting at stage aw: it
        // loads the stage's BN rows x SA atoms of bf16 activations (from
        // L2 after the first CTA's touch), quantizes them with mx_quantize's
        // rounding into the MMA operand layout (128-byte swizzled rows, the
        // tensor-core scale tile), waits for the slot to be free, writes it
        // and arrives on the stage's full barrier beside the TMA bytes.  Lane l
        // takes 32-element blocks l, l + 32, .. of the stage (row-major over
        // rows x blocks, so a warp's loads are contiguous); rows past M become
        // zero codes.  Loads and arithmetic happen before the slot wait, so
        // they overlap the MMAs still reading it.
        constexpr int BPA = KIND == KIND_F4 ? 8 : 4;   // 32-element blocks per atom
        constexpr int BPS = SA * BPA;                  // blocks per stage and row
        constexpr int PER_LANE = BN * BPS / 32;
        constexpr int AFMT = KIND == KIND_F4 ? FMT_E2M1 : FMT_E4M3;
        constexpr int CW = AFMT == FMT_E2M1 ? 4 : 8;   // code words per block
        const int aw = warp - C_::ACT_WARP0;
        int n = 0;  // the CTA's stage counter (identical in every role)
        bool live = true;
        Work w;
        for (int it = 0; live && work_at(it, w); ++it) {
            for (int kb = w.kb0; kb < w.kb1; ++kb, ++n) {
                if (n % C_::ACT_WARPS != aw) continue;
                const int stage = n % STAGES;
                const int64_t k_stage = (int64_t)(kb + p.k_atom0) * BPS * 32;  // first element of the stage
                uint8_t* bslot = smem + C_::OFF_B + stage * C_::B_BYTES;
                uint8_t* sfslot = smem + C_::OFF_SFB + stage * C_::SFB_BYTES;
                // KB blocks' loads are issued before any of them is converted;
                // the first batch's loads are in flight while the slot is
                // awaited (it is free once the MMAs of its previous fill have
                // read it; the first STAGES fills find it free)
                // (bf16 activations only: the host routes f32 to the resident path)
                auto fill = [&]() -> bool {
                    constexpr int WORDS = 16;  // one block of 32 bf16, two per word (lower element low)
                    constexpr int KB = 4;      // blocks per load batch
                    static_assert(PER_LANE % KB == 0, "whole load batches");
#pragma unroll
                    for (int b0 = 0; b0 < PER_LANE; b0 += KB) {
                        uint32_t raw[KB][WORDS];
#pragma unroll
                        for (int q = 0; q < KB; ++q) {
                            const int i = lane + 32 * (b0 + q);
                            const int r = i / BPS;
                            const int64_t k = k_stage + (int64_t)(i % BPS) * 32;
                            if (r < p.Q) {
                                const uint4* src = reinterpret_cast<const uint4*>(
                                    static_cast<const __nv_bfloat16*>(p.act) + (int64_t)r * p.act_ld + k);
#pragma unroll
                                for (int t = 0; t < WORDS / 4; ++t) {
                                    const uint4 v = __ldg(src + t);
                                    raw[q][4 * t] = v.x;
                                    raw[q][4 * t + 1] = v.y;
                                    raw[q][4 * t + 2] = v.z;
                                    raw[q][4 * t + 3] = v.w;
                                }
                            } else {
#pragma unroll
                                for (int t = 0; t < WORDS; ++t) raw[q][t] = 0;
                            }
                        }
                        if (b0 == 0) {
                            int okw = 1;
                            if (lane == 0 && n >= STAGES)
                                okw = mbar_wait(&empty[stage], ((uint32_t)(n / STAGES) & 1u) ^ 1u, p.wait_limit_ns,
                                                err);
                            if (!__shfl_sync(0xFFFFFFFFu, okw, 0)) return false;
                        }
#pragma unroll
                        for (int q = 0; q < KB; ++q) {
                            uint32_t out[CW];
                            const uint32_t sb = quantize_block_bf16<AFMT>(raw[q], out);  // word t: elements 2t, 2t + 1
                            const int i = lane + 32 * (b0 + q);
                            const int r = i / BPS, j = i % BPS;
                            const int a = j / BPA, jj = j % BPA;  // atom of the stage, block of the atom
                            uint8_t* rowp = bslot + a * C_::B_ATOM + r * kRowBytes;
                            if constexpr (AFMT == FMT_E4M3) {  // 32 bytes: 16-byte chunks 2jj, 2jj + 1
                                *reinterpret_cast<uint4*>(rowp + (((2 * jj) ^ (r & 7)) << 4)) =
                                    make_uint4(out[0], out[1], out[2], out[3]);
                                *reinterpret_cast<uint4*>(rowp + (((2 * jj + 1) ^ (r & 7)) << 4)) =
                                    make_uint4(out[4], out[5], out[6], out[7]);
                            } else {  // packed E2M1: 16 bytes, chunk jj
                                *reinterpret_cast<uint4*>(rowp + ((jj ^ (r & 7)) << 4)) =
                                    make_uint4(out[0], out[1], out[2], out[3]);
                            }
                            sfslot[(a * C_::G + jj / 4) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (jj & 3)] =
                                (uint8_t)sb;
                        }
                    }
                    return true;
                };
                const bool okf = fill();
                if (!okf) {
                    live = false;
                    if (lane == 0) *abort_flag = 1;
                    break;
                }
                fence_proxy_async_smem();  // generic writes, read by the tensor core
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[stage]);
            }
        }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // TMEM lane quarter this warp may read
        uint8_t* stage_buf = smem + C_::OFF_EPI + (warp - 2) * C_::NBUF * C_::EPI_BUF;
        (void)stage_buf;
        int nbuf = 0;  // chunks issued so far by this warp (buffer = nbuf % NBUF)
        Work w;
        for (int it = 0; work_at(it, w); ++it) {
            const int acc = it % ACC;
            const uint32_t acc_phase = (uint32_t)(it / ACC) & 1u;
            bool ok = !*abort_flag && mbar_wait(&tmem_full[acc], acc_phase, p.wait_limit_ns, err);
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int32_t p0 = w.tp * kBlockM + 32 * q;  // first MMA-A row of this warp
            const int32_t q0 = w.tq * BN;
            const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16) + kAccCol + acc * C_::MW * BN;
            if constexpr (C_::EPI_WARPS == 8) {
                // this warp: rows p0..p0+31, columns h*128 .. h*128+127 of the tile
                const int h = (warp - 2) >> 2;
                uint32_t r[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(t_row + h * 128 + 32 * c, r[c]);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tmem_empty[acc]);  // TMEM free: next tile may start
                epilogue_write_128(p, tm_c, r, p0, q0 + h * 128, stage_buf, nbuf, lane);
            } else if (SWAP) {
                // lane i holds acc(p0 + i, q0 + j), j < BN  ->  C[q0 + j][p0 + i]
                // (MW accumulators: their sum)
                uint32_t r[C_::MW][BN];
#pragma unroll
                for (int mm = 0; mm < C_::MW; ++mm)
#pragma unroll
                    for (int c = 0; c < BN / 16; ++c) {
                        uint32_t t[16];
                        tmem_ld_32x32b_x16(t_row + mm * BN + 16 * c, t);
#pragma unroll
                        for (int j = 0; j < 16; ++j) r[mm][16 * c + j] = t[j];
                    }
                tmem_ld_wait();
#pragma unroll
                for (int mm = 1; mm < C_::MW; ++mm)
#pragma unroll
                    for (int j = 0; j < BN; ++j)
                        r[0][j] = __float_as_uint(__uint_as_float(r[0][j]) + __uint_as_float(r[mm][j]));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tmem_empty[acc]);
                if (p.use_tma_epi) {
                    uint8_t* buf = stage_buf + (nbuf % C_::NBUF) * C_::EPI_BUF;
                    if (nbuf >= C_::NBUF && lane == 0) bulk_wait_group_read<C_::NBUF - 1>();
                    __syncwarp();
                    float* f = reinterpret_cast<float*>(buf);
#pragma unroll
                    for (int j = 0; j < BN; ++j) f[j * 32 + lane] = __uint_as_float(r[0][j]);  // [BN rows][32 cols]
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_reduce_add_2d(&tm_c, buf, p0, q0);
                        bulk_commit_group();
                    }
                    ++nbuf;
                } else {
                    const int32_t pr = p0 + lane;
                    if (pr < p.P) {
#pragma unroll
                        for (int j = 0; j < BN; ++j)
                            if (q0 + j < p.Q) atomicAdd(p.C + (int64_t)(q0 + j) * p.ldc + pr, __uint_as_float(r[0][j]));
                    }
                }
            } else {
                constexpr int nchunks = BN / 32;
                const int32_t pr = p0 + lane;
                for (int c = 0; c < nchunks; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(t_row + 32 * c, r);
                    tmem_ld_wait();
                    if (c == nchunks - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tmem_empty[acc]);
                    }
                    if (q0 + 32 * c >= p.Q) continue;  // chunk wholly past N
                    if (p.use_tma_epi) {
                        uint8_t* buf = stage_buf + (nbuf % C_::NBUF) * C_::EPI_BUF;
                        if (nbuf >= C_::NBUF && lane == 0) bulk_wait_group_read<C_::NBUF - 1>();
                        __syncwarp();
                        // [32 rows][32 f32] with the 128-byte swizzle: 16-B chunk j of
                        // row i sits at chunk j ^ (i & 7)
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int js = j ^ (lane & 7);
                            uint4 v = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                            *reinterpret_cast<uint4*>(buf + lane * 128 + js * 16) = v;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_reduce_add_2d(&tm_c, buf, q0 + 32 * c, p0);
                            bulk_commit_group();
                        }
                        ++nbuf;
                    } else if (pr < p.P) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (q0 + 32 * c + j < p.Q)
                                atomicAdd(p.C + (int64_t)pr * p.ldc + q0 + 32 * c + j, __uint_as_float(r[j]));
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        tmem_dealloc(tmem, kTmemCols);
    } else if (warp == 0 && *abort_flag) {
        // Drain after a give-up (every give-up raises the flag before the
        // barrier above; without one the gate saw every fill land): every
        // load this CTA issued lands before it leaves.  Each slot's earlier
        // fills were seen landing before its last one was issued, so the
        // barrier is in that fill's phase.
        if (p.sf_rowmajor) cp_async_wait_all();
        if (lane == 0) {
            const uint64_t lim = p.wait_limit_ns > kDrainLimitNs ? p.wait_limit_ns : kDrainLimitNs;
            for (int s = 0; s < STAGES && s < n_issued; ++s) {
                const int lf = s + ((n_issued - 1 - s) / STAGES) * STAGES;  // the slot's last fill
                mbar_wait(&full[s], (uint32_t)(lf / STAGES) & 1u, lim, err);
            }
        }
        __syncwarp();
    }
}

// ------------------------------------------------------------ CTA pairs
//
// 256 x 256 tiles on a cluster of two CTAs (tcgen05 .cta_group::2, M = 256).
// CTA r of the pair stages rows [256 tp + 128 r, +128) of the MMA A operand
// and rows [256 tq + 128 r, +128) of the B operand, the scale tile of its A
// rows and the scale tiles of all 256 B rows.  Every load of both CTAs counts
// its bytes on the even CTA's stage barrier; that CTA's MMA thread then issues
// the scale copies and MMAs for the pair, and its commits free the stage in
// both CTAs and hand the accumulator (rows of each CTA's half, in each CTA's
// TMEM) to both CTAs' epilogues, whose eight warps each release it back to the
// even CTA once drained into registers.  In the even CTA a gate warp waits on
// each stage's barrier and passes it to the MMA warp through a named barrier
// (one per stage slot), so the issuing thread never touches shared memory
// between MMAs.  Per SM a stage holds 32 KB of codes
// for the same MMA work that needs 48 KB with 128 x 256 tiles on one SM: more
// stages fit, and a third less data crosses from L2 per MMA.
// SA: K atoms per stage (a stage is then one 3-D box of SA atoms per operand
// and scale tensor: the per-stage issue cost is paid once per SA atoms).
// MMA-issuing warps of the two-atom pair configurations
constexpr int kPairMW = 2;

// After the pair kernel's loop, in the even CTA (one thread, after a cluster
// barrier that made the odd CTA's fill count visible): every load either CTA
// issued has landed when this returns (or the drain limit has passed).
//  - A fill is issued by a producer only after its wait on the slot's empty
//    barrier saw the MMAs of the slot's previous fill complete, which needed
//    that fill's full phase, armed by the even CTA and fed by both CTAs'
//    loads.  So the two fill counts differ by at most STAGES, no slot has two
//    fills that only one CTA issued, and when such a fill f is adjusted its
//    slot's barrier is in f's phase.
//  - A fill the even CTA issued (and armed with both CTAs' bytes) and the odd
//    CTA did not: the odd CTA's bytes are counted as arrived.  A fill only the
//    odd CTA issued: the even CTA arms it with the odd CTA's bytes.
//  - Then each slot's last fill is waited for (the slot's earlier fills were
//    consumed before it was issued, so its phase parity is unambiguous).
template <int STAGES>
__device__ void drain_pair_loads(uint64_t* full, int n_even, int n_odd, uint32_t one_cta_tx, uint64_t limit,
                                 unsigned* err) {
    const int lo = n_even < n_odd ? n_even : n_odd;
    const int hi = n_even < n_odd ? n_odd : n_even;
    for (int f = lo; f < hi; ++f) {
        if (f < n_even) mbar_complete_tx(&full[f % STAGES], one_cta_tx);
        else mbar_arrive_expect_tx(&full[f % STAGES], one_cta_tx);
    }
    for (int s = 0; s < STAGES && s < hi; ++s) {
        const int last = s + ((hi - 1 - s) / STAGES) * STAGES;
        mbar_wait(&full[s], (uint32_t)(last / STAGES) & 1u, limit, err);
    }
}

// MW: MMA-issuing warps (1, or 2 with two-atom stages: warp 1 issues atom 0
// of every stage, the warp after the gate atom 1, both into the one
// accumulator)
template <int KIND, int STAGES, int EC = 16, int SA = 1, int MW = 1>
struct PairCfg {
    static constexpr int G = KIND == KIND_F4 ? 2 : 1;  // scale groups per atom
    static constexpr int GS = SA * G;                   // scale groups per stage
    static constexpr int EPI_WARPS = 8;
    static constexpr int GATE_WARP = 2 + EPI_WARPS;  // waits on stage barriers for the MMA warp(s)
    static constexpr int THREADS = 32 * (GATE_WARP + MW);
    static constexpr int TILE_BAR = STAGES + 1;      // named barrier of the MMA warps' tile hand-off
    static constexpr int A_ATOM = 128 * kRowBytes;
    static constexpr int B_ATOM = 128 * kRowBytes;
    static constexpr int A_BYTES = SA * A_ATOM;
    static constexpr int B_BYTES = SA * B_ATOM;
    static constexpr int SFA_BYTES = GS * 512;
    static constexpr int SFB_BYTES = 2 * GS * 512;
    static constexpr int SF_COLS_A = 4 * GS;
    static constexpr int SF_COLS_STAGE = 12 * GS;
    static constexpr int SF_COL0 = 256;  // accumulator in columns [0, 256)
    static constexpr int SF_SLOTS_FIT = ((int)kTmemCols - SF_COL0) / SF_COLS_STAGE;
    static constexpr int SF_SLOTS = SF_SLOTS_FIT < STAGES ? SF_SLOTS_FIT : STAGES;
    static constexpr int EPI_BUF = 32 * EC * 4;  // one 32 x EC staging box per epilogue warp
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_EPI = (OFF_SFB + STAGES * SFB_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_BUF;
    static constexpr int BAR_BYTES = (2 * STAGES + 4) * 8 + 16;
    static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;
    static constexpr uint32_t SF_TX = (uint32_t)(SFA_BYTES + SFB_BYTES);
    static_assert(MW == 1 || (MW == 2 && SA == 2), "two MMA warps take one atom of a two-atom stage each");
    static_assert(TILE_BAR <= 15, "named barrier ids");
    static_assert(SF_SLOTS >= 2, "at least two scale slots in TMEM");
    static_assert(SMEM <= 232448, "shared memory per CTA");
    static_assert(STAGES <= 15, "one named barrier per stage");
};

template <int KIND, int STAGES, int EC = 16, int SA = 1, int MW = 1>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<KIND, STAGES, EC, SA, MW>::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const __grid_constant__ CUtensorMap tm_sfa, const __grid_constant__ CUtensorMap tm_sfb,
                     const __grid_constant__ CUtensorMap tm_c, const GemmParams p) {
    using C_ = PairCfg<KIND, STAGES, EC, SA, MW>;
    extern __shared__ uint8_t smem_raw[];
    // the same offsets in both CTAs: the MMAs and barrier addresses rely on it
    // aligned by an offset from the array itself: the compiler then keeps the
    // generic accesses below (epilogue staging, activation tiles) in the shared window
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C_::OFF_BAR);  // used in the even CTA
    uint64_t* empty = full + STAGES;
    uint64_t* tmem_full = empty + STAGES;
    uint64_t* tmem_empty = tmem_full + 1;  // used in the even CTA
    uint64_t* mma_done = tmem_empty + 1;  // [2], one per MMA warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint32_t* fills = tmem_slot + 2;  // [0]: this CTA's fills issued; [1] (even CTA): the odd CTA's

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t pair = cluster_id_x();
    const uint32_t npairs = cluster_count_x();
    unsigned* err = &g_mx_device_error;
    pdl_launch_dependents();

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], MW);  // one commit per MMA warp
        }
        mbar_init(tmem_full, MW);
        mbar_init(tmem_empty, 2 * C_::EPI_WARPS);
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tensormap(&tm_a);
        prefetch_tensormap(&tm_b);
        prefetch_tensormap(&tm_sfa);
        prefetch_tensormap(&tm_sfb);
        if (p.use_tma_epi) prefetch_tensormap(&tm_c);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA use
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // set-up above overlaps the previous kernel's tail; global memory from here on
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // A stage is four loads -- A, B, A's scales, B's scales -- issued by
        // lanes 0..3 with one instruction (3-D operand maps) or two.
        const uint32_t full_even = mapa_shared(smem_u32(full), 0);
        const int li = lane & 3;
        const void* lmap = li == 0 ? (const void*)&tm_a : li == 1 ? (const void*)&tm_b
                                                    : li == 2 ? (const void*)&tm_sfa : (const void*)&tm_sfb;
        const uint32_t lbase = smem_u32(smem) + (li == 0 ? C_::OFF_A : li == 1 ? C_::OFF_B
                                                  : li == 2 ? C_::OFF_SFA : C_::OFF_SFB);
        const uint32_t lstep = li == 0 ? C_::A_BYTES : li == 1 ? C_::B_BYTES : li == 2 ? C_::SFA_BYTES : C_::SFB_BYTES;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        uint32_t n_fill = 0;  // fills issued
        Work w;
        for (int it = 0; ok && get_work(p, pair, npairs, it, w); ++it) {
            const int32_t a_row = w.tp * 256 + (int32_t)rank * 128;
            const int32_t b_row = w.tq * 256 + (int32_t)rank * 128;
            for (int kb = w.kb0; kb < w.kb1; ++kb) {
                int okw = 1;
                if (lane == 0) okw = mbar_wait(&empty[stage], phase ^ 1, p.wait_limit_ns, err);
                okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                if (!okw) {
                    if (lane == 0) *abort_flag = 1;
                    ok = false;
                    break;
                }
                // the even CTA announces both CTAs' bytes; a load of the odd CTA
                // that lands first only takes the count below zero meanwhile
                if (lane == 0 && rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * (p.tx_a + p.tx_b + C_::SF_TX));
                const uint32_t bar = full_even + (uint32_t)stage * 8;
                const uint32_t dst = lbase + (uint32_t)stage * lstep;
                // coordinates: operands (0, row, first atom) in 3-D, (128 B * stage, row) in 2-D;
                // scales (0, 4 GS stage, 128-row tile)
                const int32_t y = li == 0 ? a_row : li == 1 ? b_row : 4 * C_::GS * kb;
                const int32_t z = li < 2 ? SA * kb : (li == 2 ? a_row >> 7 : w.tq * 2);
                if (p.op3d) {
                    if (lane < 4) tma_load_3d_pair_at(dst, lmap, 0, y, z, bar);
                } else {
                    if (lane < 2) tma_load_2d_pair_at(dst, lmap, kb * kRowBytes, y, bar);
                    else if (lane < 4) tma_load_3d_pair_at(dst, lmap, 0, y, z, bar);
                }
                __syncwarp();
                ++n_fill;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        // the fill count goes to the even CTA, which waits at the end for every
        // load of both CTAs (this CTA's loads count on its barriers)
        if (lane == 0) {
            if (rank == 0) fills[0] = n_fill;
            else st_shared_cluster_u32(mapa_shared(smem_u32(&fills[1]), 0), n_fill);
        }
        __syncwarp();
    } else if (warp == 1 || (MW > 1 && warp == C_::GATE_WARP + 1)) {
        // ---------------------------------------------------------- MMA issue
        // The whole warp walks the schedule and syncs on stage s's named
        // barrier (1 + s) with the gate warp; lane 0 issues.  After an abort
        // the warp keeps walking (and syncing) without issuing, so its syncs
        // and the gate's always pair up.  With two MMA warps, warp m issues
        // atom m of every stage (its scale copies, four MMAs, a commit) into
        // the one accumulator; the first MMA of a work unit, which overwrites
        // the accumulator, is warp 0's, and warp 1 issues nothing of that unit
        // until warp 0 has (a tcgen05 fence and the tile hand-off barrier, once
        // per unit), after which the order of the two warps' MMAs only changes
        // the rounding order of the sums.
        if (rank == 0) {
            const int m = warp == 1 ? 0 : 1;
            constexpr int AW = SA / MW;  // atoms per MMA warp
            const int a_first = m * AW;
            const uint64_t a_desc0 = smem_desc(smem_u32(smem + C_::OFF_A), 0, 1024, 2);
            const uint64_t b_desc0 = smem_desc(smem_u32(smem + C_::OFF_B), 0, 1024, 2);
            const uint64_t sfa_desc0 = smem_desc(smem_u32(smem + C_::OFF_SFA), 0, 128, 0);
            const uint64_t sfb_desc0 = smem_desc(smem_u32(smem + C_::OFF_SFB), 0, 128, 0);
            uint32_t idesc[kMmaPerStage];
#pragma unroll
            for (int i = 0; i < kMmaPerStage; ++i) {
                const uint32_t sf_id = KIND == KIND_F4 ? (uint32_t)(i & 1) * 2u : (uint32_t)i;
                idesc[i] = p.idesc | (sf_id << 4) | (sf_id << 29);
            }
            constexpr int k_elem_per_stage = SA * (KIND == KIND_F4 ? 256 : 128);
            constexpr int k_elem_per_mma = KIND == KIND_F4 ? 64 : 32;
            int stage = 0;
            int sf_slot = 0;
            bool live = true;  // false after an abort: walk without issuing
            Work w;
            for (int it = 0; get_work(p, pair, npairs, it, w); ++it) {
                // both CTAs' epilogues have drained the previous tile
                int okt = 1;
                if (lane == 0 && live)
                    okt = !*abort_flag && mbar_wait_cluster(tmem_empty, ((uint32_t)it & 1u) ^ 1u, p.wait_limit_ns, err);
                okt = __shfl_sync(0xFFFFFFFFu, okt, 0);
                if (live && !okt) {
                    live = false;
                    if (lane == 0) *abort_flag = 1;
                }
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    // the gate saw this stage's data land, or gave up waiting for it
                    if (named_bar_red_or(1 + stage, 32 * (1 + MW), false)) live = false;
                    if (MW > 1 && m == 1 && kb == w.kb0) named_bar_sync(C_::TILE_BAR, 64);  // see above
                    if (lane == 0 && live) {
                        tc_fence_after();
                        const uint32_t sf_col = tmem + C_::SF_COL0 + sf_slot * C_::SF_COLS_STAGE;
                        const uint64_t a_desc = a_desc0 + stage * (C_::A_BYTES >> 4);
                        const uint64_t b_desc = b_desc0 + stage * (C_::B_BYTES >> 4);
                        const uint64_t sfa_desc = sfa_desc0 + stage * (C_::SFA_BYTES >> 4);
                        const uint64_t sfb_desc = sfb_desc0 + stage * (C_::SFB_BYTES >> 4);
                        // scale tiles -> TMEM: A group g at sf_col + 4g; B group g, row tile t
                        // at sf_col + SF_COLS_A + 4 (2g + t); g counts the stage's groups
                        // (atom a holds groups a G ..)
#pragma unroll
                        for (int gg = 0; gg < AW * C_::G; ++gg) {
                            const int g = a_first * C_::G + gg;  // this warp's atoms' groups
                            tc_cp_pair_32x128b_warpx4(sf_col + 4 * g, sfa_desc + g * 32);
#pragma unroll
                            for (int t = 0; t < 2; ++t)
                                tc_cp_pair_32x128b_warpx4(sf_col + C_::SF_COLS_A + 4 * (2 * g + t),
                                                          sfb_desc + (t * C_::GS + g) * 32);
                        }
                        const int rem = p.K - kb * k_elem_per_stage;
                        if (SA > 1 || rem >= k_elem_per_stage) {
#pragma unroll
                            for (int aa = 0; aa < AW; ++aa) {
                                const int a = a_first + aa;
                                const uint64_t ad = a_desc + a * (C_::A_ATOM >> 4);
                                const uint64_t bd = b_desc + a * (C_::B_ATOM >> 4);
#pragma unroll
                                for (int i = 0; i < kMmaPerStage; ++i) {
                                    const int g = a * C_::G + (KIND == KIND_F4 ? (i >> 1) : 0);
                                    const uint32_t accum = (kb > w.kb0 || a > 0 || i > 0) ? 1u : 0u;
                                    if (KIND == KIND_F4)
                                        mma_pair_mxf4(tmem, ad + 2 * i, bd + 2 * i, idesc[i], sf_col + 4 * g,
                                                      sf_col + C_::SF_COLS_A + 8 * g, accum);
                                    else
                                        mma_pair_mxf8f6f4(tmem, ad + 2 * i, bd + 2 * i, idesc[i], sf_col + 4 * g,
                                                          sf_col + C_::SF_COLS_A + 8 * g, accum);
                                }
                            }
                        } else {
                            // the ragged last stage of K
                            const int n_mma = (rem + k_elem_per_mma - 1) / k_elem_per_mma;
                            for (int i = 0; i < n_mma; ++i) {
                                const int g = KIND == KIND_F4 ? (i >> 1) : 0;
                                const uint32_t sf_id = KIND == KIND_F4 ? (uint32_t)(i & 1) * 2u : (uint32_t)i;
                                const uint32_t id = p.idesc | (sf_id << 4) | (sf_id << 29);
                                const uint32_t accum = (kb > w.kb0 || i > 0) ? 1u : 0u;
                                if (KIND == KIND_F4)
                                    mma_pair_mxf4(tmem, a_desc + 2 * i, b_desc + 2 * i, id, sf_col + 4 * g,
                                                  sf_col + C_::SF_COLS_A + 8 * g, accum);
                                else
                                    mma_pair_mxf8f6f4(tmem, a_desc + 2 * i, b_desc + 2 * i, id, sf_col + 4 * g,
                                                      sf_col + C_::SF_COLS_A + 8 * g, accum);
                            }
                        }
                        tc_commit_pair(&empty[stage]);  // stage free in both CTAs once read
                    }
                    __syncwarp();
                    if (MW > 1 && m == 0 && kb == w.kb0) {
                        // hand-off: warp 1's MMAs of this unit come after the one that overwrote
                        if (lane == 0) tc_fence_before();
                        named_bar_sync(C_::TILE_BAR, 64);
                    }
                    if (++sf_slot == C_::SF_SLOTS) sf_slot = 0;
                    if (++stage == STAGES) stage = 0;
                }
                if (lane == 0 && live) tc_commit_pair(tmem_full);
                __syncwarp();
            }
            if (lane == 0) {
                // every tcgen05 op this thread issued completes before TMEM is freed
                tc_commit_pair(&mma_done[m]);
                mbar_wait(&mma_done[m], 0, p.wait_limit_ns > kDrainLimitNs ? p.wait_limit_ns : kDrainLimitNs, err);
            }
            __syncwarp();
        }
    } else if (warp == C_::GATE_WARP) {
        // ---------------------------------------------------------------- gate
        // Even CTA: for every stage of the schedule, wait (bounded) for its
        // data, then sync with the MMA warp on the stage's named barrier.  The
        // two warps sync once per stage in the same order (lockstep: neither
        // can run a generation ahead), and after a timeout the gate stops
        // waiting but keeps syncing, so every sync has its partner.  The
        // gate's wait for stage s + 1 overlaps the MMA warp's issue of stage
        // s, which the tensor pipe paces.
        if (rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool live = true;
            Work w;
            for (int it = 0; get_work(p, pair, npairs, it, w); ++it) {
                for (int kb = w.kb0; kb < w.kb1; ++kb) {
                    if (live) {
                        int okw = 1;
                        if (lane == 0) okw = mbar_wait(&full[stage], phase, p.wait_limit_ns, err);
                        okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
                        if (!okw) {
                            live = false;
                            if (lane == 0) *abort_flag = 1;
                        }
                    }
                    // the MMA warps learn here whether this stage's data landed: after
                    // a give-up they issue nothing more, so a slot is only released
                    // (and refilled) once its data has landed
                    named_bar_red_or(1 + stage, 32 * (1 + MW), !live);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;         // TMEM lane quarter this warp may read
        const int h = (warp - 2) >> 2;  // which 128 of the 256 columns
        uint8_t* stage_buf = smem + C_::OFF_EPI + (warp - 2) * C_::EPI_BUF;
        const uint32_t tmem_empty_even = mapa_shared(smem_u32(tmem_empty), 0);
        int nbuf = 0;
        Work w;
        for (int it = 0; get_work(p, pair, npairs, it, w); ++it) {
            const bool ok = !*abort_flag && mbar_wait_cluster(tmem_full, (uint32_t)it & 1u, p.wait_limit_ns, err);
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int32_t p0 = w.tp * 256 + (int32_t)rank * 128 + 32 * q;
            const uint32_t t_row = tmem + ((uint32_t)(32 * q) << 16) + h * 128;
            uint32_t r[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(t_row + 32 * c, r[c]);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(tmem_empty_even);  // next tile's MMAs may start
            epilogue_write_128<EC>(p, tm_c, r, p0, w.tq * 256 + h * 128, stage_buf, nbuf, lane);
        }
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every role is done; the odd CTA's fill count is in the even CTA
    if (rank == 0 && threadIdx.x == 0)
        drain_pair_loads<STAGES>(full, (int)fills[0], (int)fills[1], p.tx_a + p.tx_b + C_::SF_TX,
                                 p.wait_limit_ns > kDrainLimitNs ? p.wait_limit_ns : kDrainLimitNs, err);
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves before every load of both has landed
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace

bool encode_tiled_map(CUtensorMap* m, CUtensorMapDataType dt, uint32_t rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swizzle) {
    EncodeTiledFn enc = encode_fn();
    if (!enc || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], e[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) st[i] = strides_bytes[i];
    }
    return enc(m, dt, rank, const_cast<void*>(base), d, st, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

unsigned* device_error_word() {
    // the symbol's address in the current device's context, looked up once per device
    static std::mutex mu;
    static unsigned* word[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!word[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_mx_device_error) == cudaSuccess) word[dev] = static_cast<unsigned*>(p);
        else cudaGetLastError();
    }
    return word[dev];
}

namespace {

// Tensor map over the codes of an operand with `rows` rows of K elements.
// fmt_kind: 0 = one byte per element (E4M3), 1 = packed E2M1 as bytes,
// 2 = packed E2M1 expanded to one byte per element in shared memory.
bool make_operand_map(CUtensorMap* m, const void* codes, int64_t rows, int64_t K, int fmt_kind, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2];
    cuuint64_t strides[1];
    cuuint32_t box[2] = {(cuuint32_t)kRowBytes, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (fmt_kind == 0) {
        dims[0] = (cuuint64_t)K;
        strides[0] = (cuuint64_t)K;
    } else if (fmt_kind == 1) {
        dims[0] = (cuuint64_t)(K / 2);
        strides[0] = (cuuint64_t)(K / 2);
    } else {
        dt = CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
        dims[0] = (cuuint64_t)K;  // counted in 4-bit elements
        strides[0] = (cuuint64_t)(K / 2);
    }
    dims[1] = (cuuint64_t)rows;
    CUresult r = enc(m, dt, 2, const_cast<void*>(codes), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same codes viewed in 3-D as [stages][rows][one stage of K]: one stage of
// a row is a 128-byte swizzle atom (128 E4M3 codes, 256 packed E2M1 codes, or
// 128 E2M1 codes expanded to a byte each), the atom stride is its packed size
// and the row stride a row's bytes, so the box {atom, box_rows, 1} at
// (0, row, stage) is the 2-D box at (128 B * stage, row).  Only for K a whole
// number of stages: a partial last atom would read into the next row.
bool make_operand_map3n(CUtensorMap* m, const void* codes, int64_t rows, int64_t K, int fmt_kind, int box_rows,
                        int box_atoms) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[3], strides[2];
    if (fmt_kind == 0) {  // E4M3, one byte each
        dims[0] = kRowBytes;
        dims[2] = (cuuint64_t)(K / kRowBytes);
        strides[0] = (cuuint64_t)K;
        strides[1] = kRowBytes;
    } else if (fmt_kind == 1) {  // packed E2M1 as bytes: an atom is 256 elements
        dims[0] = kRowBytes;
        dims[2] = (cuuint64_t)(K / (2 * kRowBytes));
        strides[0] = (cuuint64_t)(K / 2);
        strides[1] = kRowBytes;
    } else {  // packed E2M1 expanded to a byte each in shared memory: an atom is 128 elements, 64 B in HBM
        dt = CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
        dims[0] = kRowBytes;  // counted in 4-bit elements
        dims[2] = (cuuint64_t)(K / kRowBytes);
        strides[0] = (cuuint64_t)(K / 2);
        strides[1] = kRowBytes / 2;
    }
    dims[1] = (cuuint64_t)rows;
    cuuint32_t box[3] = {(cuuint32_t)kRowBytes, (cuuint32_t)box_rows, (cuuint32_t)box_atoms};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, dt, 3, const_cast<void*>(codes), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over C (rows x cols f32, row-major) for the reduce-add epilogue.
bool make_c_map(CUtensorMap* m, float* C, int64_t rows, int64_t cols, int box_cols, int box_rows, int swizzle) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(cols * 4)};
    cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, C, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                    : (swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
                     CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Instruction descriptor (block-scaled kinds), scale-factor ids left 0:
//   [7,10) A type  [10,13) B type  [15] A K-major(0)  [16] B K-major(0)
//   [17,23) N>>3   [23] scale type UE8M0 (1)   [24,29) M>>4
uint32_t make_idesc(int kind, int a_fmt, int b_fmt, int n, int m = kBlockM) {
    auto code = [&](int f) -> uint32_t {
        if (kind == KIND_F4) return 1u;          // E2M1 in kind::mxf4
        return f == FMT_E2M1 ? 5u : 0u;          // kind::mxf8f6f4: E2M1 = 5, E4M3 = 0
    };
    uint32_t d = 0;
    d |= code(a_fmt) << 7;
    d |= code(b_fmt) << 10;
    d |= (uint32_t)(n >> 3) << 17;
    d |= 1u << 23;
    d |= (uint32_t)(m >> 4) << 24;
    return d;
}

// Tensor map over scales in the tensor-core layout, as [tiles][4 * groups][128 B]
// (a 128-row tile's group g is the 512 bytes of rows 4g .. 4g+3): a box of
// 4 * g_box rows x `tiles_box` tiles loads g_box groups of that many tiles.
bool make_sf_map(CUtensorMap* m, const uint8_t* sf, int64_t rows, int32_t sf_groups, int g_box, int tiles_box) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)sf_groups * 4, (cuuint64_t)((rows + 127) / 128)};
    cuuint64_t strides[2] = {128, (cuuint64_t)sf_groups * 512};
    cuuint32_t box[3] = {128, (cuuint32_t)(4 * g_box), (cuuint32_t)tiles_box};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(sf), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int KIND, int BN, int STAGES, int SWAP, int NBUF_ = 0, int ACT_ATOMS = 0, int SA = 1>
cudaError_t run(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa, const CUtensorMap& tsb,
                const CUtensorMap& tc, const GemmParams& p, int grid, cudaStream_t st) {
    using C_ = Cfg<KIND, BN, STAGES, SWAP, NBUF_, ACT_ATOMS, SA>;
    auto kern = gemm_kernel<KIND, BN, STAGES, SWAP, NBUF_, ACT_ATOMS, SA>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), C_::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(C_::THREADS), C_::SMEM, st, ta, tb, tsa, tsb, tc, p);
}

// CTA pairs that can be resident at once for a pair-kernel instantiation
// (pairs need two SMs of one GPU processing cluster); cached per instantiation.
template <int KIND, int STAGES, int EC = 16, int SA = 1, int MW = 1>
cudaError_t run_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tsa, const CUtensorMap& tsb,
                     const CUtensorMap& tc, const GemmParams& p, int pairs, cudaStream_t st) {
    using C_ = PairCfg<KIND, STAGES, EC, SA, MW>;
    auto kern = gemm_pair_kernel<KIND, STAGES, EC, SA, MW>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), C_::SMEM);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(2 * pairs), dim3(C_::THREADS), C_::SMEM, st, ta, tb, tsa, tsb, tc, p);
}

template <int KIND, int STAGES, int EC = 16, int SA = 1, int MW = 1>
int pair_capacity() {
    using C_ = PairCfg<KIND, STAGES, EC, SA, MW>;
    static std::mutex mu;
    static int cap[64];
    static bool known[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (known[dev]) return cap[dev];
    auto kern = gemm_pair_kernel<KIND, STAGES, EC, SA, MW>;
    int n = 0;
    if (ensure_smem_limit(reinterpret_cast<const void*>(kern), C_::SMEM) == cudaSuccess) {
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof(cfg));
        cfg.gridDim = dim3(2 * (unsigned)(sm_count() / 2), 1, 1);
        cfg.blockDim = dim3(C_::THREADS, 1, 1);
        cfg.dynamicSmemBytes = C_::SMEM;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
    } else {
        cudaGetLastError();
    }
    cap[dev] = n;
    known[dev] = true;
    return n;
}

__global__ void wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
        // nothing ever arrives on `bar`: this wait must give up and report
        mbar_wait(&bar, 0, limit_ns, &g_mx_device_error);
    }
}

}  // namespace

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(limit_ns);
    return cudaGetLastError();
}

namespace {

// Row tiles per band of the whole-tile order: as many as keep the band's A
// codes within about 40 MB (a third of L2, which C's read-modify-write traffic
// also passes through), so they are read from HBM once while every column
// tile streams past; all row tiles when A fits.
int32_t band_rows(int32_t tiles_p, int64_t a_tile_bytes) {
    const int64_t budget = 40ll << 20;
    int64_t g = a_tile_bytes > 0 ? budget / a_tile_bytes : tiles_p;
    if (g < 1) g = 1;
    return (int32_t)(g < tiles_p ? g : tiles_p);
}

// 256 x 256 tiles on CTA pairs.  Returns cudaErrorNotSupported (nothing
// launched) when no pair can be resident, so the caller takes the one-CTA path.
cudaError_t launch_pair(const GemmArgs& a, int kind, const void* x_codes, const uint8_t* x_sf, int x_fmt, int64_t P,
                        const void* y_codes, const uint8_t* y_sf, int y_fmt, int64_t Q, cudaStream_t st,
                        const char** detail) {
    // Two K atoms per stage when K allows (one 3-D box per operand and scale
    // tensor per two atoms: the per-stage issue cost is halved); three such
    // stages hold what six single-atom ones did.  FP4 stages its epilogue
    // through 32 x 8 boxes (1 KB per warp) to make room.
    const int64_t k_atom = kind == KIND_F4 ? 256 : 128;
    const int sa = (a.K % (2 * k_atom)) == 0 ? 2 : 1;
    const int cap = kind == KIND_F4 ? (sa == 2 ? pair_capacity<KIND_F4, 3, 8, 2, kPairMW>() : pair_capacity<KIND_F4, 6, 8>())
                                    : (sa == 2 ? pair_capacity<KIND_F8F6F4, 3, 16, 2, kPairMW>()
                                               : pair_capacity<KIND_F8F6F4, 6>());
    if (cap <= 0) return cudaErrorNotSupported;
    const int64_t k_per_stage = sa * k_atom;
    const int g = sa * (kind == KIND_F4 ? 2 : 1);
    auto fk = [&](int f) { return f == FMT_E4M3 ? 0 : (kind == KIND_F4 ? 1 : 2); };
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.P = (int32_t)P;
    p.Q = (int32_t)Q;
    p.K = (int32_t)a.K;
    p.tiles_p = (int32_t)((P + 255) / 256);
    p.tiles_q = (int32_t)((Q + 255) / 256);
    p.k_stages = (int32_t)((a.K + k_per_stage - 1) / k_per_stage);
    p.sf_groups = (int32_t)(round_up(a.K / 32, 4) / 4);
    p.wait_limit_ns = wait_limit_ns();
    p.idesc = make_idesc(kind, x_fmt, y_fmt, 256, 256);
    p.use_tma_epi = (a.N % 4) == 0 ? 1 : 0;
    p.C = a.C;
    p.ldc = a.N;
    p.sfa = x_sf;
    p.sfb = y_sf;
    p.tx_a = (uint32_t)(sa * 128) * (fk(x_fmt) == 2 ? kRowBytes / 2 : kRowBytes);
    p.tx_b = (uint32_t)(sa * 128) * (fk(y_fmt) == 2 ? kRowBytes / 2 : kRowBytes);
    p.nb = (int32_t)(a.K / 32);
    CUtensorMap ta, tb, tsa, tsb, tc;
    std::memset(&tc, 0, sizeof(tc));
    p.op3d = (a.K % k_atom) == 0 ? 1 : 0;
    auto opmap = [&](CUtensorMap* m, const void* codes, int64_t rows, int f) {
        return p.op3d ? make_operand_map3n(m, codes, rows, a.K, fk(f), 128, sa)
                      : make_operand_map(m, codes, rows, a.K, fk(f), 128);
    };
    if (!opmap(&ta, x_codes, P, x_fmt) || !opmap(&tb, y_codes, Q, y_fmt) ||
        !make_sf_map(&tsa, x_sf, P, p.sf_groups, g, 1) || !make_sf_map(&tsb, y_sf, Q, p.sf_groups, g, 2) ||
        (p.use_tma_epi && !(kind == KIND_F4 ? make_c_map(&tc, a.C, a.M, a.N, 8, 32, 0)
                                            : make_c_map(&tc, a.C, a.M, a.N, 16, 32, 64)))) {
        *detail = "cuTensorMapEncodeTiled rejected an operand";
        return cudaErrorInvalidValue;
    }
    const int64_t tiles = (int64_t)p.tiles_p * p.tiles_q;
    p.total_units = tiles * p.k_stages;
    p.group_p = band_rows(p.tiles_p, 256 * (x_fmt == FMT_E2M1 ? a.K / 2 : a.K));
    int pairs;
    if (tiles >= cap || p.k_stages < 4) {
        // whole tiles; a last partial round is split along K over all pairs
        p.mode = (tiles > cap && tiles % cap != 0 && p.k_stages >= 4) ? 2 : 0;
        pairs = (int)(tiles < cap ? tiles : cap);
    } else {
        p.mode = 1;  // slices of (tile, stage) per pair
        pairs = (int)(p.total_units < cap ? p.total_units : cap);
    }
    if (sa == 2) {
        if (kind == KIND_F4) return run_pair<KIND_F4, 3, 8, 2, kPairMW>(ta, tb, tsa, tsb, tc, p, pairs, st);
        return run_pair<KIND_F8F6F4, 3, 16, 2, kPairMW>(ta, tb, tsa, tsb, tc, p, pairs, st);
    }
    if (kind == KIND_F4) return run_pair<KIND_F4, 6, 8>(ta, tb, tsa, tsb, tc, p, pairs, st);
    return run_pair<KIND_F8F6F4, 6>(ta, tb, tsa, tsb, tc, p, pairs, st);
}

}  // namespace

bool block_matmul_gathers_scales_fast(int a_fmt, int b_fmt, int64_t M, int64_t N, int64_t K) {
    // the swapped one-CTA kernel with two K atoms per stage (the condition on
    // `sa` in launch_block_matmul): its producer gathers row-major scale words
    // into the tensor-core tiles at about the cost of the bulk scale copies
    const bool swap = M <= 64 && N > M;
    const int64_t k_per_stage = (a_fmt == FMT_E2M1 && b_fmt == FMT_E2M1) ? 256 : 128;
    return swap && round_up(M, 16) <= 32 && K % (2 * k_per_stage) == 0;
}

cudaError_t launch_block_matmul(const GemmArgs& a, cudaStream_t st, const char** detail) {
    *detail = nullptr;
    const bool swap = a.M <= 64 && a.N > a.M;
    // MMA orientation: operand X = rows along the 128-row MMA dimension.
    const void* x_codes = swap ? a.b_codes : a.a_codes;
    const uint8_t* x_sf = swap ? a.b_scales : a.a_scales;
    const int x_fmt = swap ? a.b_fmt : a.a_fmt;
    const int64_t P = swap ? a.N : a.M;
    const void* y_codes = swap ? a.a_codes : a.b_codes;
    const uint8_t* y_sf = swap ? a.a_scales : a.b_scales;
    const int y_fmt = swap ? a.a_fmt : a.b_fmt;
    const int64_t Q = swap ? a.M : a.N;

    const int kind = (x_fmt == FMT_E2M1 && y_fmt == FMT_E2M1) ? KIND_F4 : KIND_F8F6F4;
    const int64_t k_per_stage = kind == KIND_F4 ? 256 : 128;

    if (!swap && P > 128 && Q > 128 && a.scale_layout == LAYOUT_MMA) {
        cudaError_t e = launch_pair(a, kind, x_codes, x_sf, x_fmt, P, y_codes, y_sf, y_fmt, Q, st, detail);
        if (e != cudaErrorNotSupported) return e;
    }

    int bn;
    if (swap) {
        bn = (int)round_up(Q, 16);  // 16..64
    } else {
        bn = Q > 128 ? 256 : 128;
    }

    auto fk = [&](int f) { return f == FMT_E4M3 ? 0 : (kind == KIND_F4 ? 1 : 2); };
    CUtensorMap ta, tb, tsa, tsb, tc;
    const int op3d = (a.K % k_per_stage) == 0 ? 1 : 0;
    // decode shapes stream two K atoms per stage when K allows (the stage
    // count, not the bytes, bounds them), with either scale layout; the same
    // rule tells mx_block_matmul_ws which shapes need no scale relayout
    const int sa = block_matmul_gathers_scales_fast(a.a_fmt, a.b_fmt, a.M, a.N, a.K) ? 2 : 1;
    auto opmap = [&](CUtensorMap* m, const void* codes, int64_t rows, int f, int box_rows) {
        return op3d ? make_operand_map3n(m, codes, rows, a.K, fk(f), box_rows, sa)
                    : make_operand_map(m, codes, rows, a.K, fk(f), box_rows);
    };
    const int32_t sf_groups = (int32_t)(round_up(a.K / 32, 4) / 4);
    const int gsz = (kind == KIND_F4 ? 2 : 1) * sa;
    std::memset(&tsa, 0, sizeof(tsa));
    std::memset(&tsb, 0, sizeof(tsb));
    if (!opmap(&ta, x_codes, P, x_fmt, kBlockM) || !opmap(&tb, y_codes, Q, y_fmt, bn) ||
        (a.scale_layout == LAYOUT_MMA &&
         (!make_sf_map(&tsa, x_sf, P, sf_groups, gsz, 1) || !make_sf_map(&tsb, y_sf, Q, sf_groups, gsz, (bn + 127) / 128)))) {
        *detail = "cuTensorMapEncodeTiled rejected an operand";
        return cudaErrorInvalidValue;
    }
    const bool tma_epi = (a.N % 4) == 0;
    std::memset(&tc, 0, sizeof(tc));
    if (tma_epi) {
        bool okc = swap         ? make_c_map(&tc, a.C, a.M, a.N, 32, bn, 0)
                   : bn == 256 ? make_c_map(&tc, a.C, a.M, a.N, 16, 32, 64)
                               : make_c_map(&tc, a.C, a.M, a.N, 32, 32, 128);
        if (!okc) {
            *detail = "cuTensorMapEncodeTiled rejected C";
            return cudaErrorInvalidValue;
        }
    }

    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.P = (int32_t)P;
    p.Q = (int32_t)Q;
    p.K = (int32_t)a.K;
    p.tiles_p = (int32_t)((P + kBlockM - 1) / kBlockM);
    p.tiles_q = (int32_t)((Q + bn - 1) / bn);
    p.k_stages = (int32_t)((a.K + sa * k_per_stage - 1) / (sa * k_per_stage));
    p.sf_groups = (int32_t)(round_up(a.K / 32, 4) / 4);
    p.wait_limit_ns = wait_limit_ns();
    p.idesc = make_idesc(kind, x_fmt, y_fmt, bn);
    p.swap = swap ? 1 : 0;
    p.use_tma_epi = tma_epi ? 1 : 0;
    p.epi_red_v4 = 0;  // TMA reduce-add measured faster than vector reductions on GB300
    p.C = a.C;
    p.ldc = a.N;
    p.sfa = x_sf;
    p.sfb = y_sf;
    // A load of 4-bit codes expanded to one byte each in shared memory
    // (16U4_ALIGN16B) completes with the packed byte count: 64 B per row.
    p.tx_a = (uint32_t)(sa * kBlockM) * (fk(x_fmt) == 2 ? kRowBytes / 2 : kRowBytes);
    p.tx_b = (uint32_t)(sa * bn) * (fk(y_fmt) == 2 ? kRowBytes / 2 : kRowBytes);
    p.sf_rowmajor = a.scale_layout == LAYOUT_ROWMAJOR ? 1 : 0;
    p.nb = (int32_t)(a.K / 32);
    p.op3d = op3d;
    const int64_t tiles = (int64_t)p.tiles_p * p.tiles_q;
    p.total_units = tiles * p.k_stages;
    p.group_p = band_rows(p.tiles_p, kBlockM * (x_fmt == FMT_E2M1 ? a.K / 2 : a.K));
    const int sms = sm_count();
    int grid;
    if (tiles >= sms || p.k_stages < 4) {
        p.mode = 0;
        grid = (int)(tiles < sms ? tiles : sms);
    } else {
        p.mode = 1;  // slices of (tile, stage): keeps every SM streaming
        grid = (int)(p.total_units < sms ? p.total_units : sms);
    }

#define MX_RUN(KIND_, BN_, ST_, SW_) return run<KIND_, BN_, ST_, SW_>(ta, tb, tsa, tsb, tc, p, grid, st)
#define MX_RUN2(KIND_, BN_, ST_) return run<KIND_, BN_, ST_, 1, 0, 0, 2>(ta, tb, tsa, tsb, tc, p, grid, st)
    if (sa == 2) {
        if (kind == KIND_F4) {
            if (bn == 16) MX_RUN2(KIND_F4, 16, 5);
            MX_RUN2(KIND_F4, 32, 4);
        }
        if (bn == 16) MX_RUN2(KIND_F8F6F4, 16, 5);
        MX_RUN2(KIND_F8F6F4, 32, 4);
    }
#undef MX_RUN2
    if (swap) {
        if (kind == KIND_F4) {
            if (bn == 16) MX_RUN(KIND_F4, 16, 10, 1);
            if (bn == 32) MX_RUN(KIND_F4, 32, 8, 1);
            if (bn == 48) MX_RUN(KIND_F4, 48, 6, 1);
            MX_RUN(KIND_F4, 64, 6, 1);
        } else {
            if (bn == 16) MX_RUN(KIND_F8F6F4, 16, 11, 1);
            if (bn == 32) MX_RUN(KIND_F8F6F4, 32, 9, 1);
            if (bn == 48) MX_RUN(KIND_F8F6F4, 48, 6, 1);
            MX_RUN(KIND_F8F6F4, 64, 6, 1);
        }
    }
    if (kind == KIND_F4) {
        if (bn == 128) MX_RUN(KIND_F4, 128, 4, 0);
        MX_RUN(KIND_F4, 256, 4, 0);
    }
    if (bn == 128) MX_RUN(KIND_F8F6F4, 128, 4, 0);
    MX_RUN(KIND_F8F6F4, 256, 4, 0);
#undef MX_RUN
}

// Activations quantized inside the GEMM (swapped shapes, M <= 64): the MMA A
// operand is the weights (N rows), the MMA B operand the activations, which
// each CTA quantizes once for the K stages it touches.  K is covered by as
// many launches as the resident region needs (each adds its part into C).
namespace {
template <int KIND, int BN, int STAGES, int ATOMS, int SA = 1>
cudaError_t run_act_chunks(const GemmActArgs& a, const CUtensorMap& ta, const CUtensorMap& tsa, const CUtensorMap& tc,
                           GemmParams p, int64_t total_stages, cudaStream_t st) {
    CUtensorMap none;
    std::memset(&none, 0, sizeof(none));
    const int sms = sm_count();
    constexpr int kChunk = ATOMS / SA;  // stages of SA atoms that fit the resident region
    static_assert(ATOMS % SA == 0, "whole stages in the resident region");
    for (int64_t c0 = 0; c0 < total_stages; c0 += kChunk) {
        p.k_atom0 = (int32_t)c0;
        p.k_stages = (int32_t)(total_stages - c0 < kChunk ? total_stages - c0 : kChunk);
        const int64_t tiles = (int64_t)p.tiles_p * p.tiles_q;
        p.total_units = tiles * p.k_stages;
        int grid;
        if (tiles >= sms || p.k_stages < 4) {
            p.mode = 0;
            grid = (int)(tiles < sms ? tiles : sms);
        } else {
            p.mode = 1;
            grid = (int)(p.total_units < sms ? p.total_units : sms);
        }
        cudaError_t e = run<KIND, BN, STAGES, 1, 0, ATOMS, SA>(ta, none, tsa, none, tc, p, grid, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}
}  // namespace

cudaError_t launch_block_matmul_act(const GemmActArgs& a, cudaStream_t st, const char** detail) {
    *detail = nullptr;
    const int kind = (a.act_fmt == FMT_E2M1 && a.w_fmt == FMT_E2M1) ? KIND_F4 : KIND_F8F6F4;
    const int64_t k_per_stage = kind == KIND_F4 ? 256 : 128;
    const int bn = (int)round_up(a.M, 16);  // 16..64
    auto fk = [&](int f) { return f == FMT_E4M3 ? 0 : (kind == KIND_F4 ? 1 : 2); };
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.P = (int32_t)a.N;
    p.Q = (int32_t)a.M;
    p.K = (int32_t)a.K;
    p.tiles_p = (int32_t)((a.N + kBlockM - 1) / kBlockM);
    p.tiles_q = 1;
    p.sf_groups = (int32_t)(round_up(a.K / 32, 4) / 4);
    p.wait_limit_ns = wait_limit_ns();
    p.idesc = make_idesc(kind, a.w_fmt, a.act_fmt, bn);
    p.swap = 1;
    p.use_tma_epi = (a.N % 4) == 0 ? 1 : 0;
    p.C = a.C;
    p.ldc = a.N;
    p.sfa = a.w_scales;
    // two K atoms per stage where K allows (decode shapes: the stage count
    // bounds them)
    const int sa = (bn <= 32 && a.K % (2 * k_per_stage) == 0) ? 2 : 1;
    p.tx_a = (uint32_t)(sa * kBlockM) * (fk(a.w_fmt) == 2 ? kRowBytes / 2 : kRowBytes);
    p.nb = (int32_t)(a.K / 32);
    p.group_p = p.tiles_p;
    p.op3d = (a.K % k_per_stage) == 0 ? 1 : 0;
    p.act = a.act;
    p.act_ld = a.K;
    p.act_bf16 = a.act_dtype == DT_BF16 ? 1 : 0;
    CUtensorMap ta, tsa, tc;
    std::memset(&tc, 0, sizeof(tc));
    const bool okm = p.op3d ? make_operand_map3n(&ta, a.w_codes, a.N, a.K, fk(a.w_fmt), kBlockM, sa)
                            : make_operand_map(&ta, a.w_codes, a.N, a.K, fk(a.w_fmt), kBlockM);
    if (!okm || !make_sf_map(&tsa, a.w_scales, a.N, p.sf_groups, (kind == KIND_F4 ? 2 : 1) * sa, 1) ||
        (p.use_tma_epi && !make_c_map(&tc, a.C, a.M, a.N, 32, bn, 0))) {
        *detail = "cuTensorMapEncodeTiled rejected an operand";
        return cudaErrorInvalidValue;
    }
    const int64_t total = (a.K + sa * k_per_stage - 1) / (sa * k_per_stage);
    if (sa == 2 && bn == 16 && a.act_dtype == DT_BF16) {
        // up to 16 rows of bf16, two-atom stages: activations quantized stage
        // by stage into the ring (any K in one launch).  f32 activations take
        // the resident path: a stage's f32 blocks are twice the registers of
        // bf16's, so four warps would load them in two batches per stage
        // (measured slower than the resident path on the decode shape).
        p.k_atom0 = 0;
        p.k_stages = (int32_t)total;
        const int64_t tiles = (int64_t)p.tiles_p * p.tiles_q;
        p.total_units = tiles * p.k_stages;
        const int sms = sm_count();
        int grid;
        if (tiles >= sms || p.k_stages < 4) {
            p.mode = 0;
            grid = (int)(tiles < sms ? tiles : sms);
        } else {
            p.mode = 1;
            grid = (int)(p.total_units < sms ? p.total_units : sms);
        }
        CUtensorMap none;
        std::memset(&none, 0, sizeof(none));
        if (kind == KIND_F4) return run<KIND_F4, 16, 5, 1, 0, kActStreamed, 2>(ta, none, tsa, none, tc, p, grid, st);
        return run<KIND_F8F6F4, 16, 5, 1, 0, kActStreamed, 2>(ta, none, tsa, none, tc, p, grid, st);
    }
#define MX_ACT2(KIND_, BN_, ST_, AT_) return run_act_chunks<KIND_, BN_, ST_, AT_, 2>(a, ta, tsa, tc, p, total, st)
    if (sa == 2) {
        if (kind == KIND_F4) {
            if (bn == 16) MX_ACT2(KIND_F4, 16, 3, 32);
            MX_ACT2(KIND_F4, 32, 3, 16);
        }
        if (bn == 16) MX_ACT2(KIND_F8F6F4, 16, 3, 32);
        MX_ACT2(KIND_F8F6F4, 32, 3, 16);
    }
#undef MX_ACT2
#define MX_ACT(KIND_, BN_, ST_, AT_) return run_act_chunks<KIND_, BN_, ST_, AT_>(a, ta, tsa, tc, p, total, st)
    if (kind == KIND_F4) {
        if (bn == 16) MX_ACT(KIND_F4, 16, 6, 32);
        if (bn == 32) MX_ACT(KIND_F4, 32, 6, 16);
        if (bn == 48) MX_ACT(KIND_F4, 48, 5, 12);
        MX_ACT(KIND_F4, 64, 5, 8);
    }
    if (bn == 16) MX_ACT(KIND_F8F6F4, 16, 7, 32);
    if (bn == 32) MX_ACT(KIND_F8F6F4, 32, 7, 16);
    if (bn == 48) MX_ACT(KIND_F8F6F4, 48, 6, 12);
    MX_ACT(KIND_F8F6F4, 64, 5, 8);
#undef MX_ACT
}

}  // namespace mx
