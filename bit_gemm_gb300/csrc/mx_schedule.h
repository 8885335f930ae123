// mx_schedule.h -- how the GEMM kernels hand out work to their persistent
// workers (a CTA, or a CTA pair).  Host- and device-compilable, so the CPU
// tests can check that every schedule covers each (tile, K stage) exactly
// once.
//
// The parameter type P supplies tiles_p, tiles_q (row and column tiles),
// k_stages (pipeline stages of K per tile), total_units (tiles * k_stages),
// group_p (row tiles per band) and mode:
//   0  whole tiles round-robin over the workers, in bands (below);
//   1  each worker a contiguous, equal slice of the (tile, stage) space
//      (few tiles, long K: partial sums meet in C through a reduce-add);
//   2  whole tiles for every full round, then the tiles of the last partial
//      round cut into equal (tile, stage) slices over all workers.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define MX_HD __host__ __device__ __forceinline__
#else
#define MX_HD inline
#endif

namespace mx {

struct Work {
    int32_t tp, tq, kb0, kb1;  // row tile, column tile, K stages [kb0, kb1)
};

// Tile index -> (row tile, column tile) in bands of group_p row tiles: within
// a band the row tile varies fastest, so the band's A rows stay in L2 while
// its column tiles stream past.
template <class P>
MX_HD void banded_tile(const P& p, int64_t tile, Work& w) {
    const int64_t band_tiles = (int64_t)p.group_p * p.tiles_q;
    const int64_t band = tile / band_tiles;
    const int64_t r = tile - band * band_tiles;
    const int64_t left = (int64_t)p.tiles_p - band * p.group_p;
    const int64_t rows_in_band = left < p.group_p ? left : (int64_t)p.group_p;
    w.tp = (int32_t)(band * p.group_p + r % rows_in_band);
    w.tq = (int32_t)(r / rows_in_band);
}

// The iter-th unit of work of worker `id` of `count`; false past the last.
// Identical in every role of a worker, and a pure function of its arguments.
template <class P>
MX_HD bool get_work(const P& p, uint32_t id, uint32_t count, int iter, Work& w) {
    const int64_t tiles = (int64_t)p.tiles_p * p.tiles_q;
    int64_t tile;
    if (p.mode == 0) {
        tile = (int64_t)id + (int64_t)iter * count;
        if (tile >= tiles) return false;
        w.kb0 = 0;
        w.kb1 = p.k_stages;
        banded_tile(p, tile, w);
        return true;
    }
    if (p.mode == 2) {
        const int64_t rounds = tiles / count;
        if (iter < rounds) {
            tile = (int64_t)id + (int64_t)iter * count;
            w.kb0 = 0;
            w.kb1 = p.k_stages;
            banded_tile(p, tile, w);
            return true;
        }
        const int64_t first = rounds * count;
        const int64_t units = (tiles - first) * p.k_stages;
        const int64_t u0 = units * id / count;
        const int64_t u1 = units * (id + 1) / count;
        if (u0 >= u1) return false;
        const int64_t t = u0 / p.k_stages + (iter - rounds);
        const int64_t b = t * p.k_stages > u0 ? t * p.k_stages : u0;
        const int64_t e = (t + 1) * p.k_stages < u1 ? (t + 1) * p.k_stages : u1;
        if (b >= e) return false;
        w.kb0 = (int32_t)(b - t * p.k_stages);
        w.kb1 = (int32_t)(e - t * p.k_stages);
        banded_tile(p, first + t, w);
        return true;
    }
    if (p.total_units < ((int64_t)1 << 31) && count < 65536u) {
        // mode 1 in 32-bit arithmetic (the decode path runs this before its
        // first load; 64-bit division is a long software sequence):
        // floor(units * id / count) = q id + floor(r id / count), r id < count^2
        const uint32_t units = (uint32_t)p.total_units, ks = (uint32_t)p.k_stages;
        const uint32_t q = units / count, r = units % count;
        const uint32_t u0 = q * id + r * id / count;
        const uint32_t u1 = q * (id + 1) + r * (id + 1) / count;
        if (u0 >= u1) return false;
        const uint32_t t = u0 / ks + (uint32_t)iter;
        const uint32_t b = t * ks > u0 ? t * ks : u0;
        const uint32_t e = (t + 1) * ks < u1 ? (t + 1) * ks : u1;
        if (b >= e) return false;
        w.kb0 = (int32_t)(b - t * ks);
        w.kb1 = (int32_t)(e - t * ks);
        w.tp = (int32_t)(t % (uint32_t)p.tiles_p);
        w.tq = (int32_t)(t / (uint32_t)p.tiles_p);
        return true;
    }
    const int64_t u0 = p.total_units * id / count;
    const int64_t u1 = p.total_units * (id + 1) / count;
    if (u0 >= u1) return false;
    tile = u0 / p.k_stages + iter;
    const int64_t b = tile * p.k_stages > u0 ? tile * p.k_stages : u0;
    const int64_t e = (tile + 1) * p.k_stages < u1 ? (tile + 1) * p.k_stages : u1;
    if (b >= e) return false;
    w.kb0 = (int32_t)(b - tile * p.k_stages);
    w.kb1 = (int32_t)(e - tile * p.k_stages);
    w.tp = (int32_t)(tile % p.tiles_p);
    w.tq = (int32_t)(tile / p.tiles_p);
    return true;
}

}  // namespace mx
