// Host-side check of the GEMM work schedule (mx_schedule.h): for each case,
// every (tile, K stage) is handed to exactly one worker, every unit of work
// lies inside the problem, and in slice mode each worker's units, taken in
// order, continue exactly where the previous worker's ended.
// Built and run by test_schedule.py; prints "ok" and exits 0 on success.
#include <cstdio>
#include <vector>

#include "mx_schedule.h"

struct Params {
    int32_t tiles_p, tiles_q, k_stages, mode, group_p;
    int64_t total_units;
};

static int fail(const char* what, const Params& p, unsigned count) {
    std::printf("FAIL %s: tiles %d x %d, k_stages %d, mode %d, group %d, workers %u\n", what, p.tiles_p,
                p.tiles_q, p.k_stages, p.mode, p.group_p, count);
    return 1;
}

// modes 0, 1, 2 on a problem small enough to mark every unit
static int cover(int32_t tp, int32_t tq, int32_t ks, int32_t mode, int32_t group, unsigned count) {
    Params p{tp, tq, ks, mode, group, (int64_t)tp * tq * ks};
    std::vector<int> seen((size_t)p.total_units, 0);
    for (unsigned id = 0; id < count; ++id) {
        mx::Work w;
        for (int it = 0; mx::get_work(p, id, count, it, w); ++it) {
            if (w.tp < 0 || w.tp >= tp || w.tq < 0 || w.tq >= tq || w.kb0 < 0 || w.kb0 >= w.kb1 || w.kb1 > ks)
                return fail("unit outside the problem", p, count);
            for (int kb = w.kb0; kb < w.kb1; ++kb) ++seen[((size_t)w.tp * tq + w.tq) * ks + kb];
        }
    }
    for (int v : seen)
        if (v != 1) return fail(v ? "unit handed out twice" : "unit never handed out", p, count);
    return 0;
}

// slice mode: worker id's units continue where worker id - 1's ended
static int slices(int32_t tp, int32_t tq, int32_t ks, unsigned count) {
    Params p{tp, tq, ks, 1, 1, (int64_t)tp * tq * ks};
    int64_t next = 0;
    for (unsigned id = 0; id < count; ++id) {
        mx::Work w;
        for (int it = 0; mx::get_work(p, id, count, it, w); ++it) {
            if (w.tp < 0 || w.tp >= tp || w.tq < 0 || w.tq >= tq || w.kb0 < 0 || w.kb0 >= w.kb1 || w.kb1 > ks)
                return fail("unit outside the problem", p, count);
            const int64_t tile = (int64_t)w.tq * tp + w.tp;
            if (tile * ks + w.kb0 != next) return fail("slices not contiguous", p, count);
            next = tile * ks + w.kb1;
        }
    }
    if (next != p.total_units) return fail("slices do not reach the end", p, count);
    return 0;
}

int main() {
    int bad = 0;
    // whole tiles, banded
    bad += cover(32, 32, 4, 0, 8, 148);
    bad += cover(5, 7, 3, 0, 3, 148);
    bad += cover(9, 4, 2, 0, 4, 3);
    bad += cover(1, 1, 1, 0, 1, 1);
    // slices of (tile, stage)
    bad += cover(112, 1, 16, 1, 1, 152);
    bad += cover(3, 2, 5, 1, 1, 152);   // fewer units than workers
    bad += cover(1, 1, 1, 1, 1, 152);
    bad += cover(7, 5, 33, 1, 1, 152);
    bad += cover(1000, 3, 17, 1, 1, 148);
    // whole tiles for the full rounds, the last partial round in slices
    bad += cover(10, 8, 16, 2, 4, 76);
    bad += cover(17, 13, 9, 2, 5, 76);
    bad += cover(32, 32, 32, 2, 16, 76);
    bad += cover(3, 3, 4, 2, 2, 4);
    // slice mode on both sides of the 32-bit fast path (2^31 units)
    bad += slices(112, 1, 16, 152);
    bad += slices(97, 89, 101, 151);
    bad += slices(1 << 16, 1 << 7, 1 << 8, 152);        // exactly 2^31 units: 64-bit path
    bad += slices((1 << 16) - 1, 1 << 7, 1 << 8, 152);  // just below: 32-bit path
    if (bad) return 1;
    std::printf("ok\n");
    return 0;
}
