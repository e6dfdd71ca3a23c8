// split_plan.cuh -- the work schedule of the persistent tensor-core GEMM,
// including the split tail: which k-blocks of which output tile each unit (a
// CTA, or a CTA pair) runs, in what order.  Host and device share it: the
// kernel's roles walk it, the host plans it, and a host-only test checks that
// every (tile, k-block) is run exactly once.
#pragma once
#include <cstdint>
#include "gbr_internal.h"

namespace gbr {

// With T tiles on U units, the last R = T mod U tiles would run alone in a
// final round that leaves U - R units idle.  Instead their R * num_kb
// k-blocks are dealt out in equal runs to all U units, so that round takes
// run / num_kb of a tile's time; the units that share a tile combine their
// fp32 parts in the kernel.  At most kSplitMaxParts units share a tile (all
// but one add a whole tile's worth of fp32 at L2); a run is at least
// kSplitMinRun k-blocks.
constexpr int64_t kSplitMaxParts = 4;
constexpr int64_t kSplitMinRun = 4;
constexpr int64_t kSplitMinSaving = 8;   // auto: k-blocks the last round must shrink by
// Auto also wants the predicted saving, the k-blocks the last round loses,
// to be at least 1/kSplitMinGainDiv of the launch's rounds x num_kb: below
// that the measured gain is within run-to-run noise (bf16 8192^3 on 76 CTA
// pairs: 3.7% predicted, 0.8% measured), and an unsplit launch is
// deterministic bit for bit.
constexpr int64_t kSplitMinGainDiv = 20;

// One unit of work of a persistent CTA (or CTA pair): k-blocks [kb0, kb1) of
// output tile `tile`.  parts > 1: the tile is split along K among `parts`
// units, and this one holds part `part` of split tile `sk`.
struct WorkItem {
    uint32_t tile;
    int32_t kb0, kb1;
    int32_t part, parts;
    int32_t sk;
};

// Item j of a unit; false when the unit has no item j.  The producer, the MMA
// lane and the epilogue all walk this same sequence.  Whole tiles first
// (unit + i * units); then the unit's run of sk_iters consecutive k-blocks of
// the split region, in (tile, k-block) order, which meets at most two tiles
// because sk_iters < num_kb.  The units sharing split tile tl are those whose
// runs meet [tl * num_kb, (tl + 1) * num_kb).
__host__ __device__ __forceinline__ bool work_item(const GemmShape& s, uint32_t unit, uint32_t units,
                                          uint32_t j, WorkItem& w) {
    w.kb0 = 0;
    w.kb1 = s.num_kb;
    w.part = 0;
    w.parts = 1;
    w.sk = 0;
    if (s.sk_tiles == 0) {
        w.tile = unit + j * units;
        return w.tile < uint32_t(s.num_tiles);
    }
    const uint32_t n_whole = uint32_t(s.dp_tiles) / units;
    if (j < n_whole) {
        w.tile = unit + j * units;
        return true;
    }
    j -= n_whole;
    const int64_t nkb = s.num_kb, run = s.sk_iters;
    int64_t g = int64_t(unit) * run;
    const int64_t g_end = g + run < int64_t(s.sk_tiles) * nkb ? g + run : int64_t(s.sk_tiles) * nkb;
    for (uint32_t seg = 0; seg < 2 && g < g_end; ++seg) {
        const int64_t tl = g / nkb;
        const int64_t kb0 = g - tl * nkb;
        const int64_t kb1 = kb0 + (g_end - g) < nkb ? kb0 + (g_end - g) : nkb;
        if (seg == j) {
            const int64_t first = (tl * nkb) / run, last = ((tl + 1) * nkb - 1) / run;
            w.tile = uint32_t(s.dp_tiles + tl);
            w.kb0 = int32_t(kb0);
            w.kb1 = int32_t(kb1);
            w.part = int32_t(int64_t(unit) - first);
            w.parts = int32_t(last - first + 1);
            w.sk = int32_t(tl);
            return true;
        }
        g += kb1 - kb0;
    }
    return false;
}

inline int64_t split_cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Fills the split fields of `s` for `units` units (mode -1 auto: only when the
// last round shrinks by at least an eighth of a tile and by kSplitMinSaving
// k-blocks, so that small problems keep their single launch, and by at least
// 1/kSplitMinGainDiv of the whole launch; 1: whenever a tile can be split;
// 0: never).  Returns true when the launch splits.
inline bool plan_split_fields(GemmShape& s, int64_t units, int mode,
                              int64_t gain_div = kSplitMinGainDiv) {
    s.dp_tiles = s.sk_tiles = s.sk_iters = 0;
    s.sk_sum = nullptr;
    s.sk_count = nullptr;
    const int64_t T = s.num_tiles, nkb = s.num_kb;
    if (mode == 0 || s.inject.enabled || T <= 0 || nkb < 2 || units < 2) return false;
    const int64_t R = T % units;
    if (R == 0) return false;
    int64_t run = split_cdiv(R * nkb, units);
    const int64_t run_parts = split_cdiv(nkb, kSplitMaxParts - 1);
    const int64_t run_min = nkb < kSplitMinRun ? nkb : kSplitMinRun;
    if (run < run_parts) run = run_parts;
    if (run < run_min) run = run_min;
    if (run >= nkb) return false;
    if (mode < 0 && (run * 8 > nkb * 7 || nkb - run < kSplitMinSaving ||
                     (nkb - run) * gain_div < split_cdiv(T, units) * nkb))
        return false;
    s.dp_tiles = int32_t(T - R);
    s.sk_tiles = int32_t(R);
    s.sk_iters = int32_t(run);
    return true;
}

// Scratch of a split launch, all zeroed before it: `counters` words per split
// tile (an arrived and a done count per epilogue warp), padded to 256 bytes,
// then `sum_floats` fp32 per split tile (the tile's running sum).
struct SplitScratch {
    size_t counters;     // words per split tile
    size_t sum_floats;   // floats per split tile
};
inline size_t split_count_bytes(const GemmShape& s, SplitScratch k) {
    return (size_t(s.sk_tiles) * k.counters * sizeof(uint32_t) + 255u) & ~size_t(255);
}
inline size_t split_scratch_bytes(const GemmShape& s, SplitScratch k) {
    if (s.sk_tiles == 0) return 0;
    return split_count_bytes(s, k) + size_t(s.sk_tiles) * k.sum_floats * 4u;
}
// tcgen05 kernel: per CTA of the tile, 4 epilogue warps; 128 rows per CTA x 256.
inline SplitScratch umma_split_scratch(int pair) {
    return SplitScratch{size_t(pair) * 4u * 2u, size_t(kUmmaBM * pair) * size_t(kUmmaBN)};
}
// FFMA kernel: an arrival count per consumer warp per split tile, and one
// 128 x 128 fp32 slot per part (each part writes its own slot whole, so only
// the counts are zeroed).  Its parts are added in a fixed order, so a split launch is
// deterministic bit for bit, and auto splits from a predicted saving of
// 1/kSplitMinGainDivOrdered of the launch.
constexpr int64_t kSplitMinGainDivOrdered = 50;
constexpr uint32_t kFfmaMaxConsumerWarps = 16;
inline SplitScratch ffma_split_scratch() {
    return SplitScratch{kFfmaMaxConsumerWarps,
                        size_t(kSplitMaxParts) * size_t(kFfmaBM) * size_t(kFfmaBN)};
}

}  // namespace gbr
