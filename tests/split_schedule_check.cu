// Host-only check of the persistent tensor-core GEMM's work schedule
// (split_plan.cuh), the code the kernel's roles walk.  For many tile counts,
// unit counts and k-block counts: every (tile, k-block) is run by exactly one
// unit; the units that share a split tile agree on how many they are and hold
// distinct part indices, at most kSplitMaxParts of them; a unit runs at most
// two split items; and when the planner splits, the split round is shorter
// than a whole tile.
// Prints "ok ..." and exits 0, or prints the first violation and exits 1.
#include <cstdio>
#include <cstring>
#include <map>
#include <set>
#include <vector>

#include "split_plan.cuh"

using namespace gbr;

static int fail(const char* what, int units, int T, int nkb, int mode) {
    std::printf("FAIL %s (units %d, tiles %d, k-blocks %d, mode %d)\n", what, units, T, nkb, mode);
    return 1;
}

int main() {
    long configs = 0, split_configs = 0;
    const int unit_list[] = {2, 3, 7, 64, 76, 152};
    const int tile_list[] = {1, 2, 3, 5, 36, 63, 75, 76, 77, 100, 151, 152, 153, 256, 1024, 1120};
    const int kb_list[] = {0, 1, 2, 3, 4, 5, 7, 8, 31, 32, 64, 100, 128};
    for (int units : unit_list)
        for (int T : tile_list)
            for (int nkb : kb_list)
                for (int mode_gd = 0; mode_gd < 6; ++mode_gd) {
                    const int mode = mode_gd % 3 - 1;
                    const int64_t gain_div = mode_gd < 3 ? kSplitMinGainDiv : kSplitMinGainDivOrdered;
                    GemmShape s;
                    std::memset(&s, 0, sizeof(s));
                    s.num_tiles = T;
                    s.num_kb = nkb;
                    const bool split = plan_split_fields(s, units, mode, gain_div);
                    ++configs;
                    split_configs += split;
                    if (split != (s.sk_tiles > 0)) return fail("plan flag", units, T, nkb, mode);
                    if (split && (s.sk_iters >= nkb ||
                                  s.dp_tiles % units != 0 || s.dp_tiles + s.sk_tiles != T))
                        return fail("plan fields", units, T, nkb, mode);
                    std::vector<int> cover(size_t(T) * (nkb > 0 ? nkb : 1), 0);
                    std::map<int, std::set<int>> parts_seen;   // split tile -> part slots
                    std::map<int, std::set<int>> parts_count;  // split tile -> declared counts
                    int longest_split_run = 0;
                    for (int u = 0; u < units; ++u) {
                        int split_items = 0, split_run = 0;
                        for (uint32_t j = 0;; ++j) {
                            if (j > uint32_t(T) + 4) return fail("runaway item index", units, T, nkb, mode);
                            WorkItem w;
                            if (!work_item(s, uint32_t(u), uint32_t(units), j, w)) break;
                            if (w.tile >= uint32_t(T)) return fail("tile out of range", units, T, nkb, mode);
                            if (nkb == 0) {
                                if (w.kb0 != 0 || w.kb1 != 0) return fail("k range with K = 0", units, T, nkb, mode);
                                cover[w.tile] += 1;
                                continue;
                            }
                            if (!(0 <= w.kb0 && w.kb0 < w.kb1 && w.kb1 <= nkb))
                                return fail("k range", units, T, nkb, mode);
                            for (int kb = w.kb0; kb < w.kb1; ++kb) cover[size_t(w.tile) * nkb + kb] += 1;
                            if (w.parts > 1) {
                                ++split_items;
                                split_run += w.kb1 - w.kb0;
                                if (w.tile < uint32_t(s.dp_tiles) || w.sk != int(w.tile) - s.dp_tiles)
                                    return fail("split item outside the split region", units, T, nkb, mode);
                                if (w.part < 0 || w.part >= w.parts || w.parts > kSplitMaxParts)
                                    return fail("part slot", units, T, nkb, mode);
                                if (!parts_seen[w.sk].insert(w.part).second)
                                    return fail("part slot taken twice", units, T, nkb, mode);
                                parts_count[w.sk].insert(w.parts);
                            } else if (w.kb0 != 0 || w.kb1 != nkb) {
                                return fail("partial tile without parts", units, T, nkb, mode);
                            }
                        }
                        if (split_items > 2) return fail("more than two split items", units, T, nkb, mode);
                        if (split_run > longest_split_run) longest_split_run = split_run;
                    }
                    for (int c : cover)
                        if (c != 1) return fail("a (tile, k-block) not run exactly once", units, T, nkb, mode);
                    for (auto& kv : parts_seen) {
                        const auto& counts = parts_count[kv.first];
                        if (counts.size() != 1 || int(kv.second.size()) != *counts.begin())
                            return fail("units of a split tile disagree on their number", units, T, nkb, mode);
                    }
                    if (split && longest_split_run >= nkb)
                        return fail("split round not shorter than a tile", units, T, nkb, mode);
                }
    // The two auto rules on the workloads they were set for: fp32 4096^3 FFMA
    // (1024 tiles of 128 x 32 k-blocks on 152 CTAs) splits under the ordered
    // rule only; bf16 8192^3 on 76 CTA pairs (1024 tiles, 64 k-blocks of 128)
    // does not split under the tensor-core kernels' 5% rule.
    {
        GemmShape s;
        std::memset(&s, 0, sizeof(s));
        s.num_tiles = 1024;
        s.num_kb = 128;
        if (plan_split_fields(s, 152, -1)) return fail("ffma 4096 auto, 5% rule", 152, 1024, 128, -1);
        if (!plan_split_fields(s, 152, -1, kSplitMinGainDivOrdered))
            return fail("ffma 4096 auto, ordered rule", 152, 1024, 128, -1);
        s.num_kb = 64;
        if (plan_split_fields(s, 76, -1)) return fail("bf16 8192 auto", 76, 1024, 64, -1);
    }
    std::printf("ok %ld configurations, %ld split\n", configs, split_configs);
    return 0;
}
