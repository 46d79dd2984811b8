// Host-side check of the persistent schedules of the tensor-core kernels:
// make_schedule (whole tiles and stream-K split), sk_share_start and
// for_each_unit_of, the same code the kernels run, called from the host.
// For every case: each k-block of each tile is covered exactly once, units
// stay inside their tile, no unit spans more than kb_cap k-blocks, the split
// shares are in order, and counting the switch cost never makes the slowest
// worker slower than the even split does (count_switches, what the pair
// kernel's launch runs), and slowest_share agrees with the unit walk. Prints "cases N failures F".
#include <stdio.h>

#include <vector>

#include "sgemm_internal.h"
#include "tc_common.cuh"

using namespace sgemm;

static int g_failures = 0;
static void fail(const char *what, int tiles, int kbs, int slots, int mode, int p, int cap) {
    if (g_failures++ < 20)
        printf("FAIL %s: tiles %d k_blocks %d slots %d mode %d switch %d kb_cap %d\n", what, tiles, kbs, slots, mode,
               p, cap);
}

// The slowest worker's k-blocks plus `cost` per switch between split units.
static int64_t slowest(const tc::Args &a, int grid, int cost) {
    int64_t worst = 0;
    int abort_flag = 0;
    for (int w = 0; w < grid; ++w) {
        int64_t kb_total = 0, split_units = 0;
        tc::for_each_unit_of(a, &abort_flag, w, grid, [&](int tile, int kb, int ke) {
            kb_total += ke - kb;
            if (tile >= a.dp_tiles) ++split_units;
        });
        const int64_t c = kb_total + cost * (split_units > 1 ? split_units - 1 : 0);
        if (c > worst) worst = c;
    }
    return worst;
}

int main() {
    const int tiles_list[] = {1, 2, 5, 16, 20, 28, 64, 75, 76, 77, 96, 100, 256, 1000};
    const int kb_list[] = {1, 2, 3, 4, 16, 64, 128, 129, 300, 1000};
    const int slots_list[] = {7, 76, 152};
    const int modes[] = {SK_AUTO, SK_DP_ONLY, SK_HYBRID, SK_ALL};
    int cases = 0;
    for (int tiles : tiles_list)
        for (int kbs : kb_list)
            for (int slots : slots_list)
                for (int mode : modes)
                    for (int cap : {0, 128})
                        for (int p : {0, 6})
                        for (bool split_all : {false, true}) {  // the FFMA kernels' policy for a partial wave
                            ++cases;
                            const Schedule s = make_schedule(tiles, kbs, slots, mode, 4, 0.25, split_all);
                            tc::Args a{};
                            a.k_blocks = kbs;
                            a.dp_tiles = s.dp_tiles;
                            a.sk_ctas = s.sk_ctas;
                            a.sk_iters = s.sk_iters;
                            a.kb_cap = cap;
                            a.sk_switch_kb = p;
                            if (s.grid < 1 || s.grid < s.sk_ctas || s.dp_tiles + s.sk_iters / kbs != tiles) {
                                fail("schedule shape", tiles, kbs, slots, mode, p, cap);
                                continue;
                            }
                            for (int i = 0; s.sk_ctas > 0 && i < s.sk_ctas; ++i)
                                if (tc::sk_share_start(a, i) > tc::sk_share_start(a, i + 1))
                                    fail("shares out of order", tiles, kbs, slots, mode, p, cap);
                            if (s.sk_ctas > 0 && (tc::sk_share_start(a, 0) != 0 ||
                                                  tc::sk_share_start(a, s.sk_ctas) != s.sk_iters))
                                fail("shares do not span the split iterations", tiles, kbs, slots, mode, p, cap);
                            std::vector<int> cover(static_cast<size_t>(tiles) * kbs, 0);
                            bool bad = false;
                            int abort_flag = 0;
                            for (int w = 0; w < s.grid; ++w)
                                tc::for_each_unit_of(a, &abort_flag, w, s.grid, [&](int tile, int kb, int ke) {
                                    if (tile < 0 || tile >= tiles || kb < 0 || ke > kbs || kb >= ke ||
                                        (cap > 0 && tile >= a.dp_tiles && ke - kb > cap)) {
                                        bad = true;
                                        return;
                                    }
                                    for (int k = kb; k < ke; ++k) ++cover[static_cast<size_t>(tile) * kbs + k];
                                });
                            for (int c : cover) bad = bad || c != 1;
                            if (bad) fail("coverage", tiles, kbs, slots, mode, p, cap);
                            if (p > 0 && cap == 0 && s.sk_ctas > 0) {
                                // What the launch runs: switches counted only where that helps.
                                tc::Args chosen = a, even = a;
                                tc::count_switches(chosen, p);
                                even.sk_switch_kb = 0;
                                if (slowest(chosen, s.grid, p) > slowest(even, s.grid, p))
                                    fail("chosen shares slower than even shares", tiles, kbs, slots, mode, p, cap);
                                if (tc::slowest_share(chosen, p) + s.dp_tiles / s.grid * kbs != slowest(chosen, s.grid, p))
                                    fail("slowest_share disagrees with the unit walk", tiles, kbs, slots, mode, p, cap);
                            }
                        }
    // The benchmark shape on the pair kernel: 96 tiles of 128 k-blocks on 76
    // pairs; the slowest pair goes from 34 k-blocks plus a switch to 36.
    {
        const Schedule s = make_schedule(96, 128, 76, SK_AUTO, 4, 0.25);
        tc::Args a{};
        a.k_blocks = 128;
        a.dp_tiles = s.dp_tiles;
        a.sk_ctas = s.sk_ctas;
        a.sk_iters = s.sk_iters;
        tc::count_switches(a, 6);
        tc::Args even = a;
        even.sk_switch_kb = 0;
        const int64_t with = slowest(a, s.grid, 6), without = slowest(even, s.grid, 6);
        printf("headline: slowest pair %lld (switch-aware) vs %lld (even) k-blocks + switches\n",
               static_cast<long long>(with), static_cast<long long>(without));
        if (!(a.sk_switch_kb == 6 && s.dp_tiles == 76 && with == 128 + 36 && without == 128 + 40))
            fail("headline shares", 96, 128, 76, 0, 6, 0);
    }
    printf("cases %d failures %d\n", cases, g_failures);
    return g_failures == 0 ? 0 : 1;
}
