// Host-side check of the fused kernel's work schedule (schedule.cuh), compiled
// with g++ by tests/test_schedule.py. For each (m_tiles, n_tiles, k_blocks,
// sm_count, min_sk_iters, weight_bound, schedule mode) given on stdin it
// verifies that:
//   * the units of all CTAs cover every (tile, k-block) exactly once;
//   * data-parallel tiles are whole and spread round robin;
//   * for every stream-K tile, the contributor range [sk_owner(first),
//     sk_owner(last)] is exactly the set of CTAs that produced units for it,
//     each contributor has one unit for it, and units arrive in k order;
//   * workspace slots (2*c + sk_slot) of split tiles never collide;
//   * per-CTA MMA work differs by at most max(1 k-block, 1 whole tile split);
// and prints one summary line per case. Exit code 1 on any violation.
#define __host__
#define __device__
#define __forceinline__ inline
#include <cstdio>
#include <cstdlib>
#include <map>
#include <set>
#include <vector>

#include "../gemm_swiglu_mlp_gb300/csrc/schedule.cuh"

using namespace swiglu;

static int fail(const char *what, int a, int b) {
    std::printf("FAIL %s (%d, %d)\n", what, a, b);
    return 1;
}

int main() {
    int mt, nt, kb, sms, min_iters, wbound, mode;
    int bad = 0;
    while (std::scanf("%d %d %d %d %d %d %d", &mt, &nt, &kb, &sms, &min_iters, &wbound, &mode) ==
           7) {
        // modes 10..14: the wide down-projection kernel's planner (plan_down_wide)
        // with mode - 10, `sms` CTA pairs
        // mode 20: stream-K over all tiles with the grid searched for the
        // finishing cost (plan_stream_k_grid)
        // mode 30: the decode kernel's K ranges per tile (plan_decode_splits)
        // for nt tiles of kb k-blocks; wbound selects the cluster capacities:
        // 0 none (sms / j), 1 the ones measured on a 152-SM GB300 with ~225 KB
        // of shared memory per CTA. Checks: 1 <= j <= 16, j <= kb, at least
        // kDecodeMinKb k-blocks per range when split, a split's clusters fit
        // in one wave; prints "splits=j".
        if (mode == 30) {
            static const int gb300[17] = {0, 152, 76, 46, 36, 28, 23, 15, 15, 15, 13, 8, 8, 7, 7, 7, 7};
            int cap[17];
            for (int j = 0; j <= 16; ++j) cap[j] = wbound ? gb300[j] : (j ? sms / j : 0);
            const int j = plan_decode_splits(nt, kb, sms, cap, 16);
            if (j < 1 || j > 16 || j > kb) { bad |= fail("decode splits range", j, kb); continue; }
            if (j > 1 && (kb / j < kDecodeMinKb || cap[j] < nt || (long long)nt * j > sms)) {
                bad |= fail("decode split does not fit", j, nt);
                continue;
            }
            std::printf("nt=%d kb=%d sms=%d splits=%d\n", nt, kb, sms, j);
            continue;
        }
        const bool grid_search = mode == 20;
        const bool wide = mode >= 10 && !grid_search;
        if (wide) mode -= 10;
        if (grid_search) mode = kSchedStreamK;
        const WorkSched s = grid_search ? plan_stream_k_grid(mt, nt, kb, sms, 8, min_iters)
                            : wide      ? plan_down_wide(mt, nt, kb, sms, 8, min_iters, mode)
                                        : plan_schedule(mt, nt, kb, sms, 16, min_iters, wbound != 0, mode);
        const int T = mt * nt;
        if (s.grid < 1 || s.grid > sms) { bad |= fail("grid", s.grid, sms); continue; }
        if (s.sk_iters > 0 && s.dp_tiles % s.grid != 0) { bad |= fail("dp multiple", s.dp_tiles, s.grid); continue; }
        if (s.sk_iters == 0 && s.n_split == 1 && s.dp_tiles != T) { bad |= fail("dp-only must cover all tiles", s.dp_tiles, T); continue; }
        if (s.n_split != 1 && (s.sk_iters != 0 || s.dp_tiles % s.grid != 0 || (s.n_split != 2 && s.n_split != 4))) { bad |= fail("column split", s.n_split, s.dp_tiles); continue; }
        if (s.n_split == 1 && s.sk_iters != (long long)(T - s.dp_tiles) * kb) { bad |= fail("sk_iters", T, s.dp_tiles); continue; }
        if (s.sk_iters > 0 && s.sk_iters < s.grid) { bad |= fail("sk < grid", (int)s.sk_iters, s.grid); continue; }
        // the workspace counter region holds 2 counters per CTA-pair half: stream-K tiles < 2 * grid
        if (s.sk_iters > 0 && T - s.dp_tiles >= 2 * s.grid) { bad |= fail("sk tiles >= 2*grid", T - s.dp_tiles, s.grid); continue; }
        // coverage counts (tile, k-block, 32-column quarter) cells
        std::vector<int> cover((size_t)T * kb * 4, 0);
        std::map<int, std::vector<std::pair<int, int>>> contrib;  // sk tile -> (cta, kb0)
        std::vector<long long> work(s.grid, 0);
        std::set<long long> coords_seen;
        // the wide planner's aligned form (every tile cut into grid / T equal
        // K ranges): exactly one unit per pair, never two tiles
        const bool aligned = wide && s.dp_tiles == 0 && s.sk_iters > 0 && s.grid % T == 0 &&
                             s.grid > T && kb % (s.grid / T) == 0;
        for (int c = 0; c < s.grid; ++c) {
            UnitIter it;
            it.init(s, c);
            Unit u;
            int n_dp = 0, n_units = 0;
            while (it.next(u)) {
                ++n_units;
                if (u.tile < 0 || u.tile >= T || u.kb0 < 0 || u.kb1 > kb || u.kb0 >= u.kb1 ||
                    (u.width != 128 && u.width != 64 && u.width != 32) || u.sub < 0 ||
                    (u.sub + 1) * u.width > 128) {
                    bad |= fail("unit range", u.tile, u.kb0);
                    break;
                }
                if (u.width != 128 && (u.sk >= 0 || u.tile < s.dp_tiles || u.width != 128 / s.n_split))
                    bad |= fail("sub-tile outside the split tail", u.tile, u.width);
                for (int k = u.kb0; k < u.kb1; ++k)
                    for (int q = u.sub * u.width / 32; q < (u.sub + 1) * u.width / 32; ++q)
                        cover[((size_t)u.tile * kb + k) * 4 + q]++;
                // work in quarter-tile k-blocks (a 32-column sub-tile does a quarter of the MMA)
                work[c] += (long long)(u.kb1 - u.kb0) * (u.width / 32);
                if (u.sk < 0) {
                    ++n_dp;
                    if (u.kb0 != 0 || u.kb1 != kb) bad |= fail("dp not whole", u.tile, c);
                } else {
                    if (u.sk != u.tile - s.dp_tiles) bad |= fail("sk index", u.sk, u.tile);
                    contrib[u.sk].push_back({c, u.kb0});
                }
                int mb, nb;
                s.order.coords(u.tile, mb, nb);
                if (mb < 0 || mb >= mt || nb < 0 || nb >= nt) bad |= fail("coords", mb, nb);
                coords_seen.insert((long long)mb * nt + nb);
            }
            if (aligned && n_units != 1) bad |= fail("aligned split: units per pair", n_units, c);
            const int want_dp = s.dp_tiles / s.grid + (c < s.dp_tiles % s.grid ? 1 : 0);
            if (s.n_split == 1 && n_dp != want_dp) bad |= fail("dp per cta", n_dp, c);
        }
        for (size_t i = 0; i < cover.size(); ++i)
            if (cover[i] != 1) { bad |= fail("coverage", (int)(i / kb / 4), cover[i]); break; }
        if ((int)coords_seen.size() != T) bad |= fail("tile order not a bijection", (int)coords_seen.size(), T);
        std::set<int> slots_used;
        int split_tiles = 0, max_contrib = 0;
        for (auto &kv : contrib) {
            const long long st = kv.first;
            const int lo = s.sk_owner(st * kb), hi = s.sk_owner(st * kb + kb - 1);
            const auto &v = kv.second;
            if ((int)v.size() != hi - lo + 1) { bad |= fail("contributor count", (int)v.size(), hi - lo + 1); continue; }
            for (int i = 0; i < (int)v.size(); ++i) {
                if (v[i].first != lo + i) bad |= fail("contributor order", v[i].first, lo + i);
                if (i > 0 && v[i].second <= v[i - 1].second) bad |= fail("k order", v[i].second, v[i - 1].second);
            }
            if (hi > lo) {
                ++split_tiles;
                for (int c = lo; c <= hi; ++c) {
                    const int slot = 2 * c + s.sk_slot(c, st);
                    if (!slots_used.insert(slot).second) bad |= fail("slot collision", slot, (int)st);
                }
            }
            if (hi - lo + 1 > max_contrib) max_contrib = hi - lo + 1;
        }
        long long wmin = work[0], wmax = work[0];
        for (long long w : work) { wmin = w < wmin ? w : wmin; wmax = w > wmax ? w : wmax; }
        // stream-K: balanced to one k-block (4 quarter units); data-parallel:
        // to one whole tile, and (automatic choice) only when the grid is used
        // at least 85% or the tiles fill at least half of it;
        // column-split tail: to one sub-tile
        if (s.sk_iters > 0 && wmax - wmin > 4) bad |= fail("imbalance", (int)wmin, (int)wmax);
        if (s.sk_iters == 0 && s.n_split == 1) {
            if (wmax - wmin > 4 * kb) bad |= fail("dp imbalance", (int)wmin, (int)wmax);
            const int waves = (T + sms - 1) / sms;
            if (!wide && mode == kSchedAuto && T < 0.85 * waves * sms && 2 * T < sms)
                bad |= fail("dp chosen below threshold", T, waves * sms);
        }
        if (s.n_split > 1 && wmax - wmin > 4 * kb / s.n_split) bad |= fail("split imbalance", (int)wmin, (int)wmax);
        std::printf("mt=%d nt=%d kb=%d sms=%d grid=%d dp=%d sk_iters=%lld n_split=%d split=%d max_contrib=%d work=[%lld,%lld]\n",
                    mt, nt, kb, sms, s.grid, s.dp_tiles, s.sk_iters, s.n_split, split_tiles, max_contrib, wmin, wmax);
    }
    return bad;
}
