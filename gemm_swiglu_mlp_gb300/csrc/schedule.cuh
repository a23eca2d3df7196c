// Work schedule of one fused launch over a persistent grid (host + device).
//
// Tiles are 128 token rows x 128 output columns (one UMMA N=256 covers their
// Gate and Up columns). With T tiles, kb k-blocks per tile and G persistent
// CTAs:
//   * data-parallel part: tiles [0, dp_tiles) run whole, round robin (when a
//     stream-K part follows, dp_tiles is a multiple of G, so every CTA gets
//     the same number of them);
//   * stream-K part: the k-block iterations of tiles [dp_tiles, T) form one
//     space of sk_iters = (T - dp_tiles) * kb iterations, cut into G
//     contiguous ranges whose lengths differ by at most one. A tile whose
//     iterations span several CTAs' ranges is summed through a workspace
//     (fused_up_kernel.cuh, split epilogue).
//   * or, instead of stream-K, a column-split tail: the tiles past the last
//     full wave run as 2 or 4 sub-tiles of 64 or 32 columns each, round
//     robin (plan_schedule below says which, when).
#pragma once

#include <cstdint>

namespace swiglu {

// Persistent tile order: tiles are visited in groups of `group_m` row-tiles;
// inside a group the row-tile index runs fastest, so the CTAs working at the
// same time share a few weight blocks and a bounded slab of A in L2.
struct TileOrder {
    int m_tiles;
    int n_tiles;
    int group_m;
    __host__ __device__ __forceinline__ void coords(int t, int &mb, int &nb) const {
        const int per_group = group_m * n_tiles;
        const int g = t / per_group;
        const int first_m = g * group_m;
        const int gm = (group_m < m_tiles - first_m) ? group_m : (m_tiles - first_m);
        const int idx = t - g * per_group;
        nb = idx / gm;
        mb = first_m + idx % gm;
    }
};

struct WorkSched {
    int num_tiles;
    int k_blocks;
    int grid;
    int dp_tiles;        // a multiple of grid whenever sk_iters > 0 or n_split > 1
    long long sk_iters;  // (num_tiles - dp_tiles) * k_blocks; >= grid when > 0
    int n_split;         // 1, or: tiles [dp_tiles, num_tiles) run as n_split
                         // column sub-tiles of 128 / n_split columns each
    TileOrder order;

    // first stream-K iteration of CTA c (c = grid gives sk_iters)
    __host__ __device__ __forceinline__ long long sk_begin(int c) const {
        return sk_iters * c / grid;
    }
    // the CTA whose stream-K range holds iteration x
    __host__ __device__ __forceinline__ int sk_owner(long long x) const {
        return static_cast<int>(((x + 1) * grid - 1) / sk_iters);
    }
    // workspace slot (0: first stream-K tile of the CTA, 1: its last) that
    // CTA c uses for stream-K tile s
    __host__ __device__ __forceinline__ int sk_slot(int c, long long s) const {
        return (sk_begin(c) / k_blocks == s) ? 0 : 1;
    }
};

struct Unit {
    int tile;   // linear tile index in TileOrder
    int kb0;    // k-block range [kb0, kb1)
    int kb1;
    int sk;     // stream-K tile index (tile - dp_tiles), or -1 for a data-parallel tile
    int width;  // output columns of this unit: 128, or 128 / n_split for a sub-tile
    int sub;    // which sub-tile of the 128-column tile (columns sub*width ..)
};

// A CTA's units in execution order: its data-parallel tiles, then the pieces
// of its stream-K range (one unit per tile it touches).
struct UnitIter {
    int k_blocks, grid, dp_tiles;
    int dp_next;
    int n_split, ns_next, ns_units;  // column sub-tiles of the tail
    long long x, x_end;

    __host__ __device__ __forceinline__ void init(const WorkSched &s, int cta) {
        k_blocks = s.k_blocks;
        grid = s.grid;
        dp_tiles = s.dp_tiles;
        dp_next = cta;
        n_split = s.n_split;
        ns_next = cta;
        ns_units = s.n_split > 1 ? (s.num_tiles - s.dp_tiles) * s.n_split : 0;
        x = s.sk_begin(cta);
        x_end = s.sk_begin(cta + 1);
    }
    __host__ __device__ __forceinline__ bool next(Unit &u) {
        u.width = 128;
        u.sub = 0;
        if (dp_next < dp_tiles) {
            u.tile = dp_next;
            u.kb0 = 0;
            u.kb1 = k_blocks;
            u.sk = -1;
            dp_next += grid;
            return true;
        }
        if (ns_next < ns_units) {
            u.tile = dp_tiles + ns_next / n_split;
            u.sub = ns_next % n_split;
            u.width = 128 / n_split;
            u.kb0 = 0;
            u.kb1 = k_blocks;
            u.sk = -1;
            ns_next += grid;
            return true;
        }
        if (x >= x_end) return false;
        const long long st = x / k_blocks;
        const int k0 = static_cast<int>(x - st * k_blocks);
        const long long left = x_end - x;
        const int k1 = (k0 + left < k_blocks) ? static_cast<int>(k0 + left) : k_blocks;
        u.tile = dp_tiles + static_cast<int>(st);
        u.kb0 = k0;
        u.kb1 = k1;
        u.sk = static_cast<int>(st);
        x += k1 - k0;
        return true;
    }
};

// Host-side choice of grid and split, from how well whole tiles fill the
// grid: with W = ceil(T/G) waves the data-parallel efficiency is
// T / (W * G).
//   * >= 0.95: whole tiles round robin, nothing else.
//   * otherwise, the tiles past the last full wave may run as n_split
//     column sub-tiles (64 or 32 columns: smaller UMMA N, same k loop), which
//     shortens the last wave without any workspace. A sub-tile still loads a
//     whole A tile per k-block for a fraction of the MMA work, so where the
//     MMA feed is the limit (compute-bound shapes) a sub-tile takes nearly
//     as long as a whole tile. So on compute-bound shapes the split is taken
//     when SMs would otherwise idle outright (fewer tiles than half the
//     grid), or as halves when the halved tail still fits in one wave, where
//     it cannot lose (1.5B prefill shape: 73.5 against 73.9 us). For
//     weight-streaming shapes (`weight_bound`: few token rows, the bytes per
//     unit scale with its width) it is taken whenever it reaches 0.9.
//   * otherwise, whole tiles whenever they fill at least half the grid;
//   * otherwise (a handful of tiles: most SMs would idle) the stream-K split
//     of the k-block iterations (workspace).
// Splitting K costs a partial write and a dependent read-back at the end of
// the kernel. Measured on GB300 it costs more than an idle tail: with 0.76
// of the grid used by whole tiles (72B shape, 32 tokens) whole tiles took
// 144 us and stream-K 153 us, and on the 1.5B prefill shape stream-K of the
// last wave took 83.5 us against 73.7 us; for weight-streaming shapes a
// short last wave also loses little, as its CTAs get more bandwidth each.
// `min_sk_iters` keeps every CTA's stream-K share at a few k-blocks so tiles
// are not cut into slivers.
// Schedule choice: kSchedAuto is the rule above; the others force one form
// (for ablations and tests): whole tiles only, the column-split tail, the
// stream-K split of the last full wave plus the remainder, or the stream-K
// split of the remainder alone (the tiles past the last full wave; one more
// wave joins when the remainder gives a CTA fewer than min_sk_iters).
enum SchedMode { kSchedAuto = 0, kSchedDataParallel = 1, kSchedColumnSplit = 2,
                 kSchedStreamK = 3, kSchedStreamKTail = 4 };

inline WorkSched plan_schedule(int m_tiles, int n_tiles, int k_blocks, int sm_count,
                               int group_m, int min_sk_iters = 4, bool weight_bound = false,
                               int mode = kSchedAuto) {
    WorkSched s{};
    s.num_tiles = m_tiles * n_tiles;
    s.k_blocks = k_blocks;
    s.n_split = 1;
    s.order.m_tiles = m_tiles;
    s.order.n_tiles = n_tiles;
    s.order.group_m = group_m < m_tiles ? group_m : m_tiles;
    const int T = s.num_tiles, G = sm_count;
    const int waves = (T + G - 1) / G;
    const double eff_dp = static_cast<double>(T) / (static_cast<double>(waves) * G);
    const int full = (T / G) * G;   // tiles in complete waves
    const int tail = T - full;
    if (mode == kSchedDataParallel || (mode != kSchedAuto && tail == 0)) {
        s.grid = T < G ? T : G;
        s.dp_tiles = T;
        s.sk_iters = 0;
        return s;
    }
    if (mode == kSchedStreamKTail && full > 0) {
        s.grid = G;
        s.dp_tiles = full;
        if (static_cast<long long>(tail) * k_blocks <
            static_cast<long long>(G) * (min_sk_iters > 0 ? min_sk_iters : 1))
            s.dp_tiles -= G;
        s.sk_iters = static_cast<long long>(T - s.dp_tiles) * k_blocks;
        return s;
    }
    if ((mode == kSchedAuto && eff_dp < 0.95 && tail > 0) || mode == kSchedColumnSplit) {
        int best = 1;
        double best_eff = eff_dp;
        for (int split = 2; split <= 4; split *= 2) {
            const int units = tail * split;
            const double t = static_cast<double>(full / G) +
                             static_cast<double>((units + G - 1) / G) / split;
            const double e = (static_cast<double>(T) / G) / t;
            if (e > best_eff + 1e-9) {
                best = split;
                best_eff = e;
            }
        }
        bool take = weight_bound ? best_eff >= 0.9 : (best_eff >= 0.85 && 2 * T < G);
        if (!weight_bound && !take && mode == kSchedAuto && full > 0 && 2 * tail <= G) {
            best = 2;   // the halved tail fits in one wave
            take = true;
        }
        if (mode == kSchedColumnSplit && best == 1) best = 2;
        if (best > 1 && (take || mode == kSchedColumnSplit)) {
            s.grid = G;
            s.dp_tiles = full;
            s.n_split = best;
            s.sk_iters = 0;
            return s;
        }
    }
    if (mode == kSchedAuto && 2 * T >= G) {
        // data-parallel: every tile whole, no workspace
        s.grid = T < G ? T : G;
        s.dp_tiles = T;
        s.sk_iters = 0;
        return s;
    }
    const long long total = static_cast<long long>(T) * k_blocks;
    long long g = G;
    const long long max_grid = total / (min_sk_iters > 0 ? min_sk_iters : 1);
    if (g > max_grid) g = max_grid > 0 ? max_grid : 1;
    s.grid = static_cast<int>(g);
    const int full_waves = T / s.grid;
    // keep one full wave plus the remainder in the stream-K part
    s.dp_tiles = (full_waves >= 2 ? full_waves - 1 : 0) * s.grid;
    s.sk_iters = static_cast<long long>(T - s.dp_tiles) * k_blocks;
    if (s.sk_iters < s.grid) {  // tiny problem: one iteration per CTA at most
        s.grid = static_cast<int>(s.sk_iters);
    }
    return s;
}

// Stream-K over all T tiles (fewer than `workers`) with the grid chosen for
// its finishing cost: on g CTAs each takes about T*k/g k-blocks, and a tile
// whose k-blocks span n CTAs' ranges is summed through the workspace, which
// costs about kSplitFixKb k-blocks of time per extra participant (partial
// writes, an owner waiting for a partner that finishes at the same time,
// the reads back). Among g in [ceil(W/2), W], the grid minimising
// ceil(T*k/g) + kSplitFixKb * (n_max(g) - 1) wins. Measured on GB300 (the
// CTA-pair plain product, graph-replayed calls, us): 7B M=512, 28 tiles of
// 296 k-blocks: 28 pairs (no split) 85.9, 42 pairs 70.0, 56 (two per tile)
// 56.2, 64 65.6, 70 61.7, 76 64.5 -- about 12 us (~40 k-blocks) per extra
// participant; 1.5B, 48 tiles of 140 k-blocks: 48 pairs 45.0, 56 47.7, 64
// 45.2, 72 (every tile between exactly two) 42.0, 76 45.5.
constexpr int kSplitFixKb = 40;

inline WorkSched plan_stream_k_grid(int m_tiles, int n_tiles, int k_blocks, int workers,
                                    int group_m, int min_sk_iters) {
    const int T = m_tiles * n_tiles;
    WorkSched best = plan_schedule(m_tiles, n_tiles, k_blocks, workers, group_m, min_sk_iters,
                                   false, kSchedStreamK);
    if (best.sk_iters == 0 || best.dp_tiles != 0) return best;
    auto cost = [&](const WorkSched &s) {
        int n_max = 1;
        for (int t = 0; t < T; ++t) {
            const long long first = static_cast<long long>(t) * k_blocks;
            const int n = s.sk_owner(first + k_blocks - 1) - s.sk_owner(first) + 1;
            n_max = n > n_max ? n : n_max;
        }
        const long long per = (s.sk_iters + s.grid - 1) / s.grid;
        return static_cast<double>(per) + kSplitFixKb * (n_max - 1);
    };
    double best_c = cost(best);
    for (int g = workers - 1; g > T && 2 * g >= workers; --g) {
        const WorkSched s = plan_schedule(m_tiles, n_tiles, k_blocks, g, group_m, min_sk_iters,
                                          false, kSchedStreamK);
        if (s.grid != g || s.dp_tiles != 0 || s.sk_iters == 0) continue;
        const double c = cost(s);
        if (c < best_c - 1e-9) {
            best = s;
            best_c = c;
        }
    }
    return best;
}

// Schedule of the wide plain-product kernel (down_wide_kernel.cuh): T =
// m_tiles * n_tiles tiles of 256 rows x 512 output columns, k_blocks each, on
// `workers` CTA pairs. `mode`: kSchedDataParallel (whole tiles), kSchedStreamK
// (stream-K over all tiles on all pairs), kSchedStreamKTail (stream-K over
// the tiles past the last full wave, or over all of them when that remainder
// is too small to share); kSchedAligned: every tile cut into j = floor(W/T)
// equal K ranges, one per pair (j*T pairs, each one unit; falls back to
// stream-K over all tiles when T >= W or the ranges would be too short).
// Anything else: whole tiles.
constexpr int kSchedAligned = 5;

inline WorkSched plan_down_wide(int m_tiles, int n_tiles, int k_blocks, int workers, int group_m,
                                int min_sk_iters, int mode) {
    const int T = m_tiles * n_tiles;
    if (mode == kSchedAligned) {
        const int j = T < workers ? workers / T : 1;
        if (j >= 2 && k_blocks / j >= (min_sk_iters > 0 ? min_sk_iters : 1)) {
            const WorkSched s = plan_schedule(m_tiles, n_tiles, k_blocks, j * T, group_m,
                                              min_sk_iters, false, kSchedStreamK);
            if (s.grid == j * T && s.dp_tiles == 0) return s;
        }
        mode = kSchedStreamK;
    }
    if (mode == kSchedStreamK || mode == kSchedStreamKTail)
        return plan_schedule(m_tiles, n_tiles, k_blocks, workers, group_m, min_sk_iters, false,
                             mode);
    return plan_schedule(m_tiles, n_tiles, k_blocks, workers, group_m, min_sk_iters, false,
                         kSchedDataParallel);
}

// K ranges per tile of the decode down-projection kernel (down_decode_kernel
// .cuh), whose T tiles each run on one cluster of j CTAs. Candidates: the j
// whose T clusters fit at once (clusters[j] >= T, from the occupancy query;
// null: sms / j) with at least kDecodeMinKb k-blocks per range. A long weight
// stream (ranges of kDecodeStreamKb k-blocks or more) takes the smallest j
// that puts two thirds of the `sms` SMs to work: more SMs add no bandwidth
// there, and SMs left idle let the next launch's CTAs start their prologue
// early (7B, M=16, 28 tiles: j=4 24.5 us, j=5 25.4 us). Anything else takes
// the j with the most CTAs: short ranges are latency-bound (0.5B, 7 tiles
// of 76 k-blocks: j=15 8.7 us, j=16 8.3 us). 1 when T is the SM count or
// more. j <= max_splits (clusters[] has max_splits + 1 entries).
constexpr int kDecodeMinKb = 4;
constexpr int kDecodeStreamKb = 32;

inline int plan_decode_splits(long long T, int k_blocks, int sms, const int *clusters,
                              int max_splits) {
    if (T >= sms) return 1;
    const int jmax = max_splits < k_blocks ? max_splits : k_blocks;
    const long long target = (2LL * sms + 2) / 3;
    int best = 1;
    long long best_ctas = T;
    for (int j = 2; j <= jmax; ++j) {
        if (k_blocks / j < kDecodeMinKb) break;
        const int fit = clusters ? clusters[j] : sms / j;
        if (fit < T || T * j > sms) continue;
        if (T * j >= target && k_blocks / j >= kDecodeStreamKb) return j;
        if (T * j > best_ctas) {
            best = j;
            best_ctas = T * j;
        }
    }
    return best;
}

}  // namespace swiglu
