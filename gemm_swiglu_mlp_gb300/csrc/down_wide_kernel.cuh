// Plain product out = A x W on CTA pairs with wide tiles, for the
// down-projection out = Y x W3 that completes the gated MLP ("Tile-Level
// Activation Overlap for Efficient LLM Inference", Section 1 Introduction and
// Figure 1: the MLP whose time the fused activation shortens).
//
// Tile: 256 rows x 512 output columns per cluster of two CTAs. Each k-block
// (64 reduction values) is two 2-SM UMMAs (tcgen05.mma.cta_group::2, M=256,
// N=256) that share the A operand: the first into TMEM columns 0..255 (output
// columns 0..255 of the tile), the second into 256..511. Each CTA loads its
// 128 rows of A (16 KB) and, for each UMMA, its 128-row half of the weight
// rows (2 x 16 KB), so one 48 KB stage feeds 1024 MMA cycles per SM where
// the 256-column tile of the CTA-pair kernel feeds 512 with 32 KB: a third
// fewer operand bytes into each SM per flop. With the same number of bytes
// in flight per SM (four stages here, six there), twice the MMA work per
// stage round trip keeps the tensor pipe fed at the SM clocks where the
// narrower tile waits on its loads.
//
// The accumulator fills all 512 TMEM columns, so there is one accumulator
// stage: the next tile's MMAs start once the epilogue has read TMEM (its TMA
// stores still drain), while the producer already loads the next tile's
// first stages. With a long reduction (the MLP's intermediate size) a tile
// lasts hundreds of k-blocks and the exposed TMEM read is a small fraction.
//
// Work split (schedule.cuh, plan_down_wide): whole tiles, which the library
// picks when they fill their last wave to 90% (the extra operand bytes saved
// per flop leave more of the power cap to the SMs: a higher clock at the same
// work per cycle); or, forced for ablations, stream-K over the tiles past the
// last full wave, stream-K over all tiles, or every tile cut into equal K
// ranges. A tile split between the K ranges of pairs c_lo..c_hi is finished
// without any CTA waiting for another: its 512 accumulator columns form four
// parts of 128. Each participant CTA writes each part of its FP32 partial to
// its workspace slot and counts itself in on that part's counter; whoever
// counts in last on a part sums all participants' partials of it in k order
// (its own from TMEM) and stores the BF16 result. The participants visit the
// parts in rotated orders, so when they finish together each is last on
// about its share of the parts. A signaler warp does the counting (atomic
// add with release and acquire semantics at GPU scope) while the epilogue
// warps keep writing; when the CTA's last unit is the split tile, the
// signaler also brings the other partials of its parts into the then idle
// operand ring with bulk copies. No wait depends on another cluster, so the
// call completes whatever else occupies the GPU, and the sums do not depend
// on who finishes. (Measured: the split forms move whole 512-column FP32
// partials through L2 -- 256 KB per CTA -- and, with many tiles in flight at
// different K offsets, lose the L2 sharing of whole tiles; neither is cheaper
// than the CTA-pair kernel's 256-column split tiles on the shapes that need a
// split, so the library does not pick them.)
//
// Every wait is bounded (sm103_ptx.cuh); an abort sets both CTAs' abort
// flags, and the teardown drains loads and MMAs in flight before TMEM is
// freed, as in the CTA-pair kernel.
#pragma once

#include "epilogue.cuh"

namespace swiglu {

struct WideCfg {
    static constexpr int STAGES = 4;
    static constexpr int BM = 128;                       // rows per CTA; 256 per pair tile
    static constexpr int TILE_N = 512;                   // output columns per pair tile
    static constexpr int UMMA_M = 256;
    static constexpr int UMMA_N = 256;                   // two UMMAs per k-step
    static constexpr int A_BYTES = BM * 64 * 2;          // 16 KB
    static constexpr int BBOX_BYTES = 128 * 64 * 2;      // 16 KB: one 128-row weight box
    static constexpr int B_BYTES = 2 * BBOX_BYTES;       // this CTA's rows for both UMMAs
    static constexpr int RING_BYTES = STAGES * (A_BYTES + B_BYTES);
    static constexpr int EPI_WARPS = 4;
    static constexpr int Y_WARP_BYTES = 2 * 32 * 64 * 2; // two staged 64 x 32 output boxes
    static constexpr int PARTS = 4;                      // 128-column parts of a split tile
    static constexpr int PART_FLOATS = BM * 128;         // one part of one CTA's partial
    static constexpr int PART_BYTES = PART_FLOATS * 4;   // 64 KB
    static constexpr int SLOT_FLOATS = PARTS * PART_FLOATS;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_Y = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_Y + EPI_WARPS * Y_WARP_BYTES;
    // full x STAGES, empty x STAGES, tfull, tempty, drain, publish x PARTS
    // (one per part, so that the epilogue never runs two phases ahead of the
    // signaler on one barrier), decide, fix (bulk copies of partials), ring
    // (partials read)
    static constexpr int NUM_BARS = 2 * STAGES + 6 + PARTS;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    // producer, MMA, four epilogue warps, signaler
    static constexpr int THREADS = 64 + EPI_THREADS + 32;
    static constexpr int SIGNAL_WARP = 2 + EPI_WARPS;
    static constexpr int TMEM_COLS = 512;
    static_assert(OFF_A == 0 && OFF_B == STAGES * A_BYTES, "the ring is one block from offset 0");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Arguments of one launch: out [M, N] = A [M, K] x W [K, N], W packed as the
// down-projection weights ([KT][KB][256][64], KT = kt_tiles tiles of 256
// output columns, KB = sched.k_blocks k-blocks).
struct WideArgs {
    int M, N, K;
    int kt_tiles;
    WorkSched sched;           // over tiles of 256 rows x 512 columns
    float *partials;           // 2 slots per worker and CTA half (stream-K only)
    unsigned int *counters;    // 2 * PARTS per stream-K tile, zero between launches
#ifdef SWIGLU_TEST_FAULT_INJECTION
    int skip_first_fill;       // test build only: never fill the first pipeline stage
#endif
};

// Counter of part j of stream-K tile s for CTA half h.
__host__ __device__ __forceinline__ int wide_counter_index(int s, int j, int h) {
    return (s * WideCfg::PARTS + j) * 2 + h;
}

__device__ __forceinline__ unsigned int atom_add_acq_rel_gpu(unsigned int *p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(p), "r"(v)
                 : "memory");
    return old;
}

__global__ void __launch_bounds__(WideCfg::THREADS, 1)
    down_wide_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmOut, const WideArgs args) {
    using C = WideCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t half = rank & 1u;            // 0: leader (issues the UMMAs)
    constexpr uint32_t leader_rank = 0;
    const bool is_leader = half == 0;
    const int pair = static_cast<int>(blockIdx.x / 2);
    const WorkSched &sched = args.sched;

    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (C::STAGES + s); };
    const uint32_t tfull_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES);
    const uint32_t tempty_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 1);
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 2);
    auto pub_bar = [&](int j) { return sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 3 + j); };
    const uint32_t dec_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 3 + C::PARTS);
    const uint32_t fix_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 4 + C::PARTS);
    const uint32_t ring_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 5 + C::PARTS);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    volatile int *dec_mask = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);
    auto set_abort_both = [&]() {
        *abort_flag = 1;
        st_cluster_u32(mapa_shared(sbase + C::OFF_MISC + 4, rank ^ 1u), 1u);
    };

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, 2 * C::EPI_WARPS);   // epilogue warps of both CTAs
        mbar_init(drain_bar, 1);
        for (int j = 0; j < C::PARTS; ++j) mbar_init(pub_bar(j), C::EPI_THREADS);
        mbar_init(dec_bar, 1);
        mbar_init(fix_bar, 1);
        mbar_init(ring_bar, C::EPI_THREADS);
        *abort_flag = 0;
        *dec_mask = 0;
        fence_barrier_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmOut);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // The prologue touched no global memory: let the next launch begin, ask
    // L2 for this pair's first stages, and wait for the previous launch.
    griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        UnitIter it;
        it.init(sched, pair);
        Unit u;
        if (it.next(u)) {
            int tm, nt;
            sched.order.coords(u.tile, tm, nt);
            const int kend = (u.kb1 - u.kb0 < kPrefetchStages) ? u.kb1 : u.kb0 + kPrefetchStages;
            for (int kb = u.kb0; kb < kend; ++kb) {
                tma_prefetch_2d(&tmA, kb * 64, tm * C::UMMA_M + C::BM * static_cast<int>(half));
                tma_prefetch_3d(&tmB, 0, 128 * static_cast<int>(half),
                                2 * nt * sched.k_blocks + kb);
            }
        }
    }
    griddep_wait();

    // the stream-K participants of a unit's tile (c_lo == c_hi: not split)
    auto split_range = [&](const Unit &u, int &c_lo, int &c_hi) {
        c_lo = c_hi = pair;
        if (u.sk >= 0) {
            const long long first = static_cast<long long>(u.sk) * sched.k_blocks;
            c_lo = sched.sk_owner(first);
            c_hi = sched.sk_owner(first + sched.k_blocks - 1);
        }
    };
    // whether this CTA's units end with `u` (then the operand ring is idle
    // once u's accumulator is complete)
    auto is_last_unit = [&](const UnitIter &after) {
        UnitIter peek = after;
        Unit v;
        return !peek.next(v);
    };
    // slot of worker p's partial for stream-K tile s (this CTA half)
    auto slot_of = [&](int p, int s) {
        return args.partials + (static_cast<size_t>(2 * p + sched.sk_slot(p, s)) * 2 + half) *
                                   static_cast<size_t>(C::SLOT_FLOATS);
    };

    uint32_t issued_mask = 0, last_parity = 0;   // leader's drain bookkeeping

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            UnitIter it;
            it.init(sched, pair);
            Unit u;
            while (ok && it.next(u)) {
                int tm, nt;
                sched.order.coords(u.tile, tm, nt);
                const bool has1 = 2 * nt + 1 < args.kt_tiles;
                const uint32_t tx = 2u * static_cast<uint32_t>(C::A_BYTES + (has1 ? 2 : 1) * C::BBOX_BYTES);
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
#ifdef SWIGLU_TEST_FAULT_INJECTION
                    if (args.skip_first_fill && is_leader && kb == u.kb0 && stage == 0 &&
                        phase == 0) {
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
#endif
                    if (is_leader) mbar_arrive_expect_tx(full_bar(stage), tx);
                    const uint32_t bar = mapa_shared(full_bar(stage), leader_rank);
                    const uint32_t b_dst = sbase + C::OFF_B + stage * C::B_BYTES;
                    tma_load_2d_pair(sbase + C::OFF_A + stage * C::A_BYTES, &tmA, bar, kb * 64,
                                     tm * C::UMMA_M + C::BM * static_cast<int>(half));
                    tma_load_3d_pair(b_dst, &tmB, bar, 0, 128 * static_cast<int>(half),
                                     2 * nt * sched.k_blocks + kb);
                    if (has1)
                        tma_load_3d_pair(b_dst + C::BBOX_BYTES, &tmB, bar, 0,
                                         128 * static_cast<int>(half),
                                         (2 * nt + 1) * sched.k_blocks + kb);
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusProducerTimeout);
                set_abort_both();
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && is_leader) {
            constexpr uint32_t idesc = idesc_bf16_f32(C::UMMA_M, C::UMMA_N);
            int stage = 0;
            uint32_t phase = 0, t_phase = 0;
            bool ok = true;
            UnitIter it;
            it.init(sched, pair);
            Unit u;
            while (ok && it.next(u)) {
                int tm, nt;
                sched.order.coords(u.tile, tm, nt);
                const bool has1 = 2 * nt + 1 < args.kt_tiles;
                if (!mbar_wait(tempty_bar, t_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = smem_desc_k128(sbase + C::OFF_A + stage * C::A_BYTES);
                    const uint64_t b0 = smem_desc_k128(sbase + C::OFF_B + stage * C::B_BYTES);
                    const uint64_t b1 =
                        smem_desc_k128(sbase + C::OFF_B + stage * C::B_BYTES + C::BBOX_BYTES);
#pragma unroll
                    for (int k = 0; k < kKSteps; ++k) {
                        const uint32_t acc = (kb != u.kb0 || k != 0) ? 1u : 0u;
                        umma_bf16_pair(tmem_base, a_desc + 2u * k, b0 + 2u * k, idesc, acc);
                        if (has1)
                            umma_bf16_pair(tmem_base + C::UMMA_N, a_desc + 2u * k, b1 + 2u * k,
                                           idesc, acc);
                    }
                    umma_commit_pair_mc(empty_bar(stage), 0x3);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(tfull_bar, 0x3);
                t_phase ^= 1u;
            }
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusMmaTimeout);
                set_abort_both();
            }
        }
    } else if (warp < C::SIGNAL_WARP) {
        // ---- epilogue: one thread per accumulator row
        const int quad = warp & 3;
        const int row_in_tile = 32 * quad + lane;
        const uint32_t ybuf = sbase + C::OFF_Y + (warp - 2) * C::Y_WARP_BYTES;
        const uint32_t tempty_leader = mapa_shared(tempty_bar, leader_rank);
        uint32_t t_phase = 0, dec_phase = 0, fix_phase = 0;
        bool ok = true;
        UnitIter it;
        it.init(sched, pair);
        Unit u;
        while (ok && it.next(u)) {
            int tm, nt;
            sched.order.coords(u.tile, tm, nt);
            const bool has1 = 2 * nt + 1 < args.kt_tiles;
            const int nparts = has1 ? C::PARTS : C::PARTS / 2;
            ok = epilogue_all(mbar_wait(tfull_bar, t_phase, abort_flag, 2 * kWaitLimitCycles));
            if (!ok) break;
            t_phase ^= 1u;
            tc_fence_after();
            const int row0 = tm * C::UMMA_M + C::BM * static_cast<int>(half) + 32 * quad;
            const bool rows_live = row0 < args.M;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * quad) << 16);
            const int col0 = nt * C::TILE_N;
            int c_lo, c_hi;
            split_range(u, c_lo, c_hi);

            // BF16 output of accumulator part j (128 columns) from registers
            // already summed: staged in the warp's two boxes, stored by TMA
            auto store_part = [&](int j) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    store_staged_boxes(&tmOut, ybuf, col0 + 128 * j, row0, 2, args.N);
                    bulk_commit_group();
                }
            };

            if (c_lo == c_hi) {
                for (int j = 0; j < nparts; ++j) {
                    if (rows_live) {
                        if (lane == 0) bulk_wait_group_read0();
                        __syncwarp();
                        stage_plain_128(tbase + 128 * j, ybuf, lane);
                    }
                    if (j == nparts - 1) {
                        // TMEM read: the next unit's MMAs may start
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(tempty_leader);
                    }
                    if (rows_live) store_part(j);
                }
                continue;
            }

            // ---- a split tile: publish every part, finish those counted last
            const int n = c_hi - c_lo + 1;
            const int start = ((pair - c_lo) * nparts) / n;
            float *mine = slot_of(pair, u.sk);
            for (int q = 0; q < nparts; ++q) {
                const int j = (start + q) % nparts;
                if (rows_live) {
                    float *dst = mine + static_cast<size_t>(j) * C::PART_FLOATS;
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(tbase + 128 * j + 32 * c4, r);
                        tmem_ld_wait();
                        reg_fence32(r);
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            __stcg(reinterpret_cast<float4 *>(dst) + (8 * c4 + g) * C::BM + row_in_tile,
                                   make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                               __uint_as_float(r[4 * g + 2]),
                                               __uint_as_float(r[4 * g + 3])));
                    }
                }
                mbar_arrive(pub_bar(j));   // release: this thread's part j is written
            }
            ok = epilogue_all(mbar_wait(dec_bar, dec_phase, abort_flag));
            if (!ok) break;
            dec_phase ^= 1u;
            const int mask = *dec_mask;
            // the other participants' partials: in the operand ring (bulk
            // copies, batches of parts that fit) or read from global memory
            const int others = n - 1;
            const bool ring_path =
                is_last_unit(it) && others * C::PART_BYTES <= C::RING_BYTES;
            const int per_batch = ring_path ? C::RING_BYTES / (others * C::PART_BYTES) : 1;
            int in_batch = 0;
            for (int j = 0; j < nparts && ok; ++j) {
                if (!((mask >> j) & 1)) continue;
                if (ring_path && in_batch == 0) {
                    ok = epilogue_all(mbar_wait(fix_bar, fix_phase, abort_flag));
                    if (!ok) break;
                    fix_phase ^= 1u;
                }
                if (rows_live) {
                    if (lane == 0) bulk_wait_group_read0();
                    __syncwarp();
#pragma unroll 1
                    for (int c4 = 0; c4 < 4; ++c4) {
                        float x[32];
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(tbase + 128 * j + 32 * c4, r);
                        tmem_ld_wait();
                        reg_fence32(r);
                        int idx = 0;   // index among the other participants
                        for (int p = c_lo; p <= c_hi; ++p) {
                            float v[32];
                            if (p == pair) {
#pragma unroll
                                for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
                            } else {
                                const float4 *src;
                                if (ring_path) {
                                    src = reinterpret_cast<const float4 *>(
                                        smem + (static_cast<size_t>(in_batch) * others + idx) *
                                                   C::PART_BYTES);
                                } else {
                                    src = reinterpret_cast<const float4 *>(
                                        slot_of(p, u.sk) + static_cast<size_t>(j) * C::PART_FLOATS);
                                }
#pragma unroll
                                for (int g = 0; g < 8; ++g) {
                                    const float4 w = ring_path
                                                         ? src[(8 * c4 + g) * C::BM + row_in_tile]
                                                         : __ldcg(src + (8 * c4 + g) * C::BM +
                                                                  row_in_tile);
                                    v[4 * g] = w.x;
                                    v[4 * g + 1] = w.y;
                                    v[4 * g + 2] = w.z;
                                    v[4 * g + 3] = w.w;
                                }
                                ++idx;
                            }
                            // k order: the lowest participant's partial first
#pragma unroll
                            for (int e = 0; e < 32; ++e) x[e] = (p == c_lo) ? v[e] : x[e] + v[e];
                        }
                        stage_bf16x32(ybuf, lane, 32 * c4, x);
                    }
                    store_part(j);
                }
                if (ring_path && ++in_batch == per_batch) {
                    in_batch = 0;
                    mbar_arrive(ring_bar);   // this batch's ring copies are read
                }
            }
            if (!ok) break;
            if (ring_path && in_batch != 0) mbar_arrive(ring_bar);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader);
        }
        if (lane == 0) {
            bulk_wait_group_read0();
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusEpilogueTimeout);
                set_abort_both();
            }
        }
    } else if (lane == 0 && sched.sk_iters > 0) {
        // ---- signaler: counts this CTA in on each part of its split tiles
        // and, as the last to count in on a part, fetches the other partials
        uint32_t pub_phases = 0;   // one parity bit per part
        uint32_t t_phase = 0, fix_phase = 0, ring_phase = 0;
        bool ok = true;
        UnitIter it;
        it.init(sched, pair);
        Unit u;
        while (ok && it.next(u)) {
            // follow the accumulator unit by unit (each wait is bounded by
            // one unit's duration, not by all the whole tiles before a split)
            if (!mbar_wait(tfull_bar, t_phase, abort_flag, 2 * kWaitLimitCycles)) {
                ok = false;
                break;
            }
            t_phase ^= 1u;
            int c_lo, c_hi;
            split_range(u, c_lo, c_hi);
            if (c_lo == c_hi) continue;
            int tm, nt;
            sched.order.coords(u.tile, tm, nt);
            const bool has1 = 2 * nt + 1 < args.kt_tiles;
            const int nparts = has1 ? C::PARTS : C::PARTS / 2;
            const int n = c_hi - c_lo + 1;
            const int start = ((pair - c_lo) * nparts) / n;
            int mask = 0;
            for (int q = 0; q < nparts; ++q) {
                const int j = (start + q) % nparts;
                if (!mbar_wait(pub_bar(j), (pub_phases >> j) & 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                pub_phases ^= 1u << j;
                unsigned int *ctr = args.counters + wide_counter_index(u.sk, j, half);
                if (atom_add_acq_rel_gpu(ctr, 1u) == static_cast<unsigned int>(n - 1)) {
                    mask |= 1 << j;
                    *ctr = 0u;   // every participant is in: ready for the next launch
                }
            }
            if (!ok) break;
            *dec_mask = mask;
            mbar_arrive(dec_bar);
            const int others = n - 1;
            const bool ring_path = is_last_unit(it) && others * C::PART_BYTES <= C::RING_BYTES;
            if (!ring_path || mask == 0) continue;
            // partials written by the other CTAs (generic proxy), read by bulk
            // copies (async proxy) after the acquiring atomics above
            fence_proxy_async_global();
            const int per_batch = C::RING_BYTES / (others * C::PART_BYTES);
            int in_batch = 0, batches = 0;
            for (int j = 0; j < nparts && ok; ++j) {
                if (!((mask >> j) & 1)) continue;
                if (in_batch == 0) {
                    if (batches > 0) {
                        // the epilogue has read the previous batch
                        if (!mbar_wait(ring_bar, ring_phase, abort_flag)) {
                            ok = false;
                            break;
                        }
                        ring_phase ^= 1u;
                    }
                    int cnt = 0;
                    for (int jj = j; jj < nparts && cnt < per_batch; ++jj)
                        if ((mask >> jj) & 1) ++cnt;
                    mbar_arrive_expect_tx(fix_bar, static_cast<uint32_t>(cnt * others * C::PART_BYTES));
                }
                int idx = 0;
                for (int p = c_lo; p <= c_hi; ++p) {
                    if (p == pair) continue;
                    bulk_copy_g2s(sbase + static_cast<uint32_t>((in_batch * others + idx) * C::PART_BYTES),
                                  slot_of(p, u.sk) + static_cast<size_t>(j) * C::PART_FLOATS,
                                  C::PART_BYTES, fix_bar);
                    ++idx;
                }
                if (++in_batch == per_batch) {
                    in_batch = 0;
                    ++batches;
                    // the copies land before this warp moves on (nothing is
                    // left in flight into shared memory at exit)
                    if (!mbar_wait_drain(fix_bar, fix_phase)) ok = false;
                    fix_phase ^= 1u;
                }
            }
            if (ok && in_batch != 0) {
                ++batches;
                if (!mbar_wait_drain(fix_bar, fix_phase)) ok = false;
                fix_phase ^= 1u;
            }
            // the epilogue's arrival for the last batch
            if (ok && !mbar_wait(ring_bar, ring_phase, abort_flag)) ok = false;
            ring_phase ^= 1u;
        }
        if (!ok && !*abort_flag) {
            atomicOr(&g_status_word, kStatusEpilogueTimeout);
            set_abort_both();
        }
    }

    // ---- teardown (as in the CTA-pair kernel)
    __syncthreads();
    cluster_sync();
    if (*abort_flag) {
        if (is_leader) {
            if (warp == 0 && lane == 0) {
                for (int s = 0; s < C::STAGES; ++s)
                    if ((issued_mask >> s) & 1u)
                        if (!mbar_wait_drain(full_bar(s), (last_parity >> s) & 1u))
                            atomicOr(&g_status_word, kStatusDrainTimeout);
            }
            if (warp == 1 && lane == 0) {
                umma_commit_pair_mc(drain_bar, static_cast<uint16_t>(1u << leader_rank));
                if (!mbar_wait_drain(drain_bar, 0)) atomicOr(&g_status_word, kStatusDrainTimeout);
            }
        }
        __syncthreads();
        cluster_sync();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace swiglu
