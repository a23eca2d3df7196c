// 2-SM (CTA pair) fused SwiGLU up-projection for sm_103a.
//
// Same computation as fused_up_kernel.cuh ("Tile-Level Activation Overlap for
// Efficient LLM Inference", Section 1 Introduction: Y = SiLU(A x W1) (.)
// (A x W2), Gate and Up never written to global memory), for large M. A
// cluster of two CTAs on two SMs works on a 256-row x 128-column tile with
// one 2-SM UMMA (tcgen05.mma.cta_group::2, M=256, N=256):
//
//   * each CTA loads ITS 128 rows of A and ITS HALF of the packed weight tile
//     (leader: the 128 Gate rows, peer: the 128 Up rows) into its own
//     shared memory: 32 KB per k-block per SM instead of 48 KB, so the
//     operand traffic into each SM is two thirds of the 1-SM kernel's, and
//     six stages fit in shared memory;
//   * the leader's single MMA thread issues the UMMA; the accumulator lands
//     in both SMs' TMEM (each CTA holds its own 128 rows, all 256 Gate|Up
//     columns), so each CTA's epilogue is the 1-SM epilogue unchanged;
//   * both CTAs' TMA loads signal the leader's full barrier; the leader's
//     commits are multicast to both CTAs' empty / accumulator-full barriers;
//     both CTAs' epilogue warps arrive on the leader's accumulator-empty
//     barrier.
//
// Work split: schedule.cuh over pairs (whole pair tiles, column sub-tiles
// for the last wave, or stream-K). A tile split over the K ranges of pairs
// c_lo..c_hi (k order) is finished by its owner c_lo, whose range ends in
// it, so it is always the owner's last unit: the other contributors write
// their FP32 partials to workspace slots (slot = (2 * pair + first/last) * 2
// + half, half = 0 for the leader CTA, 1 for its peer) and count themselves
// in (counter = 2 * stream-K tile + half); the owner waits for the count
// (bounded), brings the partials into its now idle operand ring with bulk
// copies, adds them to its own accumulators in k order, activates, stores Y
// and resets the counter. Only the owner waits, on CTAs that never wait for
// it, and they finish their parts of the tile first (their range starts in
// it).
//
// Dynamic tiles: in a launch of whole tiles only and at least two waves,
// the pairs drift apart in time (some SMs are a few percent slower than
// others, so over ~100 tiles the spread grows past three tile durations):
// pairs that should share a weight tile in L2 then fetch it from DRAM at
// different times, and the fast pairs idle at the end. Such a launch hands
// out the tiles past the first wave at run time: the leader CTA's producer of
// each pair takes the next tile index from a counter in the workspace
// (atomicAdd) when it starts loading its previous tile, and publishes it in
// a small ring of tile indices in both CTAs' shared memory, which the MMA
// issuer, both CTAs' epilogue warps and the peer's producer read (tile-full
// and tile-empty mbarriers per ring slot; the index -1 ends the sequence).
// The tiles in flight are then always the lowest-numbered ones left, a
// compact window of the tile order, and every pair works until the tiles
// run out. Each tile is still computed whole by one pair in k order, so the
// result is bit-identical to the static order. The last pair to finish
// resets the counter for the next launch.
//
// Co-residency: an owner c_lo waits for pairs c_lo+1..c_hi, so those must be
// running, or done, while it waits. A launch with a K split therefore numbers
// its pairs by the order in which they start, not by cluster index: each
// pair takes a ticket t from a counter in the workspace (atomicInc wrapping
// at grid - 1, so the counter is back at its start after the launch) and
// works as pair grid - 1 - t. The pairs an owner waits for took their tickets
// before it did, so they are resident or finished, and they never wait for
// anyone of a later ticket; the wait ends whatever else shares the GPU (other
// streams, other processes) and however the clusters are dispatched.
//
// PLAIN = true: the same kernel computes a plain product out = A x W (no
// activation), the down-projection out = Y x W3 that completes the gated
// MLP. The packed weight tile then holds 256 output columns (one CTA loads
// 128 of them), the accumulator's 256 columns are those output columns, and
// the epilogue rounds them to BF16 and stores them with TMA: a whole tile in
// two passes of 128 columns through the Y staging buffer, a split tile's sum
// (its owner's last unit, when the operand ring is idle) through the last
// 64 KB of the ring. Whole tiles and stream-K only (no column sub-tiles);
// split tiles are summed exactly as above.
//
// Every wait is bounded. An abort sets the abort flag of every CTA of the
// cluster; after a cluster barrier each leader drains the loads and MMAs in
// flight (all loads into a pair complete on its leader's barriers), a second
// cluster barrier keeps the other CTAs alive until then, and all free TMEM.
#pragma once

#include "epilogue.cuh"

namespace swiglu {

constexpr int kTileRing = 8;   // slots of the dynamic tile ring

template <int STAGES>
struct PairCfg {
    static constexpr int BM = 128;                  // rows per CTA; the pair tile has 256
    static constexpr int BN = 128;                  // output columns per tile
    static constexpr int BK = 64;                   // K per stage: 128-byte rows
    static constexpr int UMMA_M = 256;
    static constexpr int UMMA_N = 2 * BN;           // Gate | Up
    static constexpr int UMMA_K = 16;
    static constexpr int A_BYTES = BM * BK * 2;     // 16 KB: this CTA's A rows
    static constexpr int B_BYTES = BN * BK * 2;     // 16 KB: this CTA's half of Gate|Up
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_WARPS = 4;
    static constexpr int Y_HALF_BYTES = 32 * 64 * 2;
    static constexpr int Y_WARP_BYTES = 2 * Y_HALF_BYTES;
    static constexpr int TMEM_COLS = 2 * UMMA_N;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_Y = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_Y + EPI_WARPS * Y_WARP_BYTES;
    // full, empty, tfull x2, tempty x2, drain, fixup (split-tile partials),
    // tile-ring full, tile-ring empty
    static constexpr int NUM_BARS = 2 * STAGES + 6 + 2 * kTileRing;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_RING = OFF_MISC + 16;           // kTileRing tile indices
    static constexpr int SMEM_BYTES = OFF_RING + 4 * kTileRing + 1024;
    // readers of a ring slot: the MMA issuer, the peer's producer and both
    // CTAs' epilogue warps, all arriving on the leader's tile-empty barrier
    static constexpr int RING_READERS = 2 + 2 * EPI_WARPS;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static_assert(TMEM_COLS == 512, "two 256-column accumulator stages fill TMEM");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(UMMA_N == kSlotCols, "workspace slot shape");
};

// IL: column-interleaved packed weights (see fused_up_kernel.cuh); a CTA's
// half of a unit's weight rows is then the unit's first or second half of
// its 2 * width packed rows.
template <int STAGES, typename E, bool PLAIN = false, bool IL = false>
__global__ void __launch_bounds__(PairCfg<STAGES>::THREADS, 1)
    fused_up_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmB64,
                         const __grid_constant__ CUtensorMap tmB32,
                         const __grid_constant__ CUtensorMap tmY, const FusedArgs args) {
    using C = PairCfg<STAGES>;
    static_assert(!PLAIN || (!E::kFp8 && !IL), "plain product: BF16 CTA pairs, blocked weights");
    // first packed row of this CTA's half of a unit's weight rows
    auto brow0 = [](const Unit &u, uint32_t h) {
        return IL ? 2 * u.width * u.sub + u.width * static_cast<int>(h)
                  : C::BN * static_cast<int>(h) + u.sub * u.width;
    };
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();      // 0 or 1
    const uint32_t half = rank & 1u;               // 0: leader (Gate rows), 1: Up rows
    constexpr uint32_t leader_rank = 0;
    const bool is_leader = half == 0;
    // schedule worker: one cluster; with a K split, by start order (below)
    int pair = static_cast<int>(blockIdx.x / 2);
    if (args.sched.sk_iters > 0) pair = args.sched.grid - 1 - pair;   // guess, for the prefetch

    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return sbase + C::OFF_BAR + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return sbase + C::OFF_BAR + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * STAGES + 4);
    const uint32_t fix_bar = sbase + C::OFF_BAR + 8u * (2 * STAGES + 5);
    auto rfull_bar = [&](int i) { return sbase + C::OFF_BAR + 8u * (2 * STAGES + 6 + i); };
    auto rempty_bar = [&](int i) {
        return sbase + C::OFF_BAR + 8u * (2 * STAGES + 6 + kTileRing + i);
    };
    volatile int *ring = reinterpret_cast<volatile int *>(smem + C::OFF_RING);
    const bool dyn = args.dyn_tiles != 0;   // the same in every CTA
    // a whole tile of the data-parallel schedule
    auto dp_unit = [&](int t) {
        Unit u;
        u.tile = t;
        u.kb0 = 0;
        u.kb1 = args.sched.k_blocks;
        u.sk = -1;
        u.width = C::BN;
        u.sub = 0;
        return u;
    };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    volatile int *last_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);
    volatile int *worker_slot = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 12);
    // the same flag in the other CTA of the pair
    auto set_abort_both = [&]() {
        *abort_flag = 1;
        st_cluster_u32(mapa_shared(sbase + C::OFF_MISC + 4, rank ^ 1u), 1u);
    };

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);       // one commit from the pair's MMA
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * C::EPI_WARPS);  // epilogue warps of both CTAs
        }
        mbar_init(drain_bar, 1);
        mbar_init(fix_bar, 1);
        for (int i = 0; i < kTileRing; ++i) {
            mbar_init(rfull_bar(i), 1);
            mbar_init(rempty_bar(i), C::RING_READERS);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmY);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const WorkSched &sched = args.sched;
    // The prologue above touched no global memory: the next launch may start
    // now, and this one waits here for the previous launch's results. While
    // it waits (the previous launch's last tiles), the producer asks L2 for
    // this CTA's first pipeline stages: a prefetch reads device memory into
    // L2 only, and L2 is where every SM's writes land, so data the previous
    // launch writes afterwards is still what the loads below see. With
    // late_trigger the next launch may start only after the wait below.
    if (!args.late_trigger) griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        UnitIter it;
        it.init(sched, pair);
        Unit u;
        if (it.next(u)) {
            int tm, nb;
            sched.order.coords(u.tile, tm, nb);
            const CUtensorMap *tmBu = (u.width == C::BN) ? &tmB : (u.width == 64 ? &tmB64 : &tmB32);
            const int kend = (u.kb1 - u.kb0 < kPrefetchStages) ? u.kb1 : u.kb0 + kPrefetchStages;
            for (int kb = u.kb0; kb < kend; ++kb) {
                tma_prefetch_2d(&tmA, kb * E::kBK, tm * C::UMMA_M + C::BM * static_cast<int>(half));
                tma_prefetch_3d(tmBu, 0, brow0(u, half), nb * sched.k_blocks + kb);
            }
        }
    }
    griddep_wait();
    if (args.late_trigger) griddep_launch_dependents();
    if (sched.sk_iters > 0) {
        // worker number by start order (see the header comment); the peer
        // CTA gets it through distributed shared memory
        if (is_leader && warp == 0 && lane == 0) {
            const unsigned int t =
                atomicInc(args.counters + args.ticket_index, static_cast<unsigned int>(sched.grid - 1));
            const int wid = sched.grid - 1 - static_cast<int>(t % static_cast<unsigned int>(sched.grid));
            *worker_slot = wid;
            st_cluster_u32(mapa_shared(sbase + C::OFF_MISC + 12, 1u), static_cast<uint32_t>(wid));
        }
        cluster_sync();
        pair = *worker_slot;
    }

    uint32_t issued_mask = 0, last_parity = 0;  // leader's drain bookkeeping

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // issue the loads of every k-block of one unit; false if a wait
            // for a free stage ran out or the launch is aborting
            auto load_unit = [&](const Unit &u) -> bool {
                int tm, nb;
                sched.order.coords(u.tile, tm, nb);
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) return false;
#ifdef SWIGLU_TEST_FAULT_INJECTION
                    // test build: the leader never arms or fills the first
                    // stage, so the MMA wait for it runs out
                    if (args.skip_first_fill && is_leader && kb == u.kb0 && stage == 0 &&
                        phase == 0) {
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
#endif
                    // every load of the pair completes on the LEADER's full barrier;
                    // a column sub-tile loads only its Gate (leader) or Up (peer) rows
                    const int brows = u.width;
                    if (is_leader)
                        mbar_arrive_expect_tx(full_bar(stage), 2 * (C::A_BYTES + brows * kRowBytes));
                    const uint32_t bar = mapa_shared(full_bar(stage), leader_rank);
                    tma_load_2d_pair(sbase + C::OFF_A + stage * C::A_BYTES, &tmA, bar, kb * E::kBK,
                                     tm * C::UMMA_M + C::BM * static_cast<int>(half));
                    const CUtensorMap *tmBu =
                        (brows == C::BN) ? &tmB : (brows == 64 ? &tmB64 : &tmB32);
                    tma_load_3d_pair(sbase + C::OFF_B + stage * C::B_BYTES, tmBu, bar, 0,
                                     brow0(u, half), nb * sched.k_blocks + kb);
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                return true;
            };
            if (!dyn) {
                UnitIter it;
                it.init(sched, pair);
                Unit u;
                while (ok && it.next(u)) ok = load_unit(u);
            } else if (is_leader) {
                // the pair's tile sequence: its first-wave tile, then whatever
                // the counter hands out, published in the ring (-1 ends it)
                unsigned int *next_tile = args.counters + args.tile_counter_index;
                int t = pair, slot = 0;
                uint32_t rph = 0;
                while (ok) {
                    const int pub = t < sched.num_tiles ? t : -1;
                    if (!mbar_wait_cluster(rempty_bar(slot), rph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    ring[slot] = pub;
                    st_cluster_u32(mapa_shared(sbase + C::OFF_RING + 4u * slot, 1u),
                                   static_cast<uint32_t>(pub));
                    mbar_arrive(rfull_bar(slot));
                    mbar_arrive_cluster(mapa_shared(rfull_bar(slot), 1u));
                    if (++slot == kTileRing) {
                        slot = 0;
                        rph ^= 1u;
                    }
                    if (pub < 0) break;
                    // the next tile's ticket is in flight while this tile's
                    // loads go out
                    const unsigned int ticket = atomicAdd(next_tile, 1u);
                    ok = load_unit(dp_unit(t));
                    t = sched.grid + static_cast<int>(ticket);
                }
            } else {
                // the peer loads its half of the tiles its leader publishes
                int slot = 0;
                uint32_t rph = 0;
                while (ok) {
                    if (!mbar_wait_cluster(rfull_bar(slot), rph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    const int t = ring[slot];
                    mbar_arrive_cluster(mapa_shared(rempty_bar(slot), leader_rank));
                    if (++slot == kTileRing) {
                        slot = 0;
                        rph ^= 1u;
                    }
                    if (t < 0) break;
                    ok = load_unit(dp_unit(t));
                }
            }
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusProducerTimeout);
                set_abort_both();
            }
            if (dyn && is_leader) {
                // this pair takes no more tiles; the last pair to get here
                // resets the counter pair for the next launch
                __threadfence();
                unsigned int *ctr = args.counters + args.tile_counter_index;
                if (atomicAdd(ctr + 1, 1u) == static_cast<unsigned int>(sched.grid - 1)) {
                    __threadfence();
                    ctr[0] = 0u;
                    ctr[1] = 0u;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && is_leader) {
            constexpr uint32_t idesc = E::idesc(C::UMMA_M, C::UMMA_N);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            UnitIter it;
            it.init(sched, pair);
            Unit u;
            int rslot = 0;
            uint32_t rph = 0;
            // the next unit: static schedule, or the leader's tile ring
            auto next_unit = [&](Unit &nu) -> int {
                if (!dyn) return it.next(nu) ? 1 : 0;
                if (!mbar_wait(rfull_bar(rslot), rph, abort_flag)) return -1;
                const int t = ring[rslot];
                mbar_arrive(rempty_bar(rslot));
                if (++rslot == kTileRing) {
                    rslot = 0;
                    rph ^= 1u;
                }
                if (t < 0) return 0;
                nu = dp_unit(t);
                return 1;
            };
            while (ok) {
                const int got = next_unit(u);
                if (got <= 0) {
                    ok = got == 0;
                    break;
                }
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::UMMA_N);
                const uint32_t idesc_u =
                    (u.width == C::BN) ? idesc : E::idesc(C::UMMA_M, 2 * u.width);
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = smem_desc_k128(sbase + C::OFF_A + stage * C::A_BYTES);
                    const uint64_t b_desc = smem_desc_k128(sbase + C::OFF_B + stage * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < kKSteps; ++k)
                        E::mma_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc_u,
                                    (kb != u.kb0 || k != 0) ? 1u : 0u);
                    // frees the stage in both CTAs of the pair
                    umma_commit_pair_mc(empty_bar(stage), 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(tfull_bar(acc), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusMmaTimeout);
                set_abort_both();
            }
        }
    } else {
        const int quad = warp & 3;
        const int row_in_tile = 32 * quad + lane;  // row within this CTA's 128 rows
        const uint32_t ybuf = sbase + C::OFF_Y + (warp - 2) * C::Y_WARP_BYTES;
        const bool lead_thread = (warp == 2 && lane == 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        UnitIter it;
        it.init(sched, pair);
        Unit u;
        int rslot = 0;
        uint32_t rph = 0;
        // the next unit: static schedule, or the leader's tile ring (every
        // epilogue warp reads the slot; each warp counts once as a reader)
        auto next_unit = [&](Unit &nu) -> int {
            if (!dyn) return it.next(nu) ? 1 : 0;
            if (!epilogue_all(mbar_wait_cluster(rfull_bar(rslot), rph, abort_flag))) return -1;
            const int t = ring[rslot];
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(rempty_bar(rslot), leader_rank));
            if (++rslot == kTileRing) {
                rslot = 0;
                rph ^= 1u;
            }
            if (t < 0) return 0;
            nu = dp_unit(t);
            return 1;
        };
        while (true) {
            const int got = next_unit(u);
            if (got <= 0) {
                ok = got == 0;
                break;
            }
            int tm, nb;
            sched.order.coords(u.tile, tm, nb);
            ok = epilogue_all(mbar_wait(tfull_bar(acc), acc_phase, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int row0 = tm * C::UMMA_M + C::BM * static_cast<int>(half) + 32 * quad;
            const bool rows_live = row0 < args.M;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) +
                                   static_cast<uint32_t>(acc * C::UMMA_N);
            const uint32_t tempty_leader = mapa_shared(tempty_bar(acc), leader_rank);

            int c_lo = pair, c_hi = pair;
            if (u.sk >= 0) {
                const long long first = static_cast<long long>(u.sk) * sched.k_blocks;
                c_lo = sched.sk_owner(first);
                c_hi = sched.sk_owner(first + sched.k_blocks - 1);
            }
            const bool split = c_hi > c_lo;
            bool store_y = !PLAIN;   // a staged Y tile waits for its TMA store
            // 32 summed columns of each accumulator half, at column c of the
            // half (plain product: straight to global memory)
            auto emit32 = [&](int c, const float (&g)[32], const float (&v)[32]) {
                if constexpr (PLAIN) {
                    store_plain32(row0 + lane, nb * C::UMMA_N + c, g, args);
                    store_plain32(row0 + lane, nb * C::UMMA_N + C::BN + c, v, args);
                } else {
                    stage_y32(ybuf, lane, c, g, v, args.gate_scale, args.up_scale);
                }
            };

            if (!PLAIN && u.width != C::BN) {
                // a 64-column sub-tile is one staged TMA box; a 32-column one
                // (half a box) is stored from registers
                if (rows_live) {
                    if (u.width == 64) {
                        if (lane == 0) bulk_wait_group_read0();
                        __syncwarp();
#pragma unroll 1
                        for (int c = 0; c < 64; c += 32) {
                            float g[32], v[32];
                            tmem_ld_gu<IL>(tbase, c, g, v, 64);
                            stage_y32(ybuf, lane, c, g, v, args.gate_scale, args.up_scale);
                        }
                    } else {
                        epilogue_subtile_store<IL>(tbase, u.width, row0 + lane,
                                               nb * C::BN + u.sub * u.width, args);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader);
                store_y = u.width == 64;
            } else if (!split) {
                if (rows_live) {
                    static_assert(C::BN == 128, "four 32-column chunks");
                    if constexpr (PLAIN) {
                        // two passes of 128 output columns through the staging buffer
                        for (int p = 0; p < 2; ++p) {
                            if (lane == 0) bulk_wait_group_read0();
                            __syncwarp();
                            stage_plain_128(tbase + 128 * p, ybuf, lane);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                store_staged_boxes(&tmY, ybuf, nb * C::UMMA_N + 128 * p, row0, 2,
                                                   args.N);
                                bulk_commit_group();
                            }
                        }
                    } else {
                        if (lane == 0) bulk_wait_group_read0();
                        __syncwarp();
                        epilogue_stage_tile<IL>(tbase, ybuf, lane, args.gate_scale, args.up_scale);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(tempty_leader);
            } else {
                const size_t slot_floats = static_cast<size_t>(kSlotCols) * args.slot_rows;
                auto slot_of = [&](int p) {
                    return args.partials +
                           static_cast<size_t>((2 * p + sched.sk_slot(p, u.sk)) * 2 + half) *
                               slot_floats;
                };
                unsigned int *counter = args.counters + 2 * u.sk + half;
                const int others = c_hi - c_lo;
                // column group width G (Gate and Up columns) whose partials of
                // every other contributor fit in the operand ring at once
                const uint32_t col_bytes = static_cast<uint32_t>(args.slot_rows) * 4u;
                // (plain product: the ring's last 64 KB stage the owner's output)
                constexpr uint32_t kPlainStage = PLAIN ? C::EPI_WARPS * 4u * 32u * 64u * 2u : 0u;
                const uint32_t ring_bytes = STAGES * (C::A_BYTES + C::B_BYTES) - kPlainStage;
                int G = 128;
                while (G > 32 && static_cast<uint32_t>(others) * 2u * G * col_bytes > ring_bytes)
                    G >>= 1;
                const bool staged = static_cast<uint32_t>(others) * 2u * G * col_bytes <= ring_bytes;
                const uint32_t pstg = sbase + ring_bytes + (warp - 2) * (4u * 32u * 64u * 2u);
                if (pair != c_lo || !staged) {
                    // a contributor (or an owner with too many partners to
                    // stage): this CTA's FP32 partial -> its workspace slot
                    float *slot = slot_of(pair);
                    if (rows_live) {
#pragma unroll 1
                        for (int c = 0; c < C::BN; c += 32) {
                            float g[32], v[32];
                            tmem_ld_gu<IL>(tbase, c, g, v);
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                __stcg(slot + static_cast<size_t>(c + i) * args.slot_rows +
                                           row_in_tile,
                                       g[i]);
                                __stcg(slot + static_cast<size_t>(C::BN + c + i) * args.slot_rows +
                                           row_in_tile,
                                       v[i]);
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_leader);
                    __threadfence();
                    epilogue_bar();
                    if (lead_thread) {
                        const unsigned int prev = atomicAdd(counter, 1u);
                        *last_flag = (prev == static_cast<unsigned int>(others)) ? 1 : 0;
                    }
                    epilogue_bar();
                    const bool last = *last_flag != 0;
                    store_y = store_y && last;
                    if (last) {
                        // the last to count itself in (only when the owner
                        // could not stage): sum every slot in k order
                        __threadfence();
                        if (rows_live) {
                            if (lane == 0) bulk_wait_group_read0();
                            __syncwarp();
#pragma unroll 1
                            for (int c = 0; c < C::BN; c += 32) {
                                float g[32], v[32];
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    g[i] = 0.0f;
                                    v[i] = 0.0f;
                                }
                                for (int p = c_lo; p <= c_hi; ++p) {
                                    const float *src = slot_of(p);
#pragma unroll
                                    for (int i = 0; i < 32; ++i) {
                                        const float pg = __ldcg(src + static_cast<size_t>(c + i) *
                                                                          args.slot_rows +
                                                                row_in_tile);
                                        const float pu = __ldcg(
                                            src + static_cast<size_t>(C::BN + c + i) * args.slot_rows +
                                            row_in_tile);
                                        g[i] = (p == c_lo) ? pg : g[i] + pg;
                                        v[i] = (p == c_lo) ? pu : v[i] + pu;
                                    }
                                }
                                emit32(c, g, v);
                            }
                        }
                        if (lead_thread) *counter = 0u;
                    }
                } else {
                    // the owner: wait until the `others` contributors have
                    // written their partials, then add them to its own
                    // accumulators, column group by column group, through
                    // the idle operand ring
                    bool got = true;
                    if (lead_thread) {
                        got = wait_counter_geq(counter, static_cast<unsigned int>(others));
                        fence_proxy_async_global();
                    }
                    ok = epilogue_all(got);
                    if (!ok) {
                        if (lead_thread && !*abort_flag) {
                            atomicOr(&g_status_word, kStatusEpilogueTimeout);
                            set_abort_both();
                        }
                        break;
                    }
                    if (rows_live) {
                        if (lane == 0) bulk_wait_group_read0();
                        __syncwarp();
                    }
                    const uint32_t part_bytes = static_cast<uint32_t>(G) * col_bytes;
                    uint32_t fix_phase = 0;
#pragma unroll 1
                    for (int g0 = 0; g0 < C::BN; g0 += G) {
                        epilogue_bar();  // everyone is done reading the ring
                        if (lead_thread) {
                            mbar_arrive_expect_tx(fix_bar, static_cast<uint32_t>(others) * 2u *
                                                               part_bytes);
                            for (int q = 0; q < others; ++q) {
                                const float *src = slot_of(c_lo + 1 + q);
                                const uint32_t dst = sbase + static_cast<uint32_t>(q) * 2u * part_bytes;
                                bulk_copy_g2s(dst, src + static_cast<size_t>(g0) * args.slot_rows,
                                              part_bytes, fix_bar);
                                bulk_copy_g2s(dst + part_bytes,
                                              src + static_cast<size_t>(C::BN + g0) * args.slot_rows,
                                              part_bytes, fix_bar);
                            }
                        }
                        ok = epilogue_all(mbar_wait(fix_bar, fix_phase, abort_flag));
                        fix_phase ^= 1u;
                        if (!ok) break;
                        if (rows_live) {
                            const float *ring = reinterpret_cast<const float *>(smem);
#pragma unroll 1
                            for (int c = g0; c < g0 + G; c += 32) {
                                float g[32], v[32];
                                tmem_ld_gu<IL>(tbase, c, g, v);  // own part: first in k order
                                for (int q = 0; q < others; ++q) {
                                    const float *pg = ring + static_cast<size_t>(q) * 2u * G *
                                                                 args.slot_rows;
                                    const float *pu = pg + static_cast<size_t>(G) * args.slot_rows;
#pragma unroll
                                    for (int i = 0; i < 32; ++i) {
                                        const size_t off = static_cast<size_t>(c - g0 + i) *
                                                               args.slot_rows + row_in_tile;
                                        g[i] += pg[off];
                                        v[i] += pu[off];
                                    }
                                }
                                if constexpr (PLAIN) {
                                    stage_bf16x32(pstg, lane, c, g);
                                    stage_bf16x32(pstg, lane, C::BN + c, v);
                                } else {
                                    emit32(c, g, v);
                                }
                            }
                        }
                    }
                    if (!ok) {
                        if (lead_thread && !*abort_flag) {
                            atomicOr(&g_status_word, kStatusEpilogueTimeout);
                            set_abort_both();
                        }
                        break;
                    }
                    if constexpr (PLAIN) {
                        if (rows_live) {
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                store_staged_boxes(&tmY, pstg, nb * C::UMMA_N, row0, 4, args.N);
                                bulk_commit_group();
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_leader);
                    if (lead_thread) *counter = 0u;
                }
            }
            if (store_y && rows_live) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int x0 = nb * C::BN + u.sub * u.width;   // whole tiles: sub = 0
                    if (x0 < args.N) tma_store_2d(&tmY, ybuf, x0, row0);
                    if (u.width == C::BN && x0 + 64 < args.N)
                        tma_store_2d(&tmY, ybuf + C::Y_HALF_BYTES, x0 + 64, row0);
                    bulk_commit_group();
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) {
            // the last store has read its staging buffer; its writes to
            // global memory complete with the grid (what the next launch's
            // griddepcontrol.wait and stream order wait for)
            bulk_wait_group_read0();
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusEpilogueTimeout);
                set_abort_both();
            }
        }
    }

    // ---- teardown
    __syncthreads();
    cluster_sync();  // every CTA out of its loops; abort flags final
    // An abort sets the flag in every CTA of the cluster before this barrier,
    // so all CTAs take the same branch. Without one, every issued load was
    // consumed and every MMA completed before its accumulator was read.
    if (*abort_flag) {
        if (is_leader) {
            if (warp == 0 && lane == 0) {
                // every load into the pair completes on the leader's full barriers
                for (int s = 0; s < STAGES; ++s)
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
        cluster_sync();  // the other CTAs stay until each leader has drained
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace swiglu
