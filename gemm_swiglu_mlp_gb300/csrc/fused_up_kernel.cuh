// Fused SwiGLU up-projection kernel for sm_103a (tcgen05 / TMEM / TMA).
//
// Computes Y = SiLU(A x W1) (.) (A x W2) ("Tile-Level Activation Overlap for
// Efficient LLM Inference", Section 1 Introduction) without writing Gate or
// Up to global memory (same paper, Abstract). Design, per persistent CTA:
//
//   warp 0        TMA producer: for each k-block loads one A tile [128 x 64]
//                 and one packed weight tile [256 x 64] (128 Gate rows then
//                 128 Up rows of the same output columns, one contiguous
//                 32 KB block of the packed operand) into a STAGES-deep
//                 shared-memory ring. Each A tile feeds both products. When
//                 M < 128 the A box has only ceil(M/8)*8 rows: the rows past
//                 it keep stale shared-memory data, which reaches only
//                 accumulator rows >= M, and those are never stored. A
//                 column sub-tile (64 or 32 output columns) loads its Gate
//                 rows and the matching Up rows in one 4-D box; a launch made
//                 only of sub-tiles uses narrow stages (BROWS weight rows),
//                 so more of them fit.
//   warp 1        MMA issuer: one tcgen05.mma (M=128, N=256, K=16) per K
//                 step puts Gate in TMEM columns [0,128) and Up in [128,256)
//                 of one accumulator stage; two stages (512 columns) let the
//                 next unit's MMAs run while the epilogue drains this one.
//   warps 2..5    epilogue: tcgen05.ld Gate and Up for 32 rows each,
//                 y = SiLU(g) * u in FP32, round to BF16, stage in 128-byte
//                 swizzled shared memory, TMA store (clipped at M and N).
//
// Work is split by schedule.cuh: whole tiles, column sub-tiles for the last
// wave, or (for a handful of tiles) an even stream-K split of the k-block
// iterations. A tile cut between CTAs is
// finished without any inter-CTA waiting: every contributor writes its FP32
// Gate/Up partial to a workspace slot and increments the tile's counter; the
// one that brings the counter to the number of contributors sums all
// partials in k order (so the result does not depend on arrival order),
// applies the activation, stores Y and resets the counter to zero. SiLU is
// nonlinear, so partial sums are always combined BEFORE it.
//
// This replaces the pages' two SM90 designs (technical summary, "Kernel-1"
// and "Kernel-2"): the packed operand plays the role of Kernel-2's fused
// weight matrix (one GEMM feeds both accumulators from one A tile), the
// paired accumulators sit in TMEM instead of registers, and the activation
// overlaps the next tile's MMA (Kernel-2's compute/store overlap) rather
// than the Up-tile load (Kernel-1).
//
// Every wait is bounded (sm103_ptx.cuh). A role that gives up sets a bit in
// the device status word and the shared abort flag; the others leave their
// loops, in-flight TMA loads and MMAs are drained with bounded waits, and
// TMEM is released before the CTA exits.
#pragma once

#include "epilogue.cuh"

namespace swiglu {

// BROWS = weight rows a stage holds: 256 (a whole tile's Gate and Up rows),
// or, for launches made only of column sub-tiles of BROWS / 2 columns (the
// narrow configurations), 128 or 64: smaller stages, so more of them fit
// and more loads are in flight per SM. Sub-tiles store Y straight from
// registers, so the narrow configurations have no Y staging buffer.
template <int STAGES, int BROWS = 256>
struct FusedCfg {
    static constexpr int BM = 128;                // token rows per tile = UMMA M
    static constexpr int BN = 128;                // output columns per tile
    static constexpr int BK = 64;                 // BF16 elements per 128-byte row
    static constexpr int UMMA_N = 2 * BN;         // Gate | Up
    static constexpr int UMMA_K = 16;
    static constexpr bool NARROW = BROWS < UMMA_N;
    static constexpr int A_BYTES = BM * BK * 2;   // 16 KB
    static constexpr int B_BYTES = BROWS * BK * 2;  // 32 KB for a whole tile
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_WARPS = 4;
    static constexpr int Y_HALF_BYTES = 32 * 64 * 2;      // 32 rows x 64 cols, 4 KB
    static constexpr int Y_WARP_BYTES = NARROW ? 0 : 2 * Y_HALF_BYTES;  // 32 rows x 128 cols
    static constexpr int TMEM_COLS = 2 * UMMA_N;          // two accumulator stages
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_Y = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_Y + EPI_WARPS * Y_WARP_BYTES;
    // full, empty, tfull x2, tempty x2, drain, fix (bulk copies of split partials)
    static constexpr int NUM_BARS = 2 * STAGES + 6;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;  // tmem base, abort flag, last flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + 1 KB alignment slack
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static_assert(TMEM_COLS == 512, "two 256-column accumulator stages fill TMEM");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(UMMA_N == kSlotCols, "workspace slot shape");
};

// IL: the packed weights are column-interleaved (even rows Gate, odd rows
// Up, the pages' Kernel-2 pairing; pack_weights_il_kernel) instead of
// 128-row blocked. Only the sub-tile weight boxes and the epilogue's TMEM
// column addressing differ.
//
// PLAIN = true: a plain product out = A x W (no activation), the
// down-projection out = Y x W3 of a decode-sized MLP (M <= 128). W is the
// down-projection's packed layout ([KT][KB][256][64]); a tile is 128 rows x
// 64 output columns, the 64 rows 64*(t%4).. of packed tile t/4 (one UMMA
// N=64 per K step), in the narrow 64-row configuration. With so few rows the
// product streams W3 from HBM, and its few output columns leave most SMs idle
// unless K is split: the stream-K partial of a tile is only 64 columns wide,
// so the last contributor's sum reads a few KB per partner. The epilogue
// rounds to BF16 and stores from registers; whole tiles and stream-K only.
template <int STAGES, int BROWS, typename E, bool IL = false, bool PLAIN = false>
__global__ void __launch_bounds__(FusedCfg<STAGES, BROWS>::THREADS, 1)
    fused_up_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmB64,
                    const __grid_constant__ CUtensorMap tmB32,
                    const __grid_constant__ CUtensorMap tmY, const FusedArgs args) {
    using C = FusedCfg<STAGES, BROWS>;
    static_assert(!PLAIN || (!IL && !E::kFp8 && BROWS == 64), "plain product: BF16, 64-row stages");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;

    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return sbase + C::OFF_BAR + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return sbase + C::OFF_BAR + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * STAGES + 4);
    const uint32_t fix_bar = sbase + C::OFF_BAR + 8u * (2 * STAGES + 5);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    volatile int *last_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 8);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), C::EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        mbar_init(fix_bar, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        prefetch_tmap(&tmY);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    const WorkSched &sched = args.sched;
    // The prologue above touched no global memory: the next launch may start
    // now, and this one waits here for the previous launch's results. While
    // it waits, the producer asks L2 for this CTA's first pipeline stages (a
    // prefetch only moves device memory into L2, where every SM's writes
    // land, so what the previous launch writes afterwards is still what the
    // loads below see). With late_trigger the next launch may start only
    // after the wait below.
    if (!args.late_trigger) griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        UnitIter it;
        it.init(sched, cta);
        Unit u;
        if (it.next(u)) {
            int mb, nb;
            sched.order.coords(u.tile, mb, nb);
            const int kend = (u.kb1 - u.kb0 < kPrefetchStages) ? u.kb1 : u.kb0 + kPrefetchStages;
            for (int kb = u.kb0; kb < kend; ++kb) {
                const int wtile = nb * sched.k_blocks + kb;
                tma_prefetch_2d(&tmA, kb * E::kBK, mb * C::BM);
                if constexpr (PLAIN) {
                    tma_prefetch_3d(&tmB, 0, 64 * (nb & 3), (nb >> 2) * sched.k_blocks + kb);
                } else if (u.width == C::BN) {
                    tma_prefetch_3d(&tmB, 0, 0, wtile);
                } else {
                    const CUtensorMap *tmBn = (u.width == 64) ? &tmB64 : &tmB32;
                    if constexpr (IL)
                        tma_prefetch_3d(tmBn, 0, 2 * u.width * u.sub, wtile);
                    else
                        tma_prefetch_4d(tmBn, 0, u.sub * u.width, 0, wtile);
                }
            }
        }
    }
    griddep_wait();
    if (args.late_trigger) griddep_launch_dependents();

    // Producer bookkeeping kept for the drain after an abort: which stages
    // received a load, and the parity of the phase of the last one.
    uint32_t issued_mask = 0, last_parity = 0;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            UnitIter it;
            it.init(sched, cta);
            Unit u;
            while (ok && it.next(u)) {
                int mb, nb;
                sched.order.coords(u.tile, mb, nb);
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
#ifdef SWIGLU_TEST_FAULT_INJECTION
                    // test build: leave the very first stage unfilled, so the
                    // MMA warp's wait for it runs out (failure-detection test)
                    if (args.skip_first_fill && kb == u.kb0 && stage == 0 && phase == 0) {
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
#endif
                    if (!PLAIN && 2 * u.width > BROWS) {  // never planned: a unit wider than a stage
                        ok = false;
                        break;
                    }
                    const uint32_t b_dst = sbase + C::OFF_B + stage * C::B_BYTES;
                    const int wtile = nb * sched.k_blocks + kb;
                    if constexpr (PLAIN) {
                        // 64 output columns: rows 64*(nb%4) of packed tile nb/4
                        mbar_arrive_expect_tx(full_bar(stage), args.a_tx_bytes + 64 * kRowBytes);
                        tma_load_2d(sbase + C::OFF_A + stage * C::A_BYTES, &tmA, full_bar(stage),
                                    kb * E::kBK, mb * C::BM);
                        tma_load_3d(b_dst, &tmB, full_bar(stage), 0, 64 * (nb & 3),
                                    (nb >> 2) * sched.k_blocks + kb);
                    } else if (u.width == C::BN) {
                        mbar_arrive_expect_tx(full_bar(stage), args.stage_tx_bytes);
                        tma_load_2d(sbase + C::OFF_A + stage * C::A_BYTES, &tmA, full_bar(stage),
                                    kb * E::kBK, mb * C::BM);
                        tma_load_3d(b_dst, &tmB, full_bar(stage), 0, 0, wtile);
                    } else {
                        // column sub-tile: its Gate rows, then the matching Up rows,
                        // in one 4-D box (both halves of the packed tile); with
                        // interleaved weights its 2 * width rows are contiguous
                        const CUtensorMap *tmBn = (u.width == 64) ? &tmB64 : &tmB32;
                        mbar_arrive_expect_tx(full_bar(stage),
                                              args.a_tx_bytes + 2 * u.width * kRowBytes);
                        tma_load_2d(sbase + C::OFF_A + stage * C::A_BYTES, &tmA, full_bar(stage),
                                    kb * E::kBK, mb * C::BM);
                        if constexpr (IL)
                            tma_load_3d(b_dst, tmBn, full_bar(stage), 0, 2 * u.width * u.sub, wtile);
                        else
                            tma_load_4d(b_dst, tmBn, full_bar(stage), 0, u.sub * u.width, 0, wtile);
                    }
                    issued_mask |= 1u << stage;
                    last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusProducerTimeout);
                *abort_flag = 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = E::idesc(C::BM, C::UMMA_N);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            UnitIter it;
            it.init(sched, cta);
            Unit u;
            while (ok && it.next(u)) {
                if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::UMMA_N);
                // Gate|Up columns of this unit: 256, or 2 x the sub-tile width
                // (plain product: the tile's 64 output columns)
                const uint32_t idesc_u = PLAIN ? E::idesc(C::BM, 64)
                                         : (u.width == C::BN) ? idesc : E::idesc(C::BM, 2 * u.width);
                for (int kb = u.kb0; kb < u.kb1; ++kb) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_desc = smem_desc_k128(sbase + C::OFF_A + stage * C::A_BYTES);
                    const uint64_t b_desc = smem_desc_k128(sbase + C::OFF_B + stage * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < kKSteps; ++k) {
                        // +32 bytes along K per step inside the 128-byte swizzle row
                        E::mma(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc_u,
                               (kb != u.kb0 || k != 0) ? 1u : 0u);
                    }
                    umma_commit(empty_bar(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(tfull_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusMmaTimeout);
                *abort_flag = 1;
            }
        }
    } else {
        // Epilogue warps 2..5. tcgen05.ld lets warp w touch TMEM lanes
        // [32*(w%4), 32*(w%4)+32): those are the tile rows it owns.
        const int quad = warp & 3;
        const int row_in_tile = 32 * quad + lane;
        const uint32_t ybuf = sbase + C::OFF_Y + (warp - 2) * C::Y_WARP_BYTES;
        const bool leader = (warp == 2 && lane == 0);
        uint32_t fix_phase = 0;   // bulk copies of split partials (plain product)
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        UnitIter it;
        it.init(sched, cta);
        Unit u;
        while (it.next(u)) {
            int mb, nb;
            sched.order.coords(u.tile, mb, nb);
            // Accumulator ready? The answer must be the same in all four warps:
            // one warp could see the barrier complete while another sees the
            // abort flag first.
            ok = epilogue_all(mbar_wait(tfull_bar(acc), acc_phase, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int row0 = mb * C::BM + 32 * quad;
            const bool rows_live = row0 < args.M;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) +
                                   static_cast<uint32_t>(acc * C::UMMA_N);

            // Contributors of a stream-K tile: CTAs c_lo..c_hi, in k order.
            int c_lo = cta, c_hi = cta;
            if (u.sk >= 0) {
                const long long first = static_cast<long long>(u.sk) * sched.k_blocks;
                c_lo = sched.sk_owner(first);
                c_hi = sched.sk_owner(first + sched.k_blocks - 1);
            }
            const bool split = c_hi > c_lo;
            bool store_y = true;

            if constexpr (PLAIN) {
                // 64 output columns from registers; a split tile goes through
                // the workspace (its first 64 slot columns), and the last
                // contributor to count in sums every partial in k order
                store_y = false;
                const int col0 = nb * 64;
                if (!split) {
                    if (rows_live) {
#pragma unroll 1
                        for (int c = 0; c < 64; c += 32) {
                            uint32_t r[32];
                            tmem_ld_32x32b_x32(tbase + c, r);
                            tmem_ld_wait();
                            reg_fence32(r);
                            float x[32];
#pragma unroll
                            for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
                            store_plain32(row0 + lane, col0 + c, x, args);
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(acc));
                } else {
                    const size_t slot_floats = static_cast<size_t>(kSlotCols) * args.slot_rows;
                    float *slot = args.partials +
                                  static_cast<size_t>(2 * cta + sched.sk_slot(cta, u.sk)) * slot_floats;
                    if (rows_live) {
#pragma unroll 1
                        for (int c = 0; c < 64; c += 32) {
                            uint32_t r[32];
                            tmem_ld_32x32b_x32(tbase + c, r);
                            tmem_ld_wait();
                            reg_fence32(r);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                __stcg(slot + static_cast<size_t>(c + i) * args.slot_rows + row_in_tile,
                                       __uint_as_float(r[i]));
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty_bar(acc));
                    __threadfence();
                    epilogue_bar();
                    if (leader) {
                        const unsigned int prev = atomicAdd(args.counters + u.sk, 1u);
                        *last_flag = (prev == static_cast<unsigned int>(c_hi - c_lo)) ? 1 : 0;
                    }
                    epilogue_bar();
                    if (*last_flag != 0) {
                        __threadfence();
                        // The sum of every contributor's partial, in k order.
                        // When this is the CTA's last unit its operand ring
                        // is idle (all its MMAs are complete): the partials'
                        // 64 columns (contiguous at the start of each slot)
                        // come in by bulk copies, as many per round as the
                        // ring holds; otherwise by loads, four contributors'
                        // at a time.
                        UnitIter peek = it;
                        Unit after;
                        const bool last_unit = !peek.next(after);
                        const uint32_t part_bytes = 64u * static_cast<uint32_t>(args.slot_rows) * 4u;
                        constexpr uint32_t kRingBytes = STAGES * (C::A_BYTES + C::B_BYTES);
                        const int per_round = static_cast<int>(kRingBytes / part_bytes);
                        if (last_unit && per_round >= 2) {
                            // the first batch of copies brings the first
                            // per_round partials to slots 0..; each later
                            // batch brings the next ones to slots 1.. and
                            // adds to the running sum in slot 0
                            float *ring = reinterpret_cast<float *>(smem);
                            for (int k0 = c_lo; k0 <= c_hi && ok;) {
                                const int first = k0 == c_lo ? 0 : 1;
                                const int room = per_round - first;
                                const int cnt = (c_hi - k0 + 1 < room) ? c_hi - k0 + 1 : room;
                                if (leader) {
                                    fence_proxy_async_global();
                                    mbar_arrive_expect_tx(fix_bar, static_cast<uint32_t>(cnt) * part_bytes);
                                    for (int q = 0; q < cnt; ++q)
                                        bulk_copy_g2s(sbase + static_cast<uint32_t>(first + q) * part_bytes,
                                                      args.partials +
                                                          static_cast<size_t>(2 * (k0 + q) +
                                                                              sched.sk_slot(k0 + q, u.sk)) *
                                                              slot_floats,
                                                      part_bytes, fix_bar);
                                }
                                ok = epilogue_all(mbar_wait(fix_bar, fix_phase, abort_flag));
                                fix_phase ^= 1u;
                                if (!ok) break;
                                if (rows_live) {
                                    // k order: slot 0 (the partials so far), then the new
                                    // ones; 32 columns at a time, each slot's 32 values
                                    // loaded before they are added (shared-memory latency
                                    // overlapped, not one dependent load per add)
#pragma unroll 1
                                    for (int c = 0; c < 64; c += 32) {
                                        float *cell = ring + static_cast<size_t>(c) * args.slot_rows + row_in_tile;
                                        float x[32];
#pragma unroll
                                        for (int i = 0; i < 32; ++i) x[i] = cell[static_cast<size_t>(i) * args.slot_rows];
#pragma unroll 1
                                        for (int q = 1; q < first + cnt; ++q) {
                                            const float *src = cell + static_cast<size_t>(q) * 64 * args.slot_rows;
                                            float v[32];
#pragma unroll
                                            for (int i = 0; i < 32; ++i) v[i] = src[static_cast<size_t>(i) * args.slot_rows];
#pragma unroll
                                            for (int i = 0; i < 32; ++i) x[i] += v[i];
                                        }
#pragma unroll
                                        for (int i = 0; i < 32; ++i) cell[static_cast<size_t>(i) * args.slot_rows] = x[i];
                                    }
                                }
                                k0 += cnt;
                                epilogue_bar();   // the ring is read before the next round lands
                            }
                            if (ok && rows_live) {
                                const float *sum = reinterpret_cast<const float *>(smem);
#pragma unroll 1
                                for (int c = 0; c < 64; c += 32) {
                                    float x[32];
#pragma unroll
                                    for (int i = 0; i < 32; ++i)
                                        x[i] = sum[static_cast<size_t>(c + i) * args.slot_rows + row_in_tile];
                                    store_plain32(row0 + lane, col0 + c, x, args);
                                }
                            }
                        } else if (rows_live) {
                            // the partials of two contributors are loaded
                            // before either is added (half as many load round
                            // trips as one at a time)
#pragma unroll 1
                            for (int c = 0; c < 64; c += 32) {
                                float x[32];
#pragma unroll 1
                                for (int k0 = c_lo; k0 <= c_hi; k0 += 2) {
                                    float v[2][32];
#pragma unroll
                                    for (int q = 0; q < 2; ++q) {
                                        if (k0 + q > c_hi) break;
                                        const int k = k0 + q;
                                        const float *src = args.partials +
                                            static_cast<size_t>(2 * k + sched.sk_slot(k, u.sk)) *
                                                slot_floats;
#pragma unroll
                                        for (int i = 0; i < 32; ++i)
                                            v[q][i] = __ldcg(src + static_cast<size_t>(c + i) *
                                                                       args.slot_rows + row_in_tile);
                                    }
#pragma unroll
                                    for (int q = 0; q < 2; ++q) {
                                        if (k0 + q > c_hi) break;
#pragma unroll
                                        for (int i = 0; i < 32; ++i)
                                            x[i] = (k0 + q == c_lo) ? v[q][i] : x[i] + v[q][i];
                                    }
                                }
                                store_plain32(row0 + lane, col0 + c, x, args);
                            }
                        }
                        if (leader) args.counters[u.sk] = 0u;  // ready for the next launch
                    }
                }
            } else if (u.width != C::BN) {
                // column sub-tile: straight from TMEM to global memory
                if (rows_live)
                    epilogue_subtile_store<IL>(tbase, u.width, row0 + lane,
                                               nb * C::BN + u.sub * u.width, args);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                store_y = false;
            } else if (C::NARROW) {
                // unreachable: a narrow launch holds only column sub-tiles (the
                // producer refuses anything wider), and it has no Y staging
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                store_y = false;
            } else if (!split) {
                if (rows_live) {
                    if (lane == 0) bulk_wait_group_read0();  // last store has read ybuf
                    __syncwarp();
                    static_assert(C::BN == 128, "four 32-column chunks");
                    epilogue_stage_tile<IL>(tbase, ybuf, lane, args.gate_scale, args.up_scale);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
            } else {
                // 1) this CTA's FP32 partial -> its workspace slot
                const size_t slot_floats = static_cast<size_t>(kSlotCols) * args.slot_rows;
                float *slot = args.partials +
                              static_cast<size_t>(2 * cta + sched.sk_slot(cta, u.sk)) * slot_floats;
                if (rows_live) {
#pragma unroll 1
                    for (int c = 0; c < C::BN; c += 32) {
                        float g[32], v[32];
                        tmem_ld_gu<IL>(tbase, c, g, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            __stcg(slot + static_cast<size_t>(c + i) * args.slot_rows + row_in_tile,
                                   g[i]);
                            __stcg(slot + static_cast<size_t>(C::BN + c + i) * args.slot_rows +
                                       row_in_tile,
                                   v[i]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                // 2) publish, and find out whether this CTA completes the tile
                __threadfence();
                epilogue_bar();
                if (leader) {
                    const unsigned int prev = atomicAdd(args.counters + u.sk, 1u);
                    *last_flag = (prev == static_cast<unsigned int>(c_hi - c_lo)) ? 1 : 0;
                }
                epilogue_bar();
                store_y = *last_flag != 0;
                if (store_y) {
                    __threadfence();
                    // 3) sum every contributor's partial in k order, then activate
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
                            for (int k = c_lo; k <= c_hi; ++k) {
                                const float *src = args.partials +
                                    static_cast<size_t>(2 * k + sched.sk_slot(k, u.sk)) * slot_floats;
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    const float pg = __ldcg(src + static_cast<size_t>(c + i) *
                                                                      args.slot_rows + row_in_tile);
                                    const float pu = __ldcg(src + static_cast<size_t>(C::BN + c + i) *
                                                                      args.slot_rows + row_in_tile);
                                    g[i] = (k == c_lo) ? pg : g[i] + pg;
                                    v[i] = (k == c_lo) ? pu : v[i] + pu;
                                }
                            }
                            stage_y32(ybuf, lane, c, g, v, args.gate_scale, args.up_scale);
                        }
                    }
                    if (leader) args.counters[u.sk] = 0u;  // ready for the next launch
                }
            }
            if (store_y && rows_live) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    const int x0 = nb * C::BN;
                    tma_store_2d(&tmY, ybuf, x0, row0);
                    if (x0 + 64 < args.N) tma_store_2d(&tmY, ybuf + C::Y_HALF_BYTES, x0 + 64, row0);
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
                *abort_flag = 1;
            }
        }
    }

    // ---- teardown: every role has left its loop.
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            // let every TMA load already issued land before shared memory goes
            for (int s = 0; s < STAGES; ++s)
                if ((issued_mask >> s) & 1u)
                    if (!mbar_wait_drain(full_bar(s), (last_parity >> s) & 1u))
                        atomicOr(&g_status_word, kStatusDrainTimeout);
        }
        if (warp == 1 && lane == 0) {
            // all MMAs issued by this thread complete before TMEM is freed
            umma_commit(drain_bar);
            if (!mbar_wait_drain(drain_bar, 0)) atomicOr(&g_status_word, kStatusDrainTimeout);
        }
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace swiglu
