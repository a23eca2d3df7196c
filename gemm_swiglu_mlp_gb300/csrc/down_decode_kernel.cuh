// Plain product out = Y x W3 for few token rows: the down-projection of the
// gated MLP at decode sizes ("Tile-Level Activation Overlap for Efficient LLM
// Inference", Section 1 Introduction and Figure 1: the MLP whose time the
// fused activation shortens; its decode shapes are the M = 1..128 columns of
// the pages' Qwen-2.5 size table).
//
// With M <= 128 token rows the product streams W3 from HBM and the tensor
// cores idle; what counts is how many weight bytes every SM keeps in flight.
// The operands' roles are swapped against the other down-projection kernels:
// the UMMA's 128-row side (A) is 128 OUTPUT COLUMNS of W3 (one half of a
// packed 256-column weight tile: 16 KB per k-block), and its N side is the
// token rows, rounded up to mt = 16..128 (B: mt x 64 values of Y per k-block,
// rows past M filled with zeros by TMA). The accumulator D [128 output
// columns x mt tokens] takes mt TMEM columns, and a stage is 16 KB of
// weights plus mt x 128 bytes of Y: 11 stages (176 KB of weights in flight)
// at mt <= 32, 9 at mt <= 64, 7 at mt <= 128. A tile-per-token-block kernel
// would instead load a whole 128-row A tile per k-block for mt useful rows.
//
// Work split: the T = ceil(N / 128) tiles of a decode shape are far fewer
// than the SMs (7B: 28, 72B: 64), so each tile is cut into j equal K ranges
// and its j CTAs form one thread-block cluster (j = 1..16, chosen on the host
// so that the T clusters fit the GPU in one wave: plan_decode_splits in
// schedule.cuh). Each CTA accumulates its K range in TMEM, then writes the
// FP32 partial [mt tokens x 128 columns] into its own shared memory (the
// operand ring, idle by then); after a cluster barrier, CTA r sums the r-th
// slice of the tile from all j partials through distributed shared memory,
// in rank order (= K order, so results are bit-reproducible), loading every
// rank's values of up to 16 / j chunks before adding any (decode_finish),
// and stores it as BF16; a second cluster barrier keeps every partial alive
// until it has been read. The reduction needs no global workspace, no atomics and no L2
// round trip, and no CTA waits for one outside its cluster, whose CTAs the
// hardware schedules together.
//
// Every mbarrier wait is bounded (sm103_ptx.cuh); a CTA that gives up still
// reaches both cluster barriers, after draining its loads and MMAs in
// flight.
#pragma once

#include "epilogue.cuh"

namespace swiglu {

constexpr int kDecodeSmemLimit = 232448;   // dynamic shared memory per CTA (227 KB)
constexpr int kDecodeMaxSplits = 16;       // K ranges per tile: the largest cluster

template <int MTB>
struct DecodeCfg {
    static_assert(MTB == 32 || MTB == 64 || MTB == 128, "token rows a stage holds");
    static constexpr int COLS = 128;                    // output columns per tile (UMMA M)
    static constexpr int W_BYTES = COLS * kRowBytes;    // 16 KB of weights per k-block
    static constexpr int Y_BYTES = MTB * kRowBytes;     // token rows per k-block
    static constexpr int STAGE_BYTES = W_BYTES + Y_BYTES;
    static constexpr int STAGES = (kDecodeSmemLimit - 2048) / STAGE_BYTES;
    static constexpr int OFF_W = 0;
    static constexpr int OFF_Y = STAGES * W_BYTES;
    static constexpr int OFF_BAR = OFF_Y + STAGES * Y_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 2;     // full, empty, tfull, drain
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;   // tmem base, abort flag
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;   // + 1 KB alignment slack
    static constexpr int EPI_WARPS = 4;
    static constexpr int EPI_THREADS = 32 * EPI_WARPS;
    static constexpr int THREADS = 64 + EPI_THREADS;    // producer, MMA, four epilogue warps
    static constexpr int TMEM_COLS = MTB;               // one accumulator
    // the FP32 partial [MTB tokens][128 columns] at offset 0, over the ring
    static constexpr int PARTIAL_BYTES = MTB * COLS * 4;
    static_assert(PARTIAL_BYTES <= OFF_BAR, "the partial fits in the operand ring");
    static_assert(SMEM_BYTES <= kDecodeSmemLimit, "shared memory budget");
    static_assert((Y_BYTES % 1024) == 0 && (W_BYTES % 1024) == 0, "128-byte swizzle atoms");
};

// Arguments of one launch: out [M, N] = Y [M, K] x W3 [K, N], W3 packed as
// the down-projection weights ([KT][KB][256][64]: KT tiles of 256 output
// columns, KB = k_blocks k-blocks of 64 reduction values). The grid is
// ceil(N / 128) * splits CTAs in clusters of `splits`: cluster t computes
// output columns 128t.., its CTA r the k-blocks [KB*r/splits, KB*(r+1)/splits).
struct DecodeArgs {
    int M;                     // token rows
    int N;                     // output columns
    int mt;                    // M rounded up to 16: UMMA N and the Y box's rows
    int k_blocks;
    int splits;                // K ranges per tile = cluster size, 1..16, <= k_blocks
    int weights_early;         // 1: no launch still in flight writes W3 (see the prologue)
    uint16_t *out;             // [M, N] row-major BF16
#ifdef SWIGLU_TEST_FAULT_INJECTION
    int skip_first_fill;       // test build only: never fill the first pipeline stage
#endif
};

// The cluster's sum of one tile slice: this thread's chunks first, first +
// STRIDE, .. (< c_hi), U of them per step. Chunk c is the float4 at byte 16c
// of every CTA's partial ([token][128 columns] FP32 at shared offset 0): all
// `splits` (<= 16 / U) CTAs' values of the step's chunks are loaded before
// any is added, then each chunk is summed in rank order and stored as BF16.
template <int U, int STRIDE>
__device__ __forceinline__ void decode_finish(const DecodeArgs &args, uint32_t sbase, int tile,
                                              int splits, int first, int c_hi) {
    constexpr int QMAX = kDecodeMaxSplits / U;
    for (int c0 = first; c0 < c_hi; c0 += STRIDE * U) {
        float4 v[U][QMAX];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + STRIDE * u;
            if (c < c_hi) {
                const uint32_t local = sbase + 16u * static_cast<uint32_t>(c);
#pragma unroll
                for (int q = 0; q < QMAX; ++q)
                    if (q < splits)
                        v[u][q] = ld_cluster_f32x4(mapa_shared(local, static_cast<uint32_t>(q)));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + STRIDE * u;
            const int col = tile * 128 + 4 * (c & 31);
            // N % 8 == 0: a chunk is all in or all out
            if (c >= c_hi || col >= args.N) continue;
            float4 s = v[u][0];
#pragma unroll
            for (int q = 1; q < QMAX; ++q) {
                if (q < splits) {
                    s.x += v[u][q].x;
                    s.y += v[u][q].y;
                    s.z += v[u][q].z;
                    s.w += v[u][q].w;
                }
            }
            uint2 packed;
            packed.x = pack_bf16x2(s.x, s.y);
            packed.y = pack_bf16x2(s.z, s.w);
            *reinterpret_cast<uint2 *>(args.out + static_cast<size_t>(c >> 5) * args.N + col) =
                packed;
        }
    }
}

template <int MTB>
__global__ void __launch_bounds__(DecodeCfg<MTB>::THREADS, 1)
    down_decode_kernel(const __grid_constant__ CUtensorMap tmY, const __grid_constant__ CUtensorMap tmW,
                       const DecodeArgs args) {
    using C = DecodeCfg<MTB>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int splits = args.splits;
    const int rank = splits > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int tile = static_cast<int>(blockIdx.x) / splits;
    const int kb0 = static_cast<int>(static_cast<long long>(args.k_blocks) * rank / splits);
    const int kb1 = static_cast<int>(static_cast<long long>(args.k_blocks) * (rank + 1) / splits);
    const int mt = args.mt;

    auto full_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::OFF_BAR + 8u * (C::STAGES + s); };
    const uint32_t tfull_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES);
    const uint32_t drain_bar = sbase + C::OFF_BAR + 8u * (2 * C::STAGES + 1);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
        prefetch_tmap(&tmY);
        prefetch_tmap(&tmW);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // The prologue touched no global memory: let the next launch begin, then
    // wait for the previous launch's results (Y). Meanwhile the producer asks
    // L2 for the first weight stages, or, when the caller guarantees that no
    // launch still in flight writes W3 (weights_early), already loads the
    // weights of the first ring pass into shared memory.
    const int wrow = 128 * (tile & 1);
    const int wtile0 = (tile >> 1) * args.k_blocks;
    const uint32_t tx = static_cast<uint32_t>(C::W_BYTES + mt * kRowBytes);
    // producer bookkeeping for the drain after an abort
    uint32_t issued_mask = 0, last_parity = 0;
    int pre = 0;   // stages whose weights were loaded before the wait
    griddep_launch_dependents();
    if (warp == 0 && lane == 0) {
        bool early = args.weights_early != 0;
#ifdef SWIGLU_TEST_FAULT_INJECTION
        early = early && !args.skip_first_fill;
#endif
        if (early) {
            // the ring's first pass: every stage is free (phase 0)
            pre = (kb1 - kb0 < C::STAGES) ? kb1 - kb0 : C::STAGES;
            for (int st = 0; st < pre; ++st) {
                mbar_arrive_expect_tx(full_bar(st), tx);
                tma_load_3d(sbase + C::OFF_W + st * C::W_BYTES, &tmW, full_bar(st), 0, wrow,
                            wtile0 + kb0 + st);
                issued_mask |= 1u << st;
            }
        } else {
            const int kend = (kb1 - kb0 < kPrefetchStages) ? kb1 : kb0 + kPrefetchStages;
            for (int kb = kb0; kb < kend; ++kb) tma_prefetch_3d(&tmW, 0, wrow, wtile0 + kb);
        }
    }
    griddep_wait();

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (kb - kb0 < pre) {
                    // this stage's weights are in flight already: its Y block
                    tma_load_2d(sbase + C::OFF_Y + stage * C::Y_BYTES, &tmY, full_bar(stage),
                                kb * ElemBF16::kBK, 0);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
#ifdef SWIGLU_TEST_FAULT_INJECTION
                if (args.skip_first_fill && kb == kb0) {
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
#endif
                mbar_arrive_expect_tx(full_bar(stage), tx);
                tma_load_3d(sbase + C::OFF_W + stage * C::W_BYTES, &tmW, full_bar(stage), 0, wrow,
                            wtile0 + kb);
                tma_load_2d(sbase + C::OFF_Y + stage * C::Y_BYTES, &tmY, full_bar(stage),
                            kb * ElemBF16::kBK, 0);
                issued_mask |= 1u << stage;
                last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusProducerTimeout);
                *abort_flag = 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(C::COLS, mt);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(full_bar(stage), phase, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t a_desc = smem_desc_k128(sbase + C::OFF_W + stage * C::W_BYTES);
                const uint64_t b_desc = smem_desc_k128(sbase + C::OFF_Y + stage * C::Y_BYTES);
#pragma unroll
                for (int k = 0; k < kKSteps; ++k)
                    umma_bf16(tmem_base, a_desc + 2u * k, b_desc + 2u * k, idesc,
                              (kb != kb0 || k != 0) ? 1u : 0u);
                umma_commit(empty_bar(stage));
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) umma_commit(tfull_bar);
            if (!ok && !*abort_flag) {
                atomicOr(&g_status_word, kStatusMmaTimeout);
                *abort_flag = 1;
            }
        }
    } else {
        // ---- epilogue: one thread per output column of the tile (TMEM lane),
        // 16 tokens (TMEM columns) per load
        const int quad = warp & 3;
        const int col_in_tile = 32 * quad + lane;
        const bool ok =
            epilogue_all(mbar_wait(tfull_bar, 0, abort_flag, 2 * kWaitLimitCycles));
        if (ok) {
            tc_fence_after();
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(32 * quad) << 16);
            const int col = tile * C::COLS + col_in_tile;
            float *partial = reinterpret_cast<float *>(smem);
#pragma unroll 1
            for (int p = 0; p < (mt >> 4); ++p) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(tbase + 16 * p, r);
                tmem_ld_wait();
                reg_fence16(r);
                if (splits == 1) {
                    // the whole K range: BF16 rows 16p .. 16p+15 of this column
                    if (col < args.N) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int t = 16 * p + i;
                            if (t < args.M) {
                                const __nv_bfloat16 h = __float2bfloat16_rn(__uint_as_float(r[i]));
                                args.out[static_cast<size_t>(t) * args.N + col] =
                                    *reinterpret_cast<const uint16_t *>(&h);
                            }
                        }
                    }
                } else {
                    // this K range's partial, [token][column] in shared memory
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        partial[(16 * p + i) * C::COLS + col_in_tile] = __uint_as_float(r[i]);
                }
            }
            tc_fence_before();
        } else if (lane == 0 && !*abort_flag) {
            atomicOr(&g_status_word, kStatusEpilogueTimeout);
            *abort_flag = 1;
        }
    }

    // ---- teardown: every role has left its loop
    __syncthreads();
    if (*abort_flag) {
        if (warp == 0 && lane == 0) {
            // every TMA load already issued lands before shared memory is reused
            for (int s = 0; s < C::STAGES; ++s)
                if ((issued_mask >> s) & 1u)
                    if (!mbar_wait_drain(full_bar(s), (last_parity >> s) & 1u))
                        atomicOr(&g_status_word, kStatusDrainTimeout);
        }
        if (warp == 1 && lane == 0) {
            // all MMAs issued by this thread complete before TMEM is freed
            umma_commit(drain_bar);
            if (!mbar_wait_drain(drain_bar, 0)) atomicOr(&g_status_word, kStatusDrainTimeout);
        }
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
    if (splits > 1) {
        // every CTA of the cluster has its partial in shared memory
        cluster_sync();
        if (warp >= 2 && !*abort_flag) {
            // slice `rank` of the tile's M x 128 outputs, in 4-column chunks
            // (chunk c: token c / 32, columns 4 * (c % 32) ..), summed over
            // the cluster's partials in rank order; U chunks per step, so
            // that U * splits (<= 16) loads from the cluster's shared
            // memories are in flight at once
            const int chunks = args.M * (C::COLS / 4);
            const int c_lo = static_cast<int>(static_cast<long long>(chunks) * rank / splits);
            const int c_hi = static_cast<int>(static_cast<long long>(chunks) * (rank + 1) / splits);
            const int first = c_lo + static_cast<int>(threadIdx.x) - 64;
            if (splits <= 2)
                decode_finish<8, C::EPI_THREADS>(args, sbase, tile, splits, first, c_hi);
            else if (splits <= 4)
                decode_finish<4, C::EPI_THREADS>(args, sbase, tile, splits, first, c_hi);
            else if (splits <= 8)
                decode_finish<2, C::EPI_THREADS>(args, sbase, tile, splits, first, c_hi);
            else
                decode_finish<1, C::EPI_THREADS>(args, sbase, tile, splits, first, c_hi);
        }
        // every partial has been read before any CTA of the cluster exits
        cluster_sync();
    }
}

}  // namespace swiglu
