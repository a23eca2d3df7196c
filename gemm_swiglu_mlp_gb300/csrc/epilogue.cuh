// Pieces shared by the 1-SM and 2-SM fused kernels: the device status word,
// the stream-K workspace slot shape, the argument block, and the epilogue
// math (SiLU(g) * u in FP32 -> BF16 into 128-byte-swizzled staging).
#pragma once

#include <cuda_bf16.h>

#include "schedule.cuh"
#include "sm103_ptx.cuh"

namespace swiglu {

// Device status word, read and cleared by swiglu_check_device_status. The
// library is one translation unit (no relocatable device code), so the
// definition lives here.
__device__ unsigned int g_status_word = 0;

enum : unsigned int {
    kStatusProducerTimeout = 1u,
    kStatusMmaTimeout = 2u,
    kStatusEpilogueTimeout = 4u,
    kStatusDrainTimeout = 8u,
};

// Input element types. A shared-memory row is always 128 bytes (one
// 128-byte swizzle row): 64 BF16 or 128 FP8 values per k-block, and one
// UMMA consumes 32 bytes of each row (K = 16 BF16 or 32 FP8), four per
// k-block either way.
struct ElemBF16 {
    static constexpr int kBK = 64;       // elements per k-block
    static constexpr bool kFp8 = false;
    __host__ __device__ static constexpr uint32_t idesc(int M, int N) { return idesc_bf16_f32(M, N); }
    __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        umma_bf16(d, a, b, id, acc);
    }
    __device__ static void mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        umma_bf16_pair(d, a, b, id, acc);
    }
};
struct ElemE4M3 {
    static constexpr int kBK = 128;
    static constexpr bool kFp8 = true;
    __host__ __device__ static constexpr uint32_t idesc(int M, int N) { return idesc_e4m3_f32(M, N); }
    __device__ static void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        umma_f8(d, a, b, id, acc);
    }
    __device__ static void mma_pair(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
        umma_f8_pair(d, a, b, id, acc);
    }
};
constexpr int kRowBytes = 128;   // bytes per shared-memory row of a k-block
constexpr int kKSteps = 4;       // UMMAs per k-block (32 bytes of each row apiece)

// FP32 Gate|Up partial of one tile in the workspace: 256 columns (Gate
// 0..127, Up 128..255) x slot_rows rows, column-major so that the 32 lanes of
// a warp (32 consecutive rows) touch 128 contiguous bytes per column.
// slot_rows = min(128, M rounded up to 32): rows past it are never live.
constexpr int kSlotCols = 256;
// Stages whose loads a CTA asks L2 for while it waits on the previous
// launch. Each TMA instruction takes ~0.1 us to issue, and the wait may
// already be over (a launch that follows an evenly finishing one), so only
// the first two.
constexpr int kPrefetchStages = 2;

__host__ __device__ __forceinline__ int slot_rows_for(long long M) {
    return M >= 128 ? 128 : static_cast<int>((M + 31) / 32 * 32);
}

struct FusedArgs {
    int M, N, K;
    int stage_tx_bytes;       // bytes one stage's TMA loads deliver (A box + weight tile)
    int a_tx_bytes;           // the A box's share of it
    uint16_t *Y;              // Y [M, N] row-major BF16 (direct stores of column sub-tiles)
    float gate_scale;         // Gate = gate_scale * accumulator (FP8: s_a * s_w1; BF16: 1)
    float up_scale;           // Up = up_scale * accumulator (FP8: s_a * s_w2; BF16: 1)
    int slot_rows;            // rows per workspace slot
    WorkSched sched;
    float *partials;          // 2 * grid slots of kSlotCols * slot_rows floats (stream-K only)
    unsigned int *counters;   // one per stream-K tile, zero between launches
    int ticket_index;         // counters[ticket_index]: start-order tickets of a K-split pair launch
    int dyn_tiles;            // 1: tiles past the first wave are handed out at run time (pair kernel)
    int tile_counter_index;   // counters[i]: next dynamic tile; counters[i + 1]: pairs finished
    int late_trigger;         // 1: let the next launch start only after this one's dependency
                              // wait (so that every launch before this one has completed)
#ifdef SWIGLU_TEST_FAULT_INJECTION
    int skip_first_fill;      // test build only: never fill the first pipeline stage
#endif
};

__device__ __forceinline__ float silu_mul(float g, float u) {
    // SiLU(g) = g / (1 + e^-g); for g << 0 the denominator is +inf and the
    // quotient 0, the limit.
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&v);
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity) {
    const int never = 0;
    return mbar_wait(bar, parity, &never);
}

// Named barrier over the four epilogue warps only.
__device__ __forceinline__ void epilogue_bar() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Named barrier over the four epilogue warps that also ANDs a predicate over
// them: every epilogue thread gets the same answer, so all four warps take
// the same branch afterwards (no warp can be left alone at a later barrier).
__device__ __forceinline__ bool epilogue_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v))
        : "memory");
    return r != 0;
}

// y for 32 consecutive columns [c, c+32) of this thread's row, from FP32 Gate
// and Up accumulators (times their scales), written as BF16 into the warp's
// swizzled staging buffer.
__device__ __forceinline__ void stage_y32(uint32_t ybuf, int lane, int c, const float (&g)[32],
                                          const float (&u)[32], float gs, float us) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 8 * j + 2 * e;
            w[e] = pack_bf16x2(silu_mul(g[i] * gs, u[i] * us), silu_mul(g[i + 1] * gs, u[i + 1] * us));
        }
        // 128-byte swizzle: 16-byte chunk index XOR (row % 8)
        const int col = c + 8 * j;
        const int half = col >> 6;
        const int chunk = (col & 63) >> 3;
        const uint32_t addr = ybuf + half * (32 * 64 * 2) + lane * 128 +
                              (static_cast<uint32_t>(chunk ^ (lane & 7)) << 4);
        st_shared_v4(addr, w[0], w[1], w[2], w[3]);
    }
}

// Where a tile's Gate and Up accumulators sit in TMEM, by packed layout:
//   * blocked (IL = false): the packed tile holds 128 Gate rows, then the
//     128 matching Up rows, so Gate of output column c is accumulator column
//     c and its Up is column up_off + c (128 for a whole tile, the sub-tile
//     width for a column sub-tile);
//   * interleaved (IL = true, the pages' Kernel-2 pairing: even packed rows
//     Gate, odd rows Up): Gate of output column c is accumulator column 2c
//     and its Up is 2c + 1, whatever the unit's width.
// Output columns [c, c+32) take two 32-column TMEM loads either way:
// columns c and up_off + c (blocked), or 2c and 2c + 32 (interleaved).
template <bool IL>
__device__ __forceinline__ void tmem_ld_pair_cols(uint32_t tbase, int c, int up_off,
                                                  uint32_t (&ra)[32], uint32_t (&rb)[32]) {
    if constexpr (IL) {
        tmem_ld_32x32b_x32(tbase + 2 * c, ra);
        tmem_ld_32x32b_x32(tbase + 2 * c + 32, rb);
    } else {
        tmem_ld_32x32b_x32(tbase + c, ra);
        tmem_ld_32x32b_x32(tbase + up_off + c, rb);
    }
}

// The 32 Gate and 32 Up values of the two loads above, in output-column
// order.
template <bool IL>
__device__ __forceinline__ void split_gu(const uint32_t (&ra)[32], const uint32_t (&rb)[32],
                                        float (&g)[32], float (&u)[32]) {
    if constexpr (IL) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            g[i] = __uint_as_float(ra[2 * i]);
            u[i] = __uint_as_float(ra[2 * i + 1]);
            g[16 + i] = __uint_as_float(rb[2 * i]);
            u[16 + i] = __uint_as_float(rb[2 * i + 1]);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            g[i] = __uint_as_float(ra[i]);
            u[i] = __uint_as_float(rb[i]);
        }
    }
}

// Gate and Up of output columns [c, c+32) of this thread's row.
template <bool IL = false>
__device__ __forceinline__ void tmem_ld_gu(uint32_t tbase, int c, float (&g)[32], float (&u)[32],
                                           int up_off = 128) {
    uint32_t gr[32], ur[32];
    tmem_ld_pair_cols<IL>(tbase, c, up_off, gr, ur);
    tmem_ld_wait();
    reg_fence32(gr);
    reg_fence32(ur);
    split_gu<IL>(gr, ur, g, u);
}

// Whole-tile epilogue into the warp's staging buffer: the four 32-column
// chunks of Gate|Up are read from TMEM one chunk ahead of the arithmetic, so
// each tcgen05.ld's latency hides behind the previous chunk's activation.
// (tcgen05.wait::ld waits for all of the thread's loads, so the next chunk
// is issued right after the wait that completes the current one.)
template <bool IL = false>
__device__ __forceinline__ void epilogue_stage_tile(uint32_t tbase, uint32_t ybuf, int lane,
                                                    float gs, float us) {
    uint32_t gr[2][32], ur[2][32];
    tmem_ld_pair_cols<IL>(tbase, 0, 128, gr[0], ur[0]);
    tmem_ld_wait();
    reg_fence32(gr[0]);
    reg_fence32(ur[0]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int cur = i & 1;
        if (i + 1 < 4) tmem_ld_pair_cols<IL>(tbase, 32 * (i + 1), 128, gr[cur ^ 1], ur[cur ^ 1]);
        float g[32], u[32];
        split_gu<IL>(gr[cur], ur[cur], g, u);
        stage_y32(ybuf, lane, 32 * i, g, u, gs, us);
        if (i + 1 < 4) {
            tmem_ld_wait();
            reg_fence32(gr[cur ^ 1]);
            reg_fence32(ur[cur ^ 1]);
        }
    }
}

// y for 32 consecutive columns [col, col+32) of one output row, from FP32
// Gate and Up (times their scales), stored straight to global memory in
// 16-byte pieces. Rows >= M and columns >= N are skipped; N is a multiple of
// 8, so a piece is either wholly inside or wholly outside.
__device__ __forceinline__ void store_y32_global(int row, int col, const float (&g)[32],
                                                 const float (&u)[32], const FusedArgs &args) {
    if (row >= args.M) return;
    uint16_t *dst = args.Y + static_cast<size_t>(row) * args.N + col;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (col + 8 * j >= args.N) break;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = 8 * j + 2 * e;
            w[e] = pack_bf16x2(silu_mul(g[i] * args.gate_scale, u[i] * args.up_scale),
                               silu_mul(g[i + 1] * args.gate_scale, u[i + 1] * args.up_scale));
        }
        *reinterpret_cast<uint4 *>(dst + 8 * j) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 32 consecutive output columns [col, col+32) of one row of a plain product
// (no activation): FP32 rounded to BF16 (nearest, ties to even) and stored
// to global memory in 16-byte pieces. Rows >= M and columns >= N are
// skipped; N is a multiple of 8, so a piece is wholly inside or outside.
__device__ __forceinline__ void store_plain32(int row, int col, const float (&x)[32],
                                              const FusedArgs &args) {
    if (row >= args.M) return;
    uint16_t *dst = args.Y + static_cast<size_t>(row) * args.N + col;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (col + 8 * j >= args.N) break;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(x[8 * j + 2 * e], x[8 * j + 2 * e + 1]);
        *reinterpret_cast<uint4 *>(dst + 8 * j) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// 32 values rounded to BF16 into a warp's staging buffer at output column
// `col` (a multiple of 32): boxes of 64 columns x 32 rows (4 KB each, one
// 128-byte row per lane, 16-byte chunks XOR-swizzled by row), the layout a
// 128-byte-swizzled TMA store of 64 x 32 reads.
__device__ __forceinline__ void stage_bf16x32(uint32_t stg, int lane, int col,
                                              const float (&x)[32]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = pack_bf16x2(x[8 * j + 2 * e], x[8 * j + 2 * e + 1]);
        const int cc = col + 8 * j;
        const uint32_t addr = stg + (cc >> 6) * (32 * 64 * 2) + lane * 128 +
                              (static_cast<uint32_t>(((cc & 63) >> 3) ^ (lane & 7)) << 4);
        st_shared_v4(addr, w[0], w[1], w[2], w[3]);
    }
}

// 128 accumulator columns [tcol, tcol+128) of this thread's row, rounded to
// BF16 into the warp's staging buffer (columns 0..127).
__device__ __forceinline__ void stage_plain_128(uint32_t tbase, uint32_t stg, int lane) {
#pragma unroll 1
    for (int c = 0; c < 128; c += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + c, r);
        tmem_ld_wait();
        reg_fence32(r);
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
        stage_bf16x32(stg, lane, c, x);
    }
}

// TMA stores of `boxes` staged 64 x 32 boxes to output columns x0, x0+64,
// ... of rows [row0, row0+32); boxes wholly past column n are skipped (TMA
// clips the rest at the tensor's edges). One thread; the caller commits.
__device__ __forceinline__ void store_staged_boxes(const CUtensorMap *tm, uint32_t stg, int x0,
                                                   int row0, int boxes, int n) {
    for (int q = 0; q < boxes; ++q)
        if (x0 + 64 * q < n) tma_store_2d(tm, stg + q * (32 * 64 * 2), x0 + 64 * q, row0);
}

// Epilogue of a column sub-tile (width 64 or 32), or of a whole tile stored
// without shared-memory staging (width 128): TMEM holds the unit's 2*width
// Gate|Up columns (blocked: Gate in [0, width), Up in [width, 2*width);
// interleaved: in pairs). Each thread owns one output row.
template <bool IL = false>
__device__ __forceinline__ void epilogue_subtile_store(uint32_t tbase, int width, int row,
                                                       int col0, const FusedArgs &args) {
    for (int c = 0; c < width; c += 32) {
        float g[32], v[32];
        tmem_ld_gu<IL>(tbase, c, g, v, width);
        store_y32_global(row, col0 + c, g, v, args);
    }
}

}  // namespace swiglu
