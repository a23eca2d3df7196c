// Host side of the C ABI declared in include/swiglu.h: argument validation,
// per-device setup, TMA tensor-map encoding, schedule choice and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "down_decode_kernel.cuh"
#include "down_wide_kernel.cuh"
#include "fused_up_kernel.cuh"
#include "fused_up_pair_kernel.cuh"
#include "pack_kernel.cuh"
#include "swiglu.h"

namespace swiglu {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kFusedStages = 4;
// narrow 1-SM configurations (launches made only of column sub-tiles):
// weight rows per stage and the stages that fit
constexpr int kNarrow64Stages = 7;   // 64-column sub-tiles: 16 KB A + 16 KB weights
constexpr int kNarrow32Stages = 9;   // 32-column sub-tiles: 16 KB A + 8 KB weights
constexpr int kGroupM = 16;          // row-tiles per L2 group in the tile order
constexpr int kMinStreamKIters = 8;  // k-blocks per CTA share, at least
constexpr int kAssumedMaxSms = 256;  // workspace sizing when no device answers
constexpr int kPairStages = 6;
constexpr int kDownTileCols = 256;   // output columns of a plain-product (down) tile
constexpr int64_t kWideMinM = 256;   // from this many rows on, the wide down-projection kernel
constexpr int64_t kPairMinM = 256;   // from this many tokens on, the 2-SM kernel
constexpr int64_t kDecodeMaxM = 128; // up to this many rows: the decode down-projection kernel
using FusedC = FusedCfg<kFusedStages>;
using Narrow64C = FusedCfg<kNarrow64Stages, 128>;
using Narrow32C = FusedCfg<kNarrow32Stages, 64>;
using PairC = PairCfg<kPairStages>;

#ifdef SWIGLU_TEST_FAULT_INJECTION
int g_test_skip_first_fill = 0;  // set by swiglu_test_set_fault_injection
#endif

// SWIGLU_FUSED_VARIANT=1sm|2sm forces the 1-SM kernel or the CTA-pair
// kernel (for ablations and tests); it is read on every call. 0: the
// automatic choice.
int variant_override() {
    const char *v = std::getenv("SWIGLU_FUSED_VARIANT");
    if (!v) return 0;
    if (std::strcmp(v, "1sm") == 0) return 1;
    if (std::strcmp(v, "2sm") == 0) return 2;
    return 0;
}

struct DeviceState {
    std::once_flag once;
    int status = SWIGLU_OK;  // result of the one-time setup
    int sm_count = 0;
    int pair_clusters = 0;   // CTA pairs of the 2-SM kernel that can run at once
    // clusters of j CTAs of the decode down-projection kernel that can run at
    // once, j = 1..kDecodeMaxSplits (0: that size cannot be launched)
    int decode_clusters[kDecodeMaxSplits + 1] = {};
};

DeviceState g_devices[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn get_encode() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

// One-time per-device setup with that device current: check that it is an
// sm_103 part, cache its SM count and raise the kernel's shared-memory limit.
int device_setup(int *dev_out, DeviceState **st_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return SWIGLU_ERR_UNSUPPORTED;
    DeviceState &st = g_devices[dev];
    std::call_once(st.once, [&st, dev] {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            st.status = SWIGLU_ERR_CUDA;
            return;
        }
        if (major != 10 || minor != 3) {  // built for sm_103a only
            st.status = SWIGLU_ERR_UNSUPPORTED;
            return;
        }
        if (cudaFuncSetAttribute(fused_up_kernel<kFusedStages, 256, ElemBF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 FusedC::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_kernel<kNarrow64Stages, 128, ElemBF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Narrow64C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_kernel<kNarrow32Stages, 64, ElemBF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Narrow32C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_kernel<kNarrow64Stages, 128, ElemE4M3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Narrow64C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_kernel<kNarrow32Stages, 64, ElemE4M3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Narrow32C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_pair_kernel<kPairStages, ElemBF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairC::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_pair_kernel<kPairStages, ElemBF16, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairC::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_kernel<kFusedStages, 256, ElemE4M3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 FusedC::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_pair_kernel<kPairStages, ElemE4M3>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairC::SMEM_BYTES) != cudaSuccess ||
            // column-interleaved packed weights (BF16)
            cudaFuncSetAttribute(fused_up_kernel<kFusedStages, 256, ElemBF16, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 FusedC::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_kernel<kNarrow64Stages, 128, ElemBF16, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Narrow64C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_kernel<kNarrow32Stages, 64, ElemBF16, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Narrow32C::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(fused_up_pair_kernel<kPairStages, ElemBF16, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PairC::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(down_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 WideCfg::SMEM_BYTES) != cudaSuccess ||
            // plain product on the 1-SM kernel (decode-sized down-projection)
            cudaFuncSetAttribute(fused_up_kernel<kNarrow32Stages, 64, ElemBF16, false, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Narrow32C::SMEM_BYTES) != cudaSuccess ||
            // the decode down-projection kernel (swapped operands), per token block
            cudaFuncSetAttribute(down_decode_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DecodeCfg<32>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(down_decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DecodeCfg<64>::SMEM_BYTES) != cudaSuccess ||
            cudaFuncSetAttribute(down_decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 DecodeCfg<128>::SMEM_BYTES) != cudaSuccess ||
            // its clusters of up to 16 CTAs (more than the portable 8)
            cudaFuncSetAttribute(down_decode_kernel<32>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
            cudaFuncSetAttribute(down_decode_kernel<64>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
            cudaFuncSetAttribute(down_decode_kernel<128>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
            cudaGetLastError();
            st.status = SWIGLU_ERR_CUDA;
            return;
        }
        // how many CTA pairs fit at once (a cluster sits inside one GPC, so
        // not every SM count divides evenly)
        auto max_clusters = [sms](int ctas, auto kernel) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(ctas);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(sms / ctas * ctas));
            cfg.blockDim = dim3(PairC::THREADS);
            cfg.dynamicSmemBytes = PairC::SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg) != cudaSuccess) {
                cudaGetLastError();
                return -1;
            }
            return std::min(clusters, sms / ctas);
        };
        const int pairs = max_clusters(2, fused_up_pair_kernel<kPairStages, ElemBF16>);
        st.pair_clusters = pairs >= 1 ? pairs : sms / 2;
        // the decode kernel's clusters (a cluster sits inside one GPC: how
        // many of j CTAs fit depends on the GPCs' SM counts, not only on sms / j)
        for (int j = 1; j <= kDecodeMaxSplits; ++j) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = static_cast<unsigned>(j);
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.gridDim = dim3(static_cast<unsigned>(j * std::max(1, sms / j)));
            cfg.blockDim = dim3(DecodeCfg<128>::THREADS);
            cfg.dynamicSmemBytes = DecodeCfg<128>::SMEM_BYTES;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int clusters = 0;
            if (cudaOccupancyMaxActiveClusters(&clusters, down_decode_kernel<128>, &cfg) !=
                cudaSuccess) {
                cudaGetLastError();
                clusters = 0;
            }
            st.decode_clusters[j] = std::min(clusters, sms / j);
        }
        st.sm_count = sms;
        st.status = SWIGLU_OK;
    });
    *dev_out = dev;
    *st_out = &st;
    return st.status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count of the current device without the sm_103 check (for sizing only).
int current_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return kAssumedMaxSms;
    }
    return sms;
}

// Schedule of one call. `workers` = CTAs (1-SM kernel) or CTA pairs (2-SM
// kernel) that run at once; a 2-SM tile has 256 rows.
// SWIGLU_SCHEDULE=dp|split|sk|sk-tail|sk-aligned forces one schedule form
// (ablations; sk-aligned applies to the wide down-projection kernel only);
// unset or anything else: the automatic choice.
int schedule_mode() {
    const char *v = std::getenv("SWIGLU_SCHEDULE");
    if (!v) return kSchedAuto;
    if (std::strcmp(v, "dp") == 0) return kSchedDataParallel;
    if (std::strcmp(v, "split") == 0) return kSchedColumnSplit;
    if (std::strcmp(v, "sk") == 0) return kSchedStreamK;
    if (std::strcmp(v, "sk-tail") == 0) return kSchedStreamKTail;
    if (std::strcmp(v, "sk-aligned") == 0) return kSchedAligned;
    return kSchedAuto;
}
// The same for the fused kernels and the CTA-pair plain mode, which have no
// aligned form.
int schedule_mode_fused() {
    const int m = schedule_mode();
    return m == kSchedAligned ? kSchedAuto : m;
}

// SWIGLU_GROUP_M=<rows> (ablation): token rows per group of the tile order
// (a multiple of the kernel's tile height; default kGroupM * 128 = 2048);
// read on every call. 0: the default.
int group_rows_override() {
    const char *v = std::getenv("SWIGLU_GROUP_M");
    if (!v) return 0;
    const long r = std::strtol(v, nullptr, 10);
    return (r >= 128 && r <= (1L << 20)) ? static_cast<int>(r) : 0;
}

// Schedule for a kernel whose clusters hold `ctas` CTAs (1 or 2: tiles of
// 128 or 256 rows), `workers` of them running at once.
WorkSched plan_for(int64_t M, int64_t N, int64_t K, int workers, int ctas, int kbk, int mode) {
    const int rows = FusedC::BM * ctas;
    const int m_tiles = static_cast<int>((M + rows - 1) / rows);
    const int n_tiles = static_cast<int>((N + FusedC::BN - 1) / FusedC::BN);
    const int k_blocks = static_cast<int>((K + kbk - 1) / kbk);
    // few token rows: the kernel streams weights (HBM-bound), see plan_schedule
    const bool weight_bound = M <= 128;
    const int grows = group_rows_override();
    const int group_m = grows ? std::max(1, grows / rows) : kGroupM / ctas;
    return plan_schedule(m_tiles, n_tiles, k_blocks, workers, group_m, kMinStreamKIters,
                         weight_bound, mode);
}

// Schedule of the plain product out = Y x W3 (Y [M, N], W3 [N, K]) on the
// CTA-pair kernel's plain mode: tiles of 256 rows x 256 output columns,
// k-blocks over N. Its output has few tiles against a long reduction (the
// hidden size is a few times smaller than the intermediate size), so whole
// tiles are kept only when they fill at least 90% of the last wave and
// stream-K splits the k-blocks otherwise (a split tile's partial sums cost a
// few k-blocks of time against tiles of a hundred): over all tiles when there
// are fewer tiles than pairs, else over the tiles past the last full wave
// (7B, M=2048: 177 us against 201 us for all tiles and 185 us for whole
// tiles). With fewer tiles than pairs the grid is picked for the split's
// finishing cost (schedule.cuh, plan_stream_k_grid: 1.5B, 48 tiles, on 72 of
// the 76 pairs, two per tile). Column sub-tiles do not apply.
// SWIGLU_SK_PAIRS=<g> (ablation, read on every call) runs that stream-K over
// all tiles on g pairs instead (clamped to 1..workers).
WorkSched plan_down(int64_t M, int64_t N, int64_t K, int workers) {
    const int rows = FusedC::BM * 2;
    const int m_tiles = static_cast<int>((M + rows - 1) / rows);
    const int n_tiles = static_cast<int>((K + kDownTileCols - 1) / kDownTileCols);
    const int k_blocks = static_cast<int>((N + ElemBF16::kBK - 1) / ElemBF16::kBK);
    int mode = schedule_mode_fused();
    if (mode == kSchedColumnSplit) mode = kSchedAuto;
    if (mode == kSchedAuto) {
        const long long T = static_cast<long long>(m_tiles) * n_tiles;
        const long long waves = (T + workers - 1) / workers;
        const double eff = static_cast<double>(T) / (static_cast<double>(waves) * workers);
        mode = eff >= 0.9 ? kSchedDataParallel : (T >= workers ? kSchedStreamKTail : kSchedStreamK);
    }
    const int grows = group_rows_override();
    const int group_m = grows ? std::max(1, grows / rows) : kGroupM / 2;
    if (mode == kSchedStreamK) {
        if (const char *v = std::getenv("SWIGLU_SK_PAIRS")) {
            const int g = std::atoi(v);
            if (g >= 1)
                return plan_schedule(m_tiles, n_tiles, k_blocks, std::min(g, workers), group_m,
                                     kMinStreamKIters, false, kSchedStreamK);
        }
    }
    if (mode == kSchedStreamK && schedule_mode_fused() == kSchedAuto)
        return plan_stream_k_grid(m_tiles, n_tiles, k_blocks, workers, group_m, kMinStreamKIters);
    return plan_schedule(m_tiles, n_tiles, k_blocks, workers, group_m, kMinStreamKIters, false,
                         mode);
}

// Schedule of the plain product on the 1-SM kernel (tiles of 128 rows x 64
// output columns, k-blocks over N). A decode-sized product streams W3 from
// HBM, and the four 64-column tiles of one packed 256-column weight tile read
// the four 8 KB quarters of each 32 KB block: they should do so at the same
// time. So with fewer tiles than SMs every tile is cut into j = floor(SMs /
// tiles) equal K ranges, one per CTA (each CTA one unit; the j CTAs of a
// range index r of the four sibling tiles run in step), as long as a range
// keeps kMinStreamKIters k-blocks; with j = 1, whole tiles. Stream-K over all
// tiles on all SMs had the siblings at unrelated k offsets (7B, M=16: the
// weights arrived at ~4.4 TB/s). With at least as many tiles as SMs: whole
// tiles when they fill 90% of the last wave, else stream-K over the tail.
WorkSched plan_down_slim(int64_t M, int64_t N, int64_t K, int sms) {
    const int m_tiles = static_cast<int>((M + FusedC::BM - 1) / FusedC::BM);
    const int n_tiles = static_cast<int>((K + 63) / 64);
    const int k_blocks = static_cast<int>((N + ElemBF16::kBK - 1) / ElemBF16::kBK);
    const int grows = group_rows_override();
    const int group_m = grows ? std::max(1, grows / FusedC::BM) : kGroupM;
    int mode = schedule_mode_fused();
    if (mode == kSchedColumnSplit) mode = kSchedAuto;
    const long long T = static_cast<long long>(m_tiles) * n_tiles;
    if (mode == kSchedAuto && T < sms) {
        const int j = std::min(static_cast<int>(sms / T), k_blocks / kMinStreamKIters);
        if (j >= 2) {
            const WorkSched s = plan_schedule(m_tiles, n_tiles, k_blocks, static_cast<int>(j * T),
                                              group_m, kMinStreamKIters, false, kSchedStreamK);
            if (s.grid == j * T && s.dp_tiles == 0) return s;
        }
        return plan_schedule(m_tiles, n_tiles, k_blocks, sms, group_m, kMinStreamKIters, false,
                             kSchedDataParallel);
    }
    if (mode == kSchedAuto) {
        const long long waves = (T + sms - 1) / sms;
        const double eff = static_cast<double>(T) / (static_cast<double>(waves) * sms);
        mode = eff >= 0.9 ? kSchedDataParallel : kSchedStreamKTail;
    }
    return plan_schedule(m_tiles, n_tiles, k_blocks, sms, group_m, kMinStreamKIters, false, mode);
}

// Split of the decode down-projection kernel (down_decode_kernel.cuh): its
// T = ceil(K / 128) tiles of 128 output columns (all token rows at once) are
// each cut into j equal K ranges, one per CTA, the j CTAs of a tile forming a
// cluster; j from plan_decode_splits (schedule.cuh). Measured on GB300
// (graph-replayed calls, us): 7B M=16 (28 tiles) j=3 30.0, j=4 24.5, j=5
// 25.4; 32B M=64 (40 tiles) j=2 61.6, j=3 46.1; 72B M=32 (64 tiles) j=2
// 76.3; the 0.5B shape (7 tiles) j=8 8.6, j=16 8.3; 1.5B M=16 (12 tiles)
// j=8 9.4, j=10 9.0. SWIGLU_SCHEDULE=dp forces j = 1, SWIGLU_DECODE_SPLITS=<j>
// any j (clamped to 1..16 and the k-blocks; more clusters than fit at once
// then run in waves); both are read on every call.
int plan_down_decode(int64_t N, int64_t K, int sms, const int *clusters) {
    const int64_t T = (K + 127) / 128;
    const int k_blocks = static_cast<int>((N + ElemBF16::kBK - 1) / ElemBF16::kBK);
    if (const char *v = std::getenv("SWIGLU_DECODE_SPLITS")) {
        const int j = std::atoi(v);
        if (j >= 1) return std::min(j, std::min(kDecodeMaxSplits, k_blocks));
    }
    if (schedule_mode() == kSchedDataParallel) return 1;
    return plan_decode_splits(T, k_blocks, sms, clusters, kDecodeMaxSplits);
}

// The down-projection's kernel and schedule. Four kernels serve it, on the
// same packed W3:
//   * kDownDecode (down_decode_kernel.cuh, swapped operands: tiles of 128
//     output columns x all token rows, split K ranges summed inside a
//     cluster, plan_down_decode): every product of up to kDecodeMaxM rows
//     (0.5B, M=128: 8.0 us; the 1-SM plain mode below took 14.4 us and
//     the CTA-pair kernel 41 us);
//   * kDownWide (down_wide_kernel.cuh, CTA pairs, tiles of 256 x 512): a
//     third fewer operand bytes per flop than 256-column tiles, which shows
//     at the power cap as a higher SM clock (7B, M=8192: 631 against 666 us;
//     72B, M=8192: 2261 against 2361 us), but one accumulator stage and
//     512-column FP32 partials for split tiles; it takes a call when whole
//     wide tiles fill at least 90% of their last wave (from kWideMinM rows
//     on), as whole tiles;
//   * kDownPair (the CTA-pair kernel's plain mode, 256 x 256, plan_down):
//     the rest (few output tiles for the pairs, e.g. the 1.5B and 7B M=2048
//     shapes);
//   * kDownSlim (the 1-SM kernel's plain mode, tiles of 128 x 64,
//     plan_down_slim): forced only (ablations and tests).
// SWIGLU_DOWN_TILE=64|128|256|512, read on every call, forces one of them
// (128 only up to kDecodeMaxM rows); with the wide kernel forced,
// SWIGLU_SCHEDULE picks its form (dp, sk, sk-tail, sk-aligned; whole tiles
// otherwise).
enum DownKind { kDownPair = 0, kDownWide = 1, kDownSlim = 2, kDownDecode = 3 };
struct DownPlan {
    int kind;
    WorkSched sched;
    int splits;   // kDownDecode: K ranges per tile (cluster size)
};
// `decode_clusters`: DeviceState::decode_clusters, or null (no device: the
// decode split is then planned as if clusters of any size filled the GPU,
// which changes nothing the caller sees, as that kernel needs no workspace).
DownPlan plan_down_any(int64_t M, int64_t N, int64_t K, int workers, int sms,
                       const int *decode_clusters) {
    const int rows = WideCfg::UMMA_M;
    const int m_tiles = static_cast<int>((M + rows - 1) / rows);
    const int n_tiles = static_cast<int>((K + WideCfg::TILE_N - 1) / WideCfg::TILE_N);
    const int k_blocks = static_cast<int>((N + ElemBF16::kBK - 1) / ElemBF16::kBK);
    const long long T = static_cast<long long>(m_tiles) * n_tiles;
    const long long waves = (T + workers - 1) / workers;
    const double eff = static_cast<double>(T) / (static_cast<double>(waves) * workers);
    int kind = M <= kDecodeMaxM ? kDownDecode
                                : (M >= kWideMinM && eff >= 0.9 ? kDownWide : kDownPair);
    const char *v = std::getenv("SWIGLU_DOWN_TILE");
    if (v && std::strcmp(v, "64") == 0) kind = kDownSlim;
    if (v && std::strcmp(v, "128") == 0 && M <= kDecodeMaxM) kind = kDownDecode;
    if (v && std::strcmp(v, "256") == 0) kind = kDownPair;
    if (v && std::strcmp(v, "512") == 0) kind = kDownWide;
    if (kind == kDownDecode)
        return {kDownDecode, WorkSched{}, plan_down_decode(N, K, sms, decode_clusters)};
    if (kind == kDownPair) return {kDownPair, plan_down(M, N, K, workers), 1};
    if (kind == kDownSlim) return {kDownSlim, plan_down_slim(M, N, K, sms), 1};
    const int grows = group_rows_override();
    const int group_m = grows ? std::max(1, grows / rows) : kGroupM / 2;
    return {kDownWide,
            plan_down_wide(m_tiles, n_tiles, k_blocks, workers, group_m, kMinStreamKIters,
                           schedule_mode()),
            1};
}

// Which kernel serves a call, and its schedule: the 1-SM kernel below 256
// rows, the CTA-pair kernel from there on.
struct LaunchPlan {
    int ctas;        // CTAs per cluster: 1 or 2
    WorkSched sched;
};
LaunchPlan choose_plan(int64_t M, int64_t N, int64_t K, int sms, int pair_clusters, int kbk) {
    const int v = variant_override();
    const int mode = schedule_mode_fused();
    if (v == 1 || (v == 0 && M < kPairMinM)) return {1, plan_for(M, N, K, sms, 1, kbk, mode)};
    return {2, plan_for(M, N, K, pair_clusters, 2, kbk, mode)};
}

// Workspace layout: a counter region at offset 0 whose size depends only on
// the device (so a counter never lands where another shape's call left
// partial sums), then the partial slots. There are fewer than 2 * grid
// stream-K tiles; a tile needs at most one counter per CTA half in the fused
// kernels and one per CTA half and part (4) in the wide down-projection
// kernel, so 16 * sm_count counters always suffice; after them come the
// CTA-pair kernel's start-order ticket counter and its dynamic-tile counter
// pair (next tile, pairs finished).
int ticket_index(int sm_count) { return 16 * sm_count; }
int tile_counter_index(int sm_count) { return 16 * sm_count + 1; }
size_t counter_region_bytes(int sm_count) {
    return (static_cast<size_t>(16 * sm_count + 3) * sizeof(unsigned int) + 255) / 256 * 256;
}

// Whether a CTA-pair launch hands out its tiles at run time (whole tiles
// only): automatically from kDynamicMinWaves waves of tiles on, where the
// pairs' drift costs DRAM re-reads (72B, M=8192, 97 waves: 15.2 -> 4.7 GB
// read per launch, 2% faster at the power cap) and the ring's hand-offs
// cost nothing (7B M=512, 3.9 waves: 1% slower dynamic, so static there).
// SWIGLU_DYNAMIC_TILES=0 keeps the static order everywhere, =1 takes the
// dynamic one from two waves on (ablations and tests); read on every call.
constexpr int kDynamicMinWaves = 8;
bool dynamic_tiles(const WorkSched &s, bool pair) {
    if (!pair || s.sk_iters != 0 || s.n_split != 1) return false;
    const char *v = std::getenv("SWIGLU_DYNAMIC_TILES");
    if (v && std::strcmp(v, "0") == 0) return false;
    const int min_waves = (v && std::strcmp(v, "1") == 0) ? 2 : kDynamicMinWaves;
    return s.num_tiles >= static_cast<long long>(min_waves) * s.grid;
}
// Partial slots: 2 per worker (its first and last stream-K tile), and for
// the 2-SM kernel one per CTA of the pair.
size_t workspace_partials_bytes(const WorkSched &s, int64_t M, bool pair) {
    return s.sk_iters > 0 ? static_cast<size_t>(2) * s.grid * (pair ? 2 : 1) * kSlotCols *
                                slot_rows_for(M) * sizeof(float)
                          : 0;
}
size_t workspace_bytes_for(const WorkSched &s, int64_t M, bool pair, int sm_count) {
    if (s.sk_iters == 0) return dynamic_tiles(s, pair) ? counter_region_bytes(sm_count) : 0;
    return counter_region_bytes(sm_count) + workspace_partials_bytes(s, M, pair);
}
// The down-projection's: the wide kernel keeps 2 slots per worker and CTA
// half of a whole FP32 partial tile half (128 rows x 512 columns).
size_t down_workspace_bytes_for(const DownPlan &p, int64_t M, int sm_count) {
    if (p.kind == kDownDecode) return 0;   // split tiles are summed inside their cluster
    if (p.kind != kDownWide) return workspace_bytes_for(p.sched, M, p.kind == kDownPair, sm_count);
    if (p.sched.sk_iters == 0) return 0;
    return counter_region_bytes(sm_count) + static_cast<size_t>(2) * p.sched.grid * 2 *
                                                WideCfg::SLOT_FLOATS * sizeof(float);
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// Tensor map over the tile-contiguous packed weights [tiles][256][row]: a
// box is box_rows rows of one tile (the whole 32 KB tile for the 1-SM kernel,
// the Gate or the Up half for one CTA of a pair, or a column sub-tile's rows),
// 128-byte swizzled. `elems` is the row length in elements (64 BF16 or 128
// FP8 values: 128 bytes either way).
bool encode_packed_weights(CUtensorMap *m, const void *base, uint64_t tiles, uint32_t box_rows,
                           bool fp8) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const uint64_t elems = fp8 ? 128 : 64;
    const cuuint64_t dims[3] = {elems, 256, tiles};
    const cuuint64_t strides[2] = {128, 256 * 128};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(elems), box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same packed weights as 4-D [tiles][2 halves][128 rows][row], with a box
// of `box_rows` rows from BOTH halves: the Gate rows and the matching Up rows
// of a column sub-tile in one load (they land back to back in shared memory).
bool encode_packed_weight_halves(CUtensorMap *m, const void *base, uint64_t tiles,
                                 uint32_t box_rows, bool fp8) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const uint64_t elems = fp8 ? 128 : 64;
    const cuuint64_t dims[4] = {elems, 128, 2, tiles};
    const cuuint64_t strides[3] = {128, 128 * 128, 256 * 128};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(elems), box_rows, 2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map over a row-major [rows, cols] matrix of BF16 (2-byte) or
// FP8 (1-byte) elements with a 128-byte-swizzled box of box_rows x box_cols
// (box_cols * element size <= 128 bytes).
bool encode_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows, bool fp8 = false) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const uint64_t esize = fp8 ? 1 : 2;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * esize};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace swiglu

using namespace swiglu;

extern "C" {

#ifdef SWIGLU_TEST_FAULT_INJECTION
// Exists only in the test-only fault-injection build (never in the product
// library): makes the following launches leave their first pipeline stage
// unfilled, so a bounded wait runs out and the timeout path can be tested.
void swiglu_test_set_fault_injection(int skip_first_fill) {
    swiglu::g_test_skip_first_fill = skip_first_fill;
}
#endif

int swiglu_version(void) { return (0 << 16) | 1; }

const char *swiglu_status_string(int status) {
    switch (status) {
        case SWIGLU_OK: return "SWIGLU_OK";
        case SWIGLU_ERR_INVALID_ARG: return "SWIGLU_ERR_INVALID_ARG";
        case SWIGLU_ERR_UNSUPPORTED: return "SWIGLU_ERR_UNSUPPORTED";
        case SWIGLU_ERR_CUDA: return "SWIGLU_ERR_CUDA";
        case SWIGLU_ERR_DEVICE_TIMEOUT: return "SWIGLU_ERR_DEVICE_TIMEOUT";
        default: return "SWIGLU_ERR_UNKNOWN";
    }
}

size_t swiglu_packed_weight_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return static_cast<size_t>(2 * round_up(N, 128)) * static_cast<size_t>(round_up(K, 64)) * 2u;
}

// Argument checks shared by both pack entry points; on success returns the
// launch grid. The weights are 2*K*N elements each way round.
static int pack_checks(const void *W1, const void *W2, int64_t K, int64_t N, void *Wpacked,
                       dim3 *grid) {
    if (!W1 || !W2 || !Wpacked) return SWIGLU_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || (K % 8) != 0 || (N % 8) != 0) return SWIGLU_ERR_INVALID_ARG;
    if (K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return SWIGLU_ERR_INVALID_ARG;
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(Wpacked)) return SWIGLU_ERR_INVALID_ARG;
    const size_t wbytes = static_cast<size_t>(K) * N * 2;
    const size_t pbytes = swiglu_packed_weight_bytes(N, K);
    if (overlaps(Wpacked, pbytes, W1, wbytes) || overlaps(Wpacked, pbytes, W2, wbytes))
        return SWIGLU_ERR_INVALID_ARG;
    const int64_t rows = 2 * round_up(N, 128);
    const int64_t kblocks = (K + kPackTile - 1) / kPackTile;
    if (rows / kPackTile > 65535) return SWIGLU_ERR_UNSUPPORTED;
    *grid = dim3(static_cast<unsigned>(kblocks), static_cast<unsigned>(rows / kPackTile));
    return SWIGLU_OK;
}

int swiglu_pack_weights(const void *W1, const void *W2, int64_t K, int64_t N, void *Wpacked,
                        void *stream) {
    dim3 grid;
    int s = pack_checks(W1, W2, K, N, Wpacked, &grid);
    if (s != SWIGLU_OK) return s;
    int dev;
    DeviceState *st;
    s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    pack_weights_kernel<uint16_t, 64><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(W1), static_cast<const uint16_t *>(W2),
        static_cast<uint16_t *>(Wpacked), static_cast<int>(K), static_cast<int>(N),
        static_cast<int>(grid.x));
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}

int swiglu_pack_weights_nk(const void *W1, const void *W2, int64_t N, int64_t K, void *Wpacked,
                           void *stream) {
    dim3 grid;
    int s = pack_checks(W1, W2, K, N, Wpacked, &grid);
    if (s != SWIGLU_OK) return s;
    int dev;
    DeviceState *st;
    s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    pack_weights_nk_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(W1), static_cast<const uint16_t *>(W2),
        static_cast<uint16_t *>(Wpacked), static_cast<int>(K), static_cast<int>(N),
        static_cast<int>(grid.x));
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}

}  // extern "C"

namespace swiglu {
namespace {

// Workspace bytes for a forward of element type E (same plan as the launch).
template <typename E>
size_t workspace_bytes_impl(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
        K >= (int64_t(1) << 31))
        return 0;
    int dev;
    DeviceState *st;
    if (device_setup(&dev, &st) == SWIGLU_OK) {  // the same plan the forward will use
        const LaunchPlan lp = choose_plan(M, N, K, st->sm_count, st->pair_clusters, E::kBK);
        return workspace_bytes_for(lp.sched, M, lp.ctas == 2, st->sm_count);
    }
    const int sms = current_sm_count();         // no usable device: a size for its SM count
    const LaunchPlan lp = choose_plan(M, N, K, sms, sms / 2, E::kBK);
    return workspace_bytes_for(lp.sched, M, lp.ctas == 2, sms);
}

// The fused forward for element type E (BF16, or FP8 E4M3 with per-tensor
// scales folded into gate_scale / up_scale). A and Wpacked hold E elements;
// Y is BF16. IL: Wpacked is column-interleaved (swiglu_pack_weights_interleaved).
template <typename E, bool IL = false>
int forward_impl(const void *A, const void *Wpacked, void *Y, int64_t M, int64_t N, int64_t K,
                 float gate_scale, float up_scale, void *workspace, size_t workspace_bytes,
                 void *stream, size_t packed_bytes, bool late_trigger = false) {
    const size_t esize = E::kFp8 ? 1 : 2;
    const int64_t kmul = E::kFp8 ? 16 : 8;   // 16-byte rows of A
    if (!A || !Wpacked || !Y) return SWIGLU_ERR_INVALID_ARG;
    if (M < 1 || N < 8 || K < kmul || (N % 8) != 0 || (K % kmul) != 0) return SWIGLU_ERR_INVALID_ARG;
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || K >= lim) return SWIGLU_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(Wpacked) || !aligned16(Y)) return SWIGLU_ERR_INVALID_ARG;
    const size_t ybytes = static_cast<size_t>(M) * N * 2;
    const size_t abytes = static_cast<size_t>(M) * K * esize;
    if (overlaps(Y, ybytes, A, abytes) || overlaps(Y, ybytes, Wpacked, packed_bytes))
        return SWIGLU_ERR_INVALID_ARG;
    const int64_t tiles = ((M + FusedC::BM - 1) / FusedC::BM) * ((N + FusedC::BN - 1) / FusedC::BN);
    if (tiles >= lim) return SWIGLU_ERR_UNSUPPORTED;

    int dev;
    DeviceState *st;
    const int s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;

    const LaunchPlan lp = choose_plan(M, N, K, st->sm_count, st->pair_clusters, E::kBK);
    const WorkSched &sched = lp.sched;
    const bool pair = lp.ctas == 2;
    const size_t ws_need = workspace_bytes_for(sched, M, pair, st->sm_count);
    if (ws_need > 0) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
            workspace_bytes < ws_need)
            return SWIGLU_ERR_INVALID_ARG;
        if (overlaps(workspace, ws_need, Y, ybytes) || overlaps(workspace, ws_need, A, abytes) ||
            overlaps(workspace, ws_need, Wpacked, packed_bytes))
            return SWIGLU_ERR_INVALID_ARG;
    }

    // A box: 128 rows, or ceil(M/8)*8 when the whole problem has fewer rows
    // (1-SM kernel only; a pair tile always loads 128 rows per CTA)
    const int a_rows =
        (pair || M >= FusedC::BM) ? FusedC::BM : static_cast<int>(round_up(M, 8));
    const uint64_t weight_tiles =
        static_cast<uint64_t>(sched.order.n_tiles) * static_cast<uint64_t>(sched.k_blocks);
    CUtensorMap tmA, tmB, tmB64, tmB32, tmY;
    if (!encode_2d(&tmA, A, K, M, E::kBK, a_rows, E::kFp8) ||
        !encode_packed_weights(&tmB, Wpacked, weight_tiles, pair ? 128u : 256u, E::kFp8) ||
        // sub-tile maps: the pair kernels load one half (Gate or Up) per CTA,
        // the 1-SM kernel both halves in one 4-D box (interleaved weights: the
        // sub-tile's 2 * width contiguous rows in one 3-D box)
        !(pair ? encode_packed_weights(&tmB64, Wpacked, weight_tiles, 64u, E::kFp8)
               : IL ? encode_packed_weights(&tmB64, Wpacked, weight_tiles, 128u, E::kFp8)
                    : encode_packed_weight_halves(&tmB64, Wpacked, weight_tiles, 64u, E::kFp8)) ||
        !(pair ? encode_packed_weights(&tmB32, Wpacked, weight_tiles, 32u, E::kFp8)
               : IL ? encode_packed_weights(&tmB32, Wpacked, weight_tiles, 64u, E::kFp8)
                    : encode_packed_weight_halves(&tmB32, Wpacked, weight_tiles, 32u, E::kFp8)) ||
        !encode_2d(&tmY, Y, N, M, 64, 32))
        return SWIGLU_ERR_CUDA;

    FusedArgs args{};
    args.M = static_cast<int>(M);
    args.N = static_cast<int>(N);
    args.K = static_cast<int>(K);
    args.stage_tx_bytes = a_rows * kRowBytes + FusedC::B_BYTES;
    args.a_tx_bytes = a_rows * kRowBytes;
    args.Y = static_cast<uint16_t *>(Y);
    args.gate_scale = gate_scale;
    args.up_scale = up_scale;
    args.slot_rows = slot_rows_for(M);
    args.sched = sched;
#ifdef SWIGLU_TEST_FAULT_INJECTION
    args.skip_first_fill = g_test_skip_first_fill;
#endif
    args.counters = ws_need ? static_cast<unsigned int *>(workspace) : nullptr;
    args.partials = ws_need ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                        counter_region_bytes(st->sm_count))
                            : nullptr;
    args.ticket_index = ticket_index(st->sm_count);
    args.tile_counter_index = tile_counter_index(st->sm_count);
    args.dyn_tiles = dynamic_tiles(sched, pair) ? 1 : 0;
    args.late_trigger = late_trigger ? 1 : 0;

    // Both kernels are launched with programmatic stream serialization: a
    // launch may begin while the previous kernel in the stream finishes; the
    // kernel waits (griddepcontrol.wait) before it reads or writes global
    // memory, so stream order is kept for every buffer.
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cudaError_t err;
    if (pair) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = static_cast<unsigned>(lp.ctas);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        cfg.gridDim = dim3(static_cast<unsigned>(lp.ctas * sched.grid));
        cfg.blockDim = dim3(PairC::THREADS);
        cfg.dynamicSmemBytes = PairC::SMEM_BYTES;
        err = cudaLaunchKernelEx(&cfg, fused_up_pair_kernel<kPairStages, E, false, IL>, tmA, tmB,
                                 tmB64, tmB32, tmY, args);
    } else {
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(sched.grid));
        cfg.blockDim = dim3(FusedC::THREADS);
        // A launch made only of column sub-tiles takes a narrow configuration:
        // stages sized for its sub-tile, so more loads are in flight per SM.
        const bool all_sub = sched.n_split > 1 && sched.dp_tiles == 0 && sched.sk_iters == 0;
        if (all_sub && sched.n_split == 2) {
            cfg.dynamicSmemBytes = Narrow64C::SMEM_BYTES;
            err = cudaLaunchKernelEx(&cfg, fused_up_kernel<kNarrow64Stages, 128, E, IL>, tmA, tmB,
                                     tmB64, tmB32, tmY, args);
        } else if (all_sub && sched.n_split == 4) {
            cfg.dynamicSmemBytes = Narrow32C::SMEM_BYTES;
            err = cudaLaunchKernelEx(&cfg, fused_up_kernel<kNarrow32Stages, 64, E, IL>, tmA, tmB,
                                     tmB64, tmB32, tmY, args);
        } else {
            cfg.dynamicSmemBytes = FusedC::SMEM_BYTES;
            err = cudaLaunchKernelEx(&cfg, fused_up_kernel<kFusedStages, 256, E, IL>, tmA, tmB,
                                     tmB64, tmB32, tmY, args);
        }
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    return SWIGLU_OK;
}

}  // namespace
}  // namespace swiglu

extern "C" {

size_t swiglu_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return workspace_bytes_impl<ElemBF16>(M, N, K);
}

int swiglu_up_forward(const void *A, const void *Wpacked, void *Y, int64_t M, int64_t N,
                      int64_t K, void *workspace, size_t workspace_bytes, void *stream) {
    return forward_impl<ElemBF16>(A, Wpacked, Y, M, N, K, 1.0f, 1.0f, workspace,
                                  workspace_bytes, stream, swiglu_packed_weight_bytes(N, K));
}

int swiglu_pack_weights_interleaved(const void *W1, const void *W2, int64_t K, int64_t N,
                                    void *Wpacked, void *stream) {
    dim3 grid;
    int s = pack_checks(W1, W2, K, N, Wpacked, &grid);
    if (s != SWIGLU_OK) return s;
    int dev;
    DeviceState *st;
    s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    pack_weights_il_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(W1), static_cast<const uint16_t *>(W2),
        static_cast<uint16_t *>(Wpacked), static_cast<int>(K), static_cast<int>(N),
        static_cast<int>(grid.x));
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}

int swiglu_up_forward_interleaved(const void *A, const void *Wpacked, void *Y, int64_t M,
                                  int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                                  void *stream) {
    return forward_impl<ElemBF16, true>(A, Wpacked, Y, M, N, K, 1.0f, 1.0f, workspace,
                                        workspace_bytes, stream, swiglu_packed_weight_bytes(N, K));
}

size_t swiglu_packed_weight_bytes_fp8(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return static_cast<size_t>(2 * round_up(N, 128)) * static_cast<size_t>(round_up(K, 128));
}

int swiglu_pack_weights_fp8(const void *W1, const void *W2, int64_t K, int64_t N, void *Wpacked,
                            void *stream) {
    if (!W1 || !W2 || !Wpacked) return SWIGLU_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || (K % 16) != 0 || (N % 8) != 0) return SWIGLU_ERR_INVALID_ARG;
    if (K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return SWIGLU_ERR_INVALID_ARG;
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(Wpacked)) return SWIGLU_ERR_INVALID_ARG;
    const size_t wbytes = static_cast<size_t>(K) * N;
    const size_t pbytes = swiglu_packed_weight_bytes_fp8(N, K);
    if (overlaps(Wpacked, pbytes, W1, wbytes) || overlaps(Wpacked, pbytes, W2, wbytes))
        return SWIGLU_ERR_INVALID_ARG;
    const int64_t rows = 2 * round_up(N, 128);
    const int64_t kblocks = (K + 127) / 128;
    if (rows / kPackTile > 65535) return SWIGLU_ERR_UNSUPPORTED;
    int dev;
    DeviceState *st;
    const int s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    const dim3 grid(static_cast<unsigned>(kblocks), static_cast<unsigned>(rows / kPackTile));
    pack_weights_kernel<uint8_t, 128><<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t *>(W1), static_cast<const uint8_t *>(W2),
        static_cast<uint8_t *>(Wpacked), static_cast<int>(K), static_cast<int>(N),
        static_cast<int>(kblocks));
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}

size_t swiglu_workspace_bytes_fp8(int64_t M, int64_t N, int64_t K) {
    return workspace_bytes_impl<ElemE4M3>(M, N, K);
}

int swiglu_up_forward_fp8(const void *A8, const void *Wpacked8, void *Y, int64_t M, int64_t N,
                          int64_t K, float scale_a, float scale_w1, float scale_w2, void *workspace,
                          size_t workspace_bytes, void *stream) {
    const float gs = scale_a * scale_w1, us = scale_a * scale_w2;
    if (!(scale_a > 0.0f) || !(scale_w1 > 0.0f) || !(scale_w2 > 0.0f) || !isfinite(scale_a) ||
        !isfinite(scale_w1) || !isfinite(scale_w2) || !isfinite(gs) || !isfinite(us) ||
        !(gs > 0.0f) || !(us > 0.0f))
        return SWIGLU_ERR_INVALID_ARG;   // also rejects NaN, and products that leave FP32
    return forward_impl<ElemE4M3>(A8, Wpacked8, Y, M, N, K, gs, us, workspace, workspace_bytes, stream,
                                  swiglu_packed_weight_bytes_fp8(N, K));
}

}  // extern "C"

namespace swiglu {
namespace {

size_t down_workspace_bytes_impl(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
        K >= (int64_t(1) << 31))
        return 0;
    int dev;
    DeviceState *st;
    if (device_setup(&dev, &st) == SWIGLU_OK)
        return down_workspace_bytes_for(
            plan_down_any(M, N, K, st->pair_clusters, st->sm_count, st->decode_clusters), M,
            st->sm_count);
    const int sms = current_sm_count();
    return down_workspace_bytes_for(plan_down_any(M, N, K, sms / 2, sms, nullptr), M, sms);
}

// Argument checks of the plain product out [M, K] = Y [M, N] x W3 [N, K].
int down_checks(const void *Y, const void *W3packed, const void *out, int64_t M, int64_t N,
                int64_t K) {
    if (!Y || !W3packed || !out) return SWIGLU_ERR_INVALID_ARG;
    if (M < 1 || N < 8 || K < 8 || (N % 8) != 0 || (K % 8) != 0) return SWIGLU_ERR_INVALID_ARG;
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || K >= lim) return SWIGLU_ERR_INVALID_ARG;
    if (!aligned16(Y) || !aligned16(W3packed) || !aligned16(out)) return SWIGLU_ERR_INVALID_ARG;
    const size_t obytes = static_cast<size_t>(M) * K * 2;
    if (overlaps(out, obytes, Y, static_cast<size_t>(M) * N * 2) ||
        overlaps(out, obytes, W3packed, swiglu_down_packed_weight_bytes(N, K)))
        return SWIGLU_ERR_INVALID_ARG;
    return SWIGLU_OK;
}

// The wide kernel's launch (plan from plan_down_any, checks done).
int down_wide_launch(const WorkSched &sched, const void *Y, const void *W3packed, void *out,
                     int64_t M, int64_t N, int64_t K, void *workspace, bool ws, int sm_count,
                     void *stream) {
    const int kt = static_cast<int>((K + kDownTileCols - 1) / kDownTileCols);
    const uint64_t weight_tiles = static_cast<uint64_t>(kt) * static_cast<uint64_t>(sched.k_blocks);
    CUtensorMap tmA, tmB, tmOut;
    if (!encode_2d(&tmA, Y, N, M, ElemBF16::kBK, WideCfg::BM) ||
        !encode_packed_weights(&tmB, W3packed, weight_tiles, 128u, false) ||
        !encode_2d(&tmOut, out, K, M, 64, 32))
        return SWIGLU_ERR_CUDA;
    WideArgs args{};
    args.M = static_cast<int>(M);
    args.N = static_cast<int>(K);   // output columns
    args.K = static_cast<int>(N);   // reduction
    args.kt_tiles = kt;
    args.sched = sched;
    args.counters = ws ? static_cast<unsigned int *>(workspace) : nullptr;
    args.partials = ws ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                   counter_region_bytes(sm_count))
                       : nullptr;
#ifdef SWIGLU_TEST_FAULT_INJECTION
    args.skip_first_fill = g_test_skip_first_fill;
#endif
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * sched.grid));
    cfg.blockDim = dim3(WideCfg::THREADS);
    cfg.dynamicSmemBytes = WideCfg::SMEM_BYTES;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, down_wide_kernel, tmA, tmB, tmOut, args);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    return SWIGLU_OK;
}

// The decode kernel's launch (plan from plan_down_any, checks done; M <= 128):
// ceil(K / 128) * splits CTAs in clusters of `splits`; `clusters` as in
// DeviceState (a size of which none fits is refused).
int down_decode_launch(int splits, const int *clusters, const void *Y, const void *W3packed,
                       void *out, int64_t M, int64_t N, int64_t K, void *stream,
                       bool weights_early) {
    const int kt = static_cast<int>((K + kDownTileCols - 1) / kDownTileCols);
    const int k_blocks = static_cast<int>((N + ElemBF16::kBK - 1) / ElemBF16::kBK);
    const int64_t tiles = (K + 127) / 128;
    if (splits < 1 || splits > kDecodeMaxSplits || splits > k_blocks ||
        tiles * splits > int64_t(1) << 30 || (splits > 1 && clusters[splits] < 1))
        return SWIGLU_ERR_UNSUPPORTED;
    const uint64_t weight_tiles = static_cast<uint64_t>(kt) * static_cast<uint64_t>(k_blocks);
    const int mt = static_cast<int>(round_up(M, 16));
    CUtensorMap tmY, tmW;
    if (!encode_2d(&tmY, Y, N, M, ElemBF16::kBK, static_cast<uint32_t>(mt)) ||
        !encode_packed_weights(&tmW, W3packed, weight_tiles, 128u, false))
        return SWIGLU_ERR_CUDA;
    DecodeArgs args{};
    args.M = static_cast<int>(M);
    args.N = static_cast<int>(K);   // output columns
    args.mt = mt;
    args.k_blocks = k_blocks;
    args.splits = splits;
    args.weights_early = weights_early ? 1 : 0;
    args.out = static_cast<uint16_t *>(out);
#ifdef SWIGLU_TEST_FAULT_INJECTION
    args.skip_first_fill = g_test_skip_first_fill;
#endif
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(splits);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = splits > 1 ? 2 : 1;
    cfg.gridDim = dim3(static_cast<unsigned>(tiles * splits));
    cudaError_t err;
    if (mt <= 32) {
        cfg.blockDim = dim3(DecodeCfg<32>::THREADS);
        cfg.dynamicSmemBytes = DecodeCfg<32>::SMEM_BYTES;
        err = cudaLaunchKernelEx(&cfg, down_decode_kernel<32>, tmY, tmW, args);
    } else if (mt <= 64) {
        cfg.blockDim = dim3(DecodeCfg<64>::THREADS);
        cfg.dynamicSmemBytes = DecodeCfg<64>::SMEM_BYTES;
        err = cudaLaunchKernelEx(&cfg, down_decode_kernel<64>, tmY, tmW, args);
    } else {
        cfg.blockDim = dim3(DecodeCfg<128>::THREADS);
        cfg.dynamicSmemBytes = DecodeCfg<128>::SMEM_BYTES;
        err = cudaLaunchKernelEx(&cfg, down_decode_kernel<128>, tmY, tmW, args);
    }
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    return SWIGLU_OK;
}

// The 1-SM kernel's plain-mode launch (plan from plan_down_any, checks done).
int down_slim_launch(const WorkSched &sched, const void *Y, const void *W3packed, void *out,
                     int64_t M, int64_t N, int64_t K, void *workspace, bool ws, int sm_count,
                     void *stream) {
    const int kt = static_cast<int>((K + kDownTileCols - 1) / kDownTileCols);
    const uint64_t weight_tiles = static_cast<uint64_t>(kt) * static_cast<uint64_t>(sched.k_blocks);
    const int a_rows = M >= FusedC::BM ? FusedC::BM : static_cast<int>(round_up(M, 8));
    CUtensorMap tmA, tmB, tmOut;
    if (!encode_2d(&tmA, Y, N, M, ElemBF16::kBK, a_rows) ||
        !encode_packed_weights(&tmB, W3packed, weight_tiles, 64u, false) ||
        !encode_2d(&tmOut, out, K, M, 64, 32))
        return SWIGLU_ERR_CUDA;
    FusedArgs args{};
    args.M = static_cast<int>(M);
    args.N = static_cast<int>(K);   // output columns
    args.K = static_cast<int>(N);   // reduction
    args.stage_tx_bytes = a_rows * kRowBytes + 64 * kRowBytes;
    args.a_tx_bytes = a_rows * kRowBytes;
    args.Y = static_cast<uint16_t *>(out);
    args.gate_scale = 1.0f;
    args.up_scale = 1.0f;
    args.slot_rows = slot_rows_for(M);
    args.sched = sched;
#ifdef SWIGLU_TEST_FAULT_INJECTION
    args.skip_first_fill = g_test_skip_first_fill;
#endif
    args.counters = ws ? static_cast<unsigned int *>(workspace) : nullptr;
    args.partials = ws ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                   counter_region_bytes(sm_count))
                       : nullptr;
    args.ticket_index = ticket_index(sm_count);
    args.tile_counter_index = tile_counter_index(sm_count);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(sched.grid));
    cfg.blockDim = dim3(Narrow32C::THREADS);
    cfg.dynamicSmemBytes = Narrow32C::SMEM_BYTES;
    const cudaError_t err =
        cudaLaunchKernelEx(&cfg, fused_up_kernel<kNarrow32Stages, 64, ElemBF16, false, true>, tmA,
                           tmB, tmB, tmB, tmOut, args);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    return SWIGLU_OK;
}

// out [M, K] = Y [M, N] x W3 [N, K] (W3 packed by swiglu_pack_down_weights),
// BF16 in and out, FP32 accumulation, on the kernel plan_down_any picks.
// weights_early: no launch still in flight on `stream` writes W3packed (the
// whole-MLP call, whose up-projection lets this launch start only after its
// own dependency wait), so the decode kernel may load W3 before waiting for
// the previous launch.
int down_forward_impl(const void *Y, const void *W3packed, void *out, int64_t M, int64_t N,
                      int64_t K, void *workspace, size_t workspace_bytes, void *stream,
                      bool weights_early = false) {
    const int c = down_checks(Y, W3packed, out, M, N, K);
    if (c != SWIGLU_OK) return c;
    const size_t obytes = static_cast<size_t>(M) * K * 2;
    const size_t ybytes = static_cast<size_t>(M) * N * 2;
    const size_t pbytes = swiglu_down_packed_weight_bytes(N, K);

    int dev;
    DeviceState *st;
    const int s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    const DownPlan plan =
        plan_down_any(M, N, K, st->pair_clusters, st->sm_count, st->decode_clusters);
    const WorkSched &sched = plan.sched;
    const size_t ws_need = down_workspace_bytes_for(plan, M, st->sm_count);
    if (ws_need > 0) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
            workspace_bytes < ws_need)
            return SWIGLU_ERR_INVALID_ARG;
        if (overlaps(workspace, ws_need, out, obytes) || overlaps(workspace, ws_need, Y, ybytes) ||
            overlaps(workspace, ws_need, W3packed, pbytes))
            return SWIGLU_ERR_INVALID_ARG;
    }
    if (plan.kind == kDownWide)
        return down_wide_launch(sched, Y, W3packed, out, M, N, K, workspace, ws_need > 0,
                                st->sm_count, stream);
    if (plan.kind == kDownDecode)
        return down_decode_launch(plan.splits, st->decode_clusters, Y, W3packed, out, M, N, K,
                                  stream, weights_early);
    if (plan.kind == kDownSlim)
        return down_slim_launch(sched, Y, W3packed, out, M, N, K, workspace, ws_need > 0,
                                st->sm_count, stream);
    const uint64_t weight_tiles =
        static_cast<uint64_t>(sched.order.n_tiles) * static_cast<uint64_t>(sched.k_blocks);
    // the sub-tile maps are never used in the plain mode: the whole-tile map
    // stands in for them
    CUtensorMap tmA, tmB, tmOut;
    if (!encode_2d(&tmA, Y, N, M, ElemBF16::kBK, FusedC::BM) ||
        !encode_packed_weights(&tmB, W3packed, weight_tiles, 128u, false) ||
        !encode_2d(&tmOut, out, K, M, 64, 32))
        return SWIGLU_ERR_CUDA;

    FusedArgs args{};
    args.M = static_cast<int>(M);
    args.N = static_cast<int>(K);   // output columns
    args.K = static_cast<int>(N);   // reduction
    args.stage_tx_bytes = FusedC::BM * kRowBytes + FusedC::B_BYTES;
    args.a_tx_bytes = FusedC::BM * kRowBytes;
    args.Y = static_cast<uint16_t *>(out);
    args.gate_scale = 1.0f;
    args.up_scale = 1.0f;
    args.slot_rows = slot_rows_for(M);
    args.sched = sched;
#ifdef SWIGLU_TEST_FAULT_INJECTION
    args.skip_first_fill = g_test_skip_first_fill;
#endif
    args.counters = ws_need ? static_cast<unsigned int *>(workspace) : nullptr;
    args.partials = ws_need ? reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                                        counter_region_bytes(st->sm_count))
                            : nullptr;
    args.ticket_index = ticket_index(st->sm_count);
    args.tile_counter_index = tile_counter_index(st->sm_count);
    args.dyn_tiles = dynamic_tiles(sched, true) ? 1 : 0;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * sched.grid));
    cfg.blockDim = dim3(PairC::THREADS);
    cfg.dynamicSmemBytes = PairC::SMEM_BYTES;
    const cudaError_t err =
        cudaLaunchKernelEx(&cfg, fused_up_pair_kernel<kPairStages, ElemBF16, true>, tmA, tmB,
                           tmB, tmB, tmOut, args);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    return SWIGLU_OK;
}

// Shared checks of the two down-weight packs; on success the launch grid.
int pack_down_checks(const void *W, int64_t N, int64_t K, void *W3packed, dim3 *grid) {
    if (!W || !W3packed) return SWIGLU_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || (N % 8) != 0 || (K % 8) != 0) return SWIGLU_ERR_INVALID_ARG;
    if (N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return SWIGLU_ERR_INVALID_ARG;
    if (!aligned16(W) || !aligned16(W3packed)) return SWIGLU_ERR_INVALID_ARG;
    if (overlaps(W3packed, swiglu_down_packed_weight_bytes(N, K), W, static_cast<size_t>(N) * K * 2))
        return SWIGLU_ERR_INVALID_ARG;
    const int64_t rows = round_up(K, kDownTileCols);
    if (rows / kPackTile > 65535) return SWIGLU_ERR_UNSUPPORTED;
    *grid = dim3(static_cast<unsigned>((N + kPackTile - 1) / kPackTile),
                 static_cast<unsigned>(rows / kPackTile));
    return SWIGLU_OK;
}

}  // namespace
}  // namespace swiglu

extern "C" {

size_t swiglu_down_packed_weight_bytes(int64_t N, int64_t K) {
    if (N <= 0 || K <= 0) return 0;
    return static_cast<size_t>(round_up(K, kDownTileCols)) * static_cast<size_t>(round_up(N, 64)) *
           2u;
}

int swiglu_pack_down_weights(const void *W3, int64_t N, int64_t K, void *W3packed, void *stream) {
    dim3 grid;
    int s = pack_down_checks(W3, N, K, W3packed, &grid);
    if (s != SWIGLU_OK) return s;
    int dev;
    DeviceState *st;
    s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    pack_down_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(W3), static_cast<uint16_t *>(W3packed), static_cast<int>(N),
        static_cast<int>(K), static_cast<int>(grid.x));
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}

int swiglu_pack_down_weights_nk(const void *W3t, int64_t K, int64_t N, void *W3packed,
                                void *stream) {
    dim3 grid;
    int s = pack_down_checks(W3t, N, K, W3packed, &grid);
    if (s != SWIGLU_OK) return s;
    int dev;
    DeviceState *st;
    s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    pack_down_nk_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(W3t), static_cast<uint16_t *>(W3packed), static_cast<int>(N),
        static_cast<int>(K), static_cast<int>(grid.x));
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}

size_t swiglu_down_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return down_workspace_bytes_impl(M, N, K);
}

int swiglu_down_forward(const void *Y, const void *W3packed, void *out, int64_t M, int64_t N,
                        int64_t K, void *workspace, size_t workspace_bytes, void *stream) {
    return down_forward_impl(Y, W3packed, out, M, N, K, workspace, workspace_bytes, stream);
}

size_t swiglu_mlp_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    return std::max(swiglu_workspace_bytes(M, N, K), down_workspace_bytes_impl(M, N, K));
}

int swiglu_mlp_forward(const void *A, const void *Wpacked, const void *W3packed, void *Y,
                       void *out, int64_t M, int64_t N, int64_t K, void *workspace,
                       size_t workspace_bytes, void *stream) {
    // everything the two launches need is checked before the first one
    if (!A || !Wpacked) return SWIGLU_ERR_INVALID_ARG;
    const int c = down_checks(Y, W3packed, out, M, N, K);
    if (c != SWIGLU_OK) return c;
    const size_t obytes = static_cast<size_t>(M) * K * 2;
    const size_t ybytes = static_cast<size_t>(M) * N * 2;
    const size_t p3bytes = swiglu_down_packed_weight_bytes(N, K);
    if (overlaps(out, obytes, A, obytes) ||
        overlaps(out, obytes, Wpacked, swiglu_packed_weight_bytes(N, K)) ||
        overlaps(Y, ybytes, W3packed, p3bytes))
        return SWIGLU_ERR_INVALID_ARG;
    const size_t need = swiglu_mlp_workspace_bytes(M, N, K);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return SWIGLU_ERR_INVALID_ARG;
        if (overlaps(workspace, need, out, obytes) || overlaps(workspace, need, W3packed, p3bytes))
            return SWIGLU_ERR_INVALID_ARG;
    }
    // The up-projection lets the down-projection start only after its own
    // dependency wait: every launch before this call has then completed,
    // and the up-projection writes Y and the workspace only, so the
    // down-projection may read W3packed before its own wait.
    int s = forward_impl<ElemBF16>(A, Wpacked, Y, M, N, K, 1.0f, 1.0f, workspace,
                                   workspace_bytes, stream, swiglu_packed_weight_bytes(N, K),
                                   true);
    if (s != SWIGLU_OK) return s;
    return down_forward_impl(Y, W3packed, out, M, N, K, workspace, workspace_bytes, stream,
                             true);
}

int swiglu_check_device_status(void *stream, uint32_t *raw_word) {
    int dev;
    DeviceState *st;
    const int s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaMemcpyFromSymbol(&word, g_status_word, sizeof word) != cudaSuccess ||
        cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    if (raw_word) *raw_word = word;
    return word ? SWIGLU_ERR_DEVICE_TIMEOUT : SWIGLU_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// swiglu_up_forward_noalloc: the same forward for callers that cannot
// allocate device memory (see include/swiglu.h). Its scratch is this
// file-scope device array: every GPU that loads the library holds
// SWIGLU_NOALLOC_SCRATCH_BYTES of it until the process exits. In host code
// the name below is only a host-side stand-in for the array; the device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_swiglu_noalloc_scratch[SWIGLU_NOALLOC_SCRATCH_BYTES];

namespace swiglu {
namespace {

struct NoAllocSetup {
    std::once_flag once;
    int status = SWIGLU_OK;
    void *scratch = nullptr;  // device address of g_swiglu_noalloc_scratch
};
NoAllocSetup g_noalloc[kMaxDevices];

}  // namespace
}  // namespace swiglu

extern "C" int swiglu_up_forward_noalloc(const void *A, const void *Wpacked, void *Y, int64_t M,
                                         int64_t N, int64_t K, void *stream) {
    if (!A || !Wpacked || !Y) return SWIGLU_ERR_INVALID_ARG;
    if (M < 1 || N < 8 || K < 8 || (N % 8) != 0 || (K % 8) != 0) return SWIGLU_ERR_INVALID_ARG;
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || K >= lim) return SWIGLU_ERR_INVALID_ARG;
    int dev;
    DeviceState *st;
    const int s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    // First call on this device (which is current): look up the array's
    // device address.
    NoAllocSetup &na = g_noalloc[dev];
    std::call_once(na.once, [&na] {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_swiglu_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            na.status = SWIGLU_ERR_CUDA;
            return;
        }
        na.scratch = p;
        na.status = SWIGLU_OK;
    });
    if (na.status != SWIGLU_OK) return na.status;
    const size_t need = swiglu_workspace_bytes(M, N, K);
    if (need > SWIGLU_NOALLOC_SCRATCH_BYTES) return SWIGLU_ERR_UNSUPPORTED;
    if (need > 0) {
        // The array keeps whatever the previous call left: zero the tile
        // counters (the only part that must start at zero) on this stream.
        if (cudaMemsetAsync(na.scratch, 0, counter_region_bytes(st->sm_count),
                            static_cast<cudaStream_t>(stream)) != cudaSuccess) {
            cudaGetLastError();
            return SWIGLU_ERR_CUDA;
        }
    }
    return swiglu_up_forward(A, Wpacked, Y, M, N, K, need ? na.scratch : nullptr,
                             need ? static_cast<size_t>(SWIGLU_NOALLOC_SCRATCH_BYTES) : 0, stream);
}

#ifdef SWIGLU_TEST_FAULT_INJECTION
namespace swiglu {
namespace {
// Test build only: other work that holds SMs for a fixed time. Each block
// (one warp, with enough shared memory that no other large-footprint block
// fits beside it on its SM) sleeps until `ns` nanoseconds of %globaltimer
// have passed; the iteration count is capped as well, so it always returns.
__global__ void test_busy_kernel(unsigned long long ns, unsigned long long max_iters) {
    extern __shared__ uint8_t hold[];
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (unsigned long long i = 0; i < max_iters; ++i) {
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 >= ns) break;
        __nanosleep(1000);
    }
    if (ns == 0 && threadIdx.x == 0) hold[0] = 0;
}
constexpr int kBusySmemBytes = 200 * 1024;
}  // namespace
}  // namespace swiglu

extern "C" int swiglu_test_busy_sms(int blocks, unsigned long long ns, void *stream) {
    if (blocks < 1 || blocks > 4096 || ns > 10000000000ULL) return SWIGLU_ERR_INVALID_ARG;
    if (cudaFuncSetAttribute(swiglu::test_busy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             swiglu::kBusySmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return SWIGLU_ERR_CUDA;
    }
    swiglu::test_busy_kernel<<<blocks, 32, swiglu::kBusySmemBytes,
                               static_cast<cudaStream_t>(stream)>>>(ns, ns / 10 + 1000000ULL);
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}
#endif
