// Host side of the C ABI declared in include/swiglu.h: argument validation,
// per-device setup, TMA tensor-map encoding, schedule choice and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fused_up_kernel.cuh"
#include "pack_kernel.cuh"
#include "swiglu.h"

namespace swiglu {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kFusedStages = 4;
using FusedC = FusedCfg<kFusedStages>;

struct DeviceState {
    std::once_flag once;
    int status = SWIGLU_OK;  // result of the one-time setup
    int sm_count = 0;
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
        if (cudaFuncSetAttribute(fused_up_kernel<kFusedStages>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 FusedC::SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            st.status = SWIGLU_ERR_CUDA;
            return;
        }
        st.sm_count = sms;
        st.status = SWIGLU_OK;
    });
    *dev_out = dev;
    *st_out = &st;
    return st.status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// 2-D BF16 tensor map over a row-major [rows, cols] matrix with a
// 128-byte-swizzled box of box_rows x box_cols (box_cols * 2 <= 128 bytes).
bool encode_bf16_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                    uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace swiglu

using namespace swiglu;

extern "C" {

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
    return static_cast<size_t>(2 * round_up(N, 128)) * static_cast<size_t>(K) * 2u;
}

int swiglu_pack_weights(const void *W1, const void *W2, int64_t K, int64_t N, void *Wpacked,
                        void *stream) {
    if (!W1 || !W2 || !Wpacked) return SWIGLU_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || (K % 8) != 0 || (N % 8) != 0) return SWIGLU_ERR_INVALID_ARG;
    if (K >= (int64_t(1) << 31) || N >= (int64_t(1) << 31)) return SWIGLU_ERR_INVALID_ARG;
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(Wpacked)) return SWIGLU_ERR_INVALID_ARG;
    const size_t wbytes = static_cast<size_t>(K) * N * 2;
    const size_t pbytes = swiglu_packed_weight_bytes(N, K);
    if (overlaps(Wpacked, pbytes, W1, wbytes) || overlaps(Wpacked, pbytes, W2, wbytes))
        return SWIGLU_ERR_INVALID_ARG;
    const int64_t rows = 2 * round_up(N, 128);
    if (rows / kPackTile > 65535) return SWIGLU_ERR_UNSUPPORTED;
    int dev;
    DeviceState *st;
    const int s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;
    const dim3 grid(static_cast<unsigned>((K + kPackTile - 1) / kPackTile),
                    static_cast<unsigned>(rows / kPackTile));
    pack_weights_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(W1), static_cast<const uint16_t *>(W2),
        static_cast<uint16_t *>(Wpacked), static_cast<int>(K), static_cast<int>(N));
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
}

size_t swiglu_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    (void)M;
    (void)N;
    (void)K;
    return 0;
}

int swiglu_up_forward(const void *A, const void *Wpacked, void *Y, int64_t M, int64_t N,
                      int64_t K, void *workspace, size_t workspace_bytes, void *stream) {
    (void)workspace;
    if (!A || !Wpacked || !Y) return SWIGLU_ERR_INVALID_ARG;
    if (M < 1 || N < 8 || K < 8 || (N % 8) != 0 || (K % 8) != 0) return SWIGLU_ERR_INVALID_ARG;
    const int64_t lim = int64_t(1) << 31;
    if (M >= lim || N >= lim || K >= lim) return SWIGLU_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(Wpacked) || !aligned16(Y)) return SWIGLU_ERR_INVALID_ARG;
    if (workspace_bytes < swiglu_workspace_bytes(M, N, K)) return SWIGLU_ERR_INVALID_ARG;
    const size_t ybytes = static_cast<size_t>(M) * N * 2;
    if (overlaps(Y, ybytes, A, static_cast<size_t>(M) * K * 2) ||
        overlaps(Y, ybytes, Wpacked, swiglu_packed_weight_bytes(N, K)))
        return SWIGLU_ERR_INVALID_ARG;

    int dev;
    DeviceState *st;
    const int s = device_setup(&dev, &st);
    if (s != SWIGLU_OK) return s;

    const int64_t n_pad = round_up(N, 128);
    CUtensorMap tmA, tmB, tmY;
    if (!encode_bf16_2d(&tmA, A, K, M, FusedC::BK, FusedC::BM) ||
        !encode_bf16_2d(&tmB, Wpacked, K, 2 * n_pad, FusedC::BK, FusedC::UMMA_N) ||
        !encode_bf16_2d(&tmY, Y, N, M, 64, 32))
        return SWIGLU_ERR_CUDA;

    FusedArgs args;
    args.M = static_cast<int>(M);
    args.N = static_cast<int>(N);
    args.K = static_cast<int>(K);
    args.k_blocks = static_cast<int>((K + FusedC::BK - 1) / FusedC::BK);
    args.order.m_tiles = static_cast<int>((M + FusedC::BM - 1) / FusedC::BM);
    args.order.n_tiles = static_cast<int>(n_pad / FusedC::BN);
    args.order.group_m = std::min(16, args.order.m_tiles);
    const int64_t tiles = int64_t(args.order.m_tiles) * args.order.n_tiles;
    if (tiles >= lim) return SWIGLU_ERR_UNSUPPORTED;
    args.num_tiles = static_cast<int>(tiles);

    const int grid = static_cast<int>(std::min<int64_t>(tiles, st->sm_count));
    fused_up_kernel<kFusedStages><<<grid, FusedC::THREADS, FusedC::SMEM_BYTES,
                                     static_cast<cudaStream_t>(stream)>>>(tmA, tmB, tmY, args);
    if (cudaGetLastError() != cudaSuccess) return SWIGLU_ERR_CUDA;
    return SWIGLU_OK;
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
