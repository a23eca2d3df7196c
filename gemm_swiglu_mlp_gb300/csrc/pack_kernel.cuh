// Weight packing: W1, W2 [K, N] row-major BF16 -> Wpacked [2*Np, K] K-major.
//
// Packed row p belongs to block j = p / 256; r = p % 256; rows r < 128 are
// Gate columns n = 128j + r (W1[:, n] transposed), rows r >= 128 are Up
// columns n = 128j + r - 128 (W2[:, n] transposed); n >= N gives a zero row.
// This is the tensor-core-friendly form of the pages' fused weight matrix
// (technical summary, "Kernel-2": W1 and W2 merged into one K x 2N operand so
// one GEMM feeds Gate and Up from the same A tile). A permutation: bit-exact.
#pragma once

#include <cstdint>

namespace swiglu {

constexpr int kPackTile = 64;

// One CTA transposes a 64 (k) x 64 (n) tile through shared memory so that
// both the reads (along n) and the writes (along k) are coalesced.
__global__ void __launch_bounds__(256) pack_weights_kernel(const uint16_t *__restrict__ W1,
                                                            const uint16_t *__restrict__ W2,
                                                            uint16_t *__restrict__ Wp, int K,
                                                            int N) {
    __shared__ uint16_t tile[kPackTile][kPackTile + 2];
    const int k0 = blockIdx.x * kPackTile;
    const int p0 = blockIdx.y * kPackTile;   // first packed row of this CTA
    const int j = p0 / 256;
    const int r0 = p0 % 256;                 // 64-row chunks never straddle Gate/Up halves
    const bool up = r0 >= 128;
    const int n0 = 128 * j + (r0 & 127);
    const uint16_t *__restrict__ W = up ? W2 : W1;

    for (int i = threadIdx.x; i < kPackTile * kPackTile; i += blockDim.x) {
        const int kk = i / kPackTile, nn = i % kPackTile;
        const int k = k0 + kk, n = n0 + nn;
        tile[kk][nn] = (k < K && n < N) ? W[static_cast<int64_t>(k) * N + n] : uint16_t(0);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < kPackTile * kPackTile; i += blockDim.x) {
        const int nn = i / kPackTile, kk = i % kPackTile;
        const int k = k0 + kk;
        if (k < K) Wp[static_cast<int64_t>(p0 + nn) * K + k] = tile[kk][nn];
    }
}

}  // namespace swiglu
