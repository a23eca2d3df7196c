// Weight packing: W1, W2 [K, N] row-major -> Wpacked, tile-contiguous.
//
// BF16: Wpacked is [NB][KB][256][64] with NB = ceil(N/128), KB = ceil(K/64)
// (FP8: [NB][KB][256][128], KB = ceil(K/128); the same 128-byte rows):
// element (j, b, r, kk) is W1[64b + kk][128j + r] for r < 128 (Gate) and
// W2[64b + kk][128j + r - 128] for r >= 128 (Up); zero where the column is
// >= N or the k index is >= K. One (j, b) tile is one contiguous 32 KB block
// holding exactly what one k-block of one output tile needs (both Gate and
// Up rows, K-major), so each weight load is a single contiguous read.
// This is the tensor-core-friendly form of the pages' fused weight matrix
// (technical summary, "Kernel-2": W1 and W2 merged into one K x 2N operand so
// one GEMM feeds Gate and Up from the same A tile). A permutation plus zero
// padding: bit-exact.
#pragma once

#include <cstdint>

namespace swiglu {

constexpr int kPackTile = 64;

// One CTA transposes a KT (k) x 64 (n) tile through shared memory: reads are
// coalesced along n, and the 64 packed rows it writes (64 x 128 bytes) are
// one contiguous 8 KB run of the output. T = uint16_t with KT = 64 packs
// BF16 weights; T = uint8_t with KT = 128 packs FP8 weights into the same
// byte geometry (128-byte rows).
template <typename T, int KT>
__global__ void __launch_bounds__(256) pack_weights_kernel(const T *__restrict__ W1,
                                                            const T *__restrict__ W2,
                                                            T *__restrict__ Wp, int K, int N,
                                                            int KB) {
    __shared__ T tile[KT][kPackTile + 2];
    const int b = blockIdx.x;                // k-block
    const int k0 = b * KT;
    const int p0 = blockIdx.y * kPackTile;   // first packed row (over all 2*Np rows)
    const int j = p0 / 256;                  // output-column block
    const int r0 = p0 % 256;                 // 64-row chunks never straddle Gate/Up halves
    const bool up = r0 >= 128;
    const int n0 = 128 * j + (r0 & 127);
    const T *__restrict__ W = up ? W2 : W1;

    for (int i = threadIdx.x; i < KT * kPackTile; i += blockDim.x) {
        const int kk = i / kPackTile, nn = i % kPackTile;
        const int k = k0 + kk, n = n0 + nn;
        tile[kk][nn] = (k < K && n < N) ? W[static_cast<int64_t>(k) * N + n] : T(0);
    }
    __syncthreads();
    T *__restrict__ out = Wp + ((static_cast<int64_t>(j) * KB + b) * 256 + r0) * KT;
    for (int i = threadIdx.x; i < KT * kPackTile; i += blockDim.x) {
        const int nn = i / KT, kk = i % KT;
        out[nn * KT + kk] = tile[kk][nn];
    }
}

// Column-interleaved packing, the pages' Kernel-2 pairing (technical
// summary, "Kernel-2": the fused weight's even columns are Gate, odd columns
// Up, so matching Gate and Up results sit side by side): the same
// [NB][KB][256][64] tiles, with tile (j, b) row 2i = W1[64b..64b+63][128j + i]
// and row 2i + 1 = W2[64b..64b+63][128j + i] (i < 128); zero outside N and
// K. One 64-row chunk holds 32 output columns of both weights. A
// permutation plus zero padding: bit-exact.
__global__ void __launch_bounds__(256) pack_weights_il_kernel(const uint16_t *__restrict__ W1,
                                                               const uint16_t *__restrict__ W2,
                                                               uint16_t *__restrict__ Wp, int K,
                                                               int N, int KB) {
    __shared__ uint16_t tile[kPackTile][kPackTile + 2];
    const int b = blockIdx.x;                // k-block
    const int k0 = b * kPackTile;
    const int p0 = blockIdx.y * kPackTile;   // first packed row (over all 2*Np rows)
    const int j = p0 / 256;
    const int r0 = p0 % 256;
    const int n0 = 128 * j + r0 / 2;         // 32 output columns
    for (int i = threadIdx.x; i < kPackTile * kPackTile; i += blockDim.x) {
        const int kk = i / kPackTile, rr = i % kPackTile;
        const int k = k0 + kk, n = n0 + rr / 2;
        const uint16_t *__restrict__ W = (rr & 1) ? W2 : W1;
        tile[kk][rr] = (k < K && n < N) ? W[static_cast<int64_t>(k) * N + n] : uint16_t(0);
    }
    __syncthreads();
    uint16_t *__restrict__ out = Wp + ((static_cast<int64_t>(j) * KB + b) * 256 + r0) * kPackTile;
    for (int i = threadIdx.x; i < kPackTile * kPackTile; i += blockDim.x) {
        const int rr = i / kPackTile, kk = i % kPackTile;
        out[rr * kPackTile + kk] = tile[kk][rr];
    }
}

// Packing from nn.Linear-style weights: W1, W2 [N, K] row-major (each row is
// one output column's K weights). The packed tile wants exactly such rows
// (K-major), so this is a row gather: tile (j, b) row r < 128 is
// W1[128j + r][64b .. 64b+63], row r >= 128 the same of W2; zero outside N
// and K. Same output layout as pack_weights_kernel.
__global__ void __launch_bounds__(256) pack_weights_nk_kernel(const uint16_t *__restrict__ W1,
                                                               const uint16_t *__restrict__ W2,
                                                               uint16_t *__restrict__ Wp, int K,
                                                               int N, int KB) {
    const int b = blockIdx.x;                // k-block
    const int p0 = blockIdx.y * kPackTile;   // first packed row (over all 2*Np rows)
    const int j = p0 / 256;
    const int r0 = p0 % 256;
    const bool up = r0 >= 128;
    const int n0 = 128 * j + (r0 & 127);
    const uint16_t *__restrict__ W = up ? W2 : W1;
    uint16_t *__restrict__ out =
        Wp + ((static_cast<int64_t>(j) * KB + b) * 256 + r0) * kPackTile;
    // 64 rows x 64 k: each thread moves 16 bytes (8 elements) per step
    for (int i = threadIdx.x; i < kPackTile * kPackTile / 8; i += blockDim.x) {
        const int rr = i / (kPackTile / 8), c8 = (i % (kPackTile / 8)) * 8;
        const int n = n0 + rr, k = b * kPackTile + c8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (n < N && k < K)   // K % 8 == 0: an 8-element piece is wholly in or out
            v = *reinterpret_cast<const uint4 *>(W + static_cast<int64_t>(n) * K + k);
        *reinterpret_cast<uint4 *>(out + rr * kPackTile + c8) = v;
    }
}

// Down-projection weights, for the plain product out = Y x W3 that
// completes the gated MLP: W3 [N, K] row-major (N, the intermediate size, is
// the product's reduction; K, the hidden size, its output columns) ->
// W3packed [KT][NB][256][64], KT = ceil(K/256) tiles of 256 output columns,
// NB = ceil(N/64) k-blocks: element (j, b, r, nn) is W3[64b + nn][256j + r],
// zero where the column is >= K or the k index is >= N. The same
// tile-contiguous K-major form as the up-projection's packed weights, with
// 256 output columns per tile in place of 128 Gate + 128 Up rows; the packed
// row index 256j + r is the output column itself. A permutation plus zero
// padding: bit-exact.
__global__ void __launch_bounds__(256) pack_down_kernel(const uint16_t *__restrict__ W3,
                                                         uint16_t *__restrict__ Wp, int N, int K,
                                                         int NB) {
    __shared__ uint16_t tile[kPackTile][kPackTile + 2];
    const int b = blockIdx.x;                 // k-block (over N)
    const int n0 = b * kPackTile;
    const int p0 = blockIdx.y * kPackTile;    // first packed row = first output column
    const int j = p0 / 256;
    const int r0 = p0 % 256;
    for (int i = threadIdx.x; i < kPackTile * kPackTile; i += blockDim.x) {
        const int nn = i / kPackTile, cc = i % kPackTile;
        const int n = n0 + nn, col = p0 + cc;
        tile[nn][cc] = (n < N && col < K) ? W3[static_cast<int64_t>(n) * K + col] : uint16_t(0);
    }
    __syncthreads();
    uint16_t *__restrict__ out = Wp + ((static_cast<int64_t>(j) * NB + b) * 256 + r0) * kPackTile;
    for (int i = threadIdx.x; i < kPackTile * kPackTile; i += blockDim.x) {
        const int cc = i / kPackTile, nn = i % kPackTile;
        out[cc * kPackTile + nn] = tile[nn][cc];
    }
}

// The same from the nn.Linear layout of the down-projection weight, W3t
// [K, N] row-major (row c holds output column c's N weights, already
// K-major): a row gather, packed row 256j + r = W3t[256j + r][64b .. 64b+63].
__global__ void __launch_bounds__(256) pack_down_nk_kernel(const uint16_t *__restrict__ W3t,
                                                            uint16_t *__restrict__ Wp, int N,
                                                            int K, int NB) {
    const int b = blockIdx.x;
    const int p0 = blockIdx.y * kPackTile;
    const int j = p0 / 256;
    const int r0 = p0 % 256;
    uint16_t *__restrict__ out = Wp + ((static_cast<int64_t>(j) * NB + b) * 256 + r0) * kPackTile;
    for (int i = threadIdx.x; i < kPackTile * kPackTile / 8; i += blockDim.x) {
        const int rr = i / (kPackTile / 8), c8 = (i % (kPackTile / 8)) * 8;
        const int col = p0 + rr, n = b * kPackTile + c8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (col < K && n < N)   // N % 8 == 0: an 8-element piece is wholly in or out
            v = *reinterpret_cast<const uint4 *>(W3t + static_cast<int64_t>(col) * N + n);
        *reinterpret_cast<uint4 *>(out + rr * kPackTile + c8) = v;
    }
}

}  // namespace swiglu
