/*
 * swiglu.h - C ABI of the GB300 (sm_103a) fused SwiGLU up-projection library.
 *
 * The library computes the gated-MLP up-projection with its activation,
 *
 *     Y[m,n] = SiLU(Gate[m,n]) * Up[m,n],  Gate = A x W1,  Up = A x W2,
 *     SiLU(x) = x / (1 + e^-x),
 *
 * ("Tile-Level Activation Overlap for Efficient LLM Inference", Section 1
 * Introduction, the gated-MLP definition) in one kernel per call: Gate and
 * Up are accumulated in FP32 in tensor memory and never written to global
 * memory (same paper, Abstract: the activation is fused into the GEMM at tile
 * level). Inputs and output are BF16; accumulation is FP32; the FP32 result
 * SiLU(g)*u is rounded once to BF16 (round to nearest even).
 *
 * Conventions for every entry point
 *   - Pointers marked "device" are CUDA device pointers on the current device
 *     (cudaSetDevice / torch's current device). The caller allocates and owns
 *     every buffer; the library keeps no per-call allocation. It caches, per
 *     device and for the life of the process, a few host-side values (SM
 *     count, kernel attributes) and one 4-byte device status word.
 *   - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *     stream. Every call is asynchronous on `stream` and never synchronizes,
 *     except swiglu_check_device_status.
 *   - Return value: a swiglu_status. Arguments are validated on the host
 *     before anything is launched; a rejected call launches nothing. No C++
 *     exception crosses this boundary.
 *   - BF16 arrays are passed as raw 16-bit patterns (uint16_t storage).
 */
#ifndef SWIGLU_GB300_H
#define SWIGLU_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SWIGLU_OK = 0,
    SWIGLU_ERR_INVALID_ARG = 1,     /* null/misaligned pointer, bad size */
    SWIGLU_ERR_UNSUPPORTED = 2,     /* valid but not supported (no sm_103a device, sizes over limits) */
    SWIGLU_ERR_CUDA = 3,            /* a CUDA runtime/driver call or a launch failed */
    SWIGLU_ERR_DEVICE_TIMEOUT = 4   /* a kernel gave up on a bounded wait (see check_device_status) */
} swiglu_status;

/* Library ABI version, (major << 16) | minor. */
int swiglu_version(void);

/* Human-readable name of a swiglu_status value (static string, never NULL). */
const char *swiglu_status_string(int status);

/*
 * Size in bytes of the packed weight operand for an N x K pair (W1, W2).
 *
 * Packed layout (this library's own; the pages' Kernel-2 interleaves W1 and
 * W2 column by column into one K x 2N operand, technical summary
 * "Kernel-2", and this is the same idea in the tiled, K-major form the
 * tensor cores consume): BF16 [NB][KB][256][64], NB = ceil(N/128),
 * KB = ceil(K/64). Tile (j, b) is one contiguous 32 KB block: its rows
 * 0..127 are W1[64b..64b+63, 128j..128j+127] transposed (Gate), rows
 * 128..255 the same columns of W2 (Up), each row 64 consecutive k values.
 * Entries for columns n >= N or k >= K are zero. Size = 4 * NB*128 * KB*64.
 * Returns 0 if N <= 0 or K <= 0.
 */
size_t swiglu_packed_weight_bytes(int64_t N, int64_t K);

/*
 * Packs W1 and W2 (device, BF16, [K, N] row-major each) into Wpacked
 * (device, swiglu_packed_weight_bytes(N, K) bytes, layout above). A pure
 * permutation plus zero padding: bit-exact. One-time per weight set; runs as
 * one kernel on `stream`.
 * Requirements: K > 0, N > 0, N % 8 == 0, K % 8 == 0; all pointers non-null
 * and 16-byte aligned; Wpacked must not overlap W1 or W2.
 * Errors: SWIGLU_ERR_INVALID_ARG (arguments), SWIGLU_ERR_CUDA (launch).
 */
int swiglu_pack_weights(const void *W1, const void *W2, int64_t K, int64_t N,
                        void *Wpacked, void *stream);

/*
 * Same as swiglu_pack_weights, from weights stored the way PyTorch's
 * nn.Linear stores them: W1 and W2 (device, BF16) are [N, K] row-major (one
 * row of K weights per output column; Gate = A x W1^T). The packed layout
 * keeps such rows K-major, so this is a row gather without a transpose.
 * Same requirements, errors and output as swiglu_pack_weights; the packed
 * result is byte-identical to swiglu_pack_weights(W1^T, W2^T).
 */
int swiglu_pack_weights_nk(const void *W1, const void *W2, int64_t N, int64_t K,
                           void *Wpacked, void *stream);

/*
 * Bytes of device workspace that swiglu_up_forward needs for (M, N, K) on
 * the current device (the split of K over CTAs depends on its SM count).
 * 0 means none: pass workspace = NULL, workspace_bytes = 0. The workspace
 * holds FP32 Gate/Up partial tiles for tiles whose K range is split between
 * CTAs, plus one counter per such tile. K is split only for problems of a
 * handful of output tiles (whole tiles or column sub-tiles would leave most
 * SMs idle), or when SWIGLU_SCHEDULE forces it (see swiglu_up_forward).
 * Launches of whole tiles on CTA pairs with eight or more waves of tiles
 * need only the counter region (a few KB): their tiles past the first wave
 * are handed out at run time from a counter there, so that the pairs, which
 * drift apart over many tiles, keep working on neighbouring tiles and share
 * them in L2 (SWIGLU_DYNAMIC_TILES=0 turns this off, =1 uses it from two
 * waves on; the result is the same either way).
 */
size_t swiglu_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * Y = SiLU(A x W1) (.) (A x W2) in one fused kernel.
 *   A        device, BF16, [M, K] row-major (row stride K elements)
 *   Wpacked  device, output of swiglu_pack_weights for this (N, K)
 *   Y        device, BF16, [M, N] row-major; fully overwritten
 *   workspace, workspace_bytes: device scratch of at least
 *            swiglu_workspace_bytes(M, N, K) bytes, 256-byte aligned (may be
 *            NULL when that is 0). It must be zero-filled before its first
 *            use; every completed call leaves it ready for the next one
 *            (its tile counters back at zero), whatever the shape. After a
 *            SWIGLU_ERR_DEVICE_TIMEOUT, zero it again. Calls that run at the
 *            same time on the GPU (different streams) need separate
 *            workspaces.
 *            Why a workspace at all: the operation itself (the paper's
 *            problem statement) needs only A, the weights and Y. The
 *            workspace serves this library's K split for problems of a
 *            handful of output tiles, whose FP32 partial sums are combined
 *            through global memory before the activation (SiLU is not
 *            linear). Combining them inside a thread-block cluster through
 *            distributed shared memory instead needs no workspace, but was
 *            measured slower on GB300 (0.5B-shaped problem: 9.0 against
 *            8.2 us), so the interface keeps a caller-owned workspace, and
 *            swiglu_up_forward_noalloc below serves callers that cannot
 *            provide one.
 *            A split tile on CTA pairs is finished by one pair, which waits
 *            (bounded) for the others' partial sums. The pairs of such a
 *            launch are numbered by the order in which they start (a
 *            ticket counter in the workspace, back at its starting value
 *            after every launch), so a pair only ever waits for pairs that
 *            are already running: the call completes even while other
 *            kernels occupy part of the GPU.
 * Requirements: M >= 1, N >= 8, K >= 8, N % 8 == 0, K % 8 == 0 (16-byte row
 * strides), M, N, K < 2^31; A, Wpacked, Y 16-byte aligned; Y must not overlap
 * A, Wpacked or the workspace. M, N and K need not be multiples of any tile
 * size. The schedule (tile shape, CTA count) is chosen from M, N, K and the
 * device's SM count; the result is bit-identical from run to run. Two
 * environment variables, read on every call, force a choice for ablations:
 * SWIGLU_FUSED_VARIANT=1sm|2sm (1-SM kernel or CTA pairs) and
 * SWIGLU_SCHEDULE=dp|split|sk|sk-tail
 * (whole tiles, column sub-tiles in the last wave, split K over the last wave
 * and the remainder, or over the remainder only); swiglu_workspace_bytes
 * follows them too. SWIGLU_GROUP_M=<rows> sets how many token rows the
 * persistent tile order keeps together (default 2048) before it moves to
 * the next output columns.
 * The first call on a device does one-time set-up (kernel attributes); after
 * it, calls may be captured into CUDA graphs and replayed.
 * Errors: SWIGLU_ERR_INVALID_ARG, SWIGLU_ERR_UNSUPPORTED (the current device
 * is not an sm_103 part), SWIGLU_ERR_CUDA (tensor-map encode or launch
 * failure). Device-side timeouts are reported later by
 * swiglu_check_device_status.
 */
int swiglu_up_forward(const void *A, const void *Wpacked, void *Y,
                      int64_t M, int64_t N, int64_t K,
                      void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Column-interleaved packing: the pages' own Kernel-2 pairing (technical
 * summary, "Kernel-2": the fused weight matrix takes Gate in its even and Up
 * in its odd columns, so each Gate result sits next to its Up partner).
 * Kept beside the default 128-row-blocked layout to measure the two against
 * each other; the result is the same computation, bit for bit.
 * ---------------------------------------------------------------------- */

/*
 * Packs W1 and W2 (device, BF16, [K, N] row-major each) into Wpacked
 * (device, swiglu_packed_weight_bytes(N, K) bytes) column-interleaved:
 * BF16 [NB][KB][256][64] as for swiglu_pack_weights, but tile (j, b) row 2i
 * is W1[64b..64b+63, 128j+i] and row 2i+1 is W2[64b..64b+63, 128j+i]
 * (i < 128); zero outside N and K. Valid only for
 * swiglu_up_forward_interleaved. Requirements and errors as
 * swiglu_pack_weights.
 */
int swiglu_pack_weights_interleaved(const void *W1, const void *W2, int64_t K, int64_t N,
                                    void *Wpacked, void *stream);

/*
 * swiglu_up_forward on interleaved packed weights: the same kernels, tiles,
 * schedule and workspace (sized by swiglu_workspace_bytes); the epilogue
 * pairs accumulator columns 2i and 2i+1 instead of i and 128+i. Arguments,
 * requirements and errors as swiglu_up_forward; Wpacked must come from
 * swiglu_pack_weights_interleaved.
 */
int swiglu_up_forward_interleaved(const void *A, const void *Wpacked, void *Y,
                                  int64_t M, int64_t N, int64_t K,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * Scratch size of swiglu_up_forward_noalloc, fixed at build time: 32 MiB.
 */
#define SWIGLU_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/*
 * swiglu_up_forward for callers that cannot allocate device memory. (The
 * paper has no counterpart; this is a property of this library's interface.)
 * Some callers cannot provide the workspace that swiglu_up_forward may need:
 * a runtime that plans all of its device memory when it starts and must not
 * call cudaMalloc afterwards (cudaMalloc may synchronize the device and can
 * fail once memory is fully committed), or a plugin interface that passes a
 * kernel only its input and output buffers. This entry point takes the same
 * A, Wpacked, Y, M, N, K and stream, and allocates nothing: it calls no
 * cudaMalloc or cudaFree and no allocating library routine.
 *
 * Scratch: a device array inside the library of SWIGLU_NOALLOC_SCRATCH_BYTES
 * (32 MiB), held by every GPU that loads the library until the process exits.
 * Problems whose workspace (swiglu_workspace_bytes) is larger are rejected
 * with SWIGLU_ERR_UNSUPPORTED before anything is launched; use
 * swiglu_up_forward with a caller workspace for those. Problems that need no
 * workspace never touch the array.
 *
 * Set-up: the first call on a device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * Each call that uses the array first clears its tile counters with an
 * asynchronous memset on `stream`; the rest keeps the previous call's
 * contents and is overwritten before it is read.
 *
 * All calls on one device share the one array: calls that overlap on the GPU
 * (different streams running at the same time) race and may return wrong
 * results. Serialize them (one stream, or events between streams).
 * Results are bit-identical to swiglu_up_forward's for the same inputs.
 * Errors: as swiglu_up_forward, plus SWIGLU_ERR_UNSUPPORTED for problems over
 * the scratch size and SWIGLU_ERR_CUDA if the set-up or the memset fails.
 */
int swiglu_up_forward_noalloc(const void *A, const void *Wpacked, void *Y,
                              int64_t M, int64_t N, int64_t K, void *stream);

/* ------------------------------------------------------------------------
 * FP8 (E4M3) inputs with per-tensor scales. The paper names FP8 only as the
 * motivation for fusing (Section 1: as tensor-core arithmetic gets cheaper,
 * the activation's memory traffic matters more); these entry points are this
 * library's extension. The inputs stand for A = scale_a * A8,
 * W1 = scale_w1 * W1_8, W2 = scale_w2 * W2_8 (E4M3: 1 sign, 4 exponent bits
 * with bias 7, 3 significand bits, max 448). Gate and Up are accumulated from
 * the raw E4M3 products in FP32 in tensor memory (tcgen05.mma kind::f8f6f4),
 * multiplied by scale_a*scale_w1 and scale_a*scale_w2, then
 * Y = SiLU(Gate) * Up is rounded to BF16 as in swiglu_up_forward.
 * ---------------------------------------------------------------------- */

/* Packed FP8 weight bytes: [NB][KB][256][128] bytes, NB = ceil(N/128),
 * KB = ceil(K/128): the BF16 layout with 128 E4M3 values per 128-byte row.
 * Returns 0 if N <= 0 or K <= 0. */
size_t swiglu_packed_weight_bytes_fp8(int64_t N, int64_t K);

/* Packs W1_8 and W2_8 (device, E4M3 bytes, [K, N] row-major each) into
 * Wpacked8 (device, swiglu_packed_weight_bytes_fp8(N, K) bytes). A byte
 * permutation plus zero padding. Requirements: K > 0, N > 0, K % 16 == 0,
 * N % 8 == 0, pointers non-null and 16-byte aligned, no overlap. */
int swiglu_pack_weights_fp8(const void *W1_8, const void *W2_8, int64_t K, int64_t N,
                            void *Wpacked8, void *stream);

/* Workspace bytes of swiglu_up_forward_fp8 for (M, N, K) on the current
 * device (0: none needed). Same rules as swiglu_workspace_bytes. */
size_t swiglu_workspace_bytes_fp8(int64_t M, int64_t N, int64_t K);

/* Y = SiLU(A x W1) (.) (A x W2) from FP8 inputs.
 *   A8        device, E4M3, [M, K] row-major
 *   Wpacked8  device, output of swiglu_pack_weights_fp8 for this (N, K)
 *   Y         device, BF16, [M, N] row-major; fully overwritten
 *   scale_a, scale_w1, scale_w2: the per-tensor scales (finite, > 0)
 *   workspace: as swiglu_up_forward, sized by swiglu_workspace_bytes_fp8
 * Requirements: as swiglu_up_forward, with K % 16 == 0 (16-byte rows of A8).
 * Errors: as swiglu_up_forward; SWIGLU_ERR_INVALID_ARG also for a scale that
 * is not a positive number. */
int swiglu_up_forward_fp8(const void *A8, const void *Wpacked8, void *Y,
                          int64_t M, int64_t N, int64_t K,
                          float scale_a, float scale_w1, float scale_w2,
                          void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * The whole gated MLP: out = Y x W3 after the fused up-projection. The paper
 * defines Gate, Up and Y (Section 1 Introduction) and measures the
 * activation's share of the whole MLP's run time (Figure 1), but gives no
 * down-projection; out = Y x W3 with W3 [N, K] (N the intermediate size, K
 * the hidden size) is the usual completion of that MLP, and these entry
 * points are this library's extension. The down-projection is a plain
 * product: BF16 Y and W3, FP32 accumulation in tensor memory, each output
 * rounded once to BF16 (round to nearest even). Four kernels serve it, on
 * the same packed W3: for M <= 128 a decode kernel with the operands' roles
 * swapped (128 output columns of W3 on the tensor cores' 128-row side, all
 * token rows on the N side), each 128-column tile cut into j equal K ranges
 * on one cluster of j CTAs (j up to 16) whose partials are summed through
 * distributed shared memory (no workspace); a wide one (tiles of 256 rows x
 * 512 output columns, one accumulator stage; a third fewer operand bytes per
 * flop) when whole wide tiles fill at least 90% of their last wave and
 * M >= 256; otherwise the CTA-pair kernel in a plain mode (tiles of 256 rows
 * x 256 output columns; stream-K over N when whole tiles would leave the
 * last wave less than 90% full); and, forced only, the 1-SM kernel in a
 * plain mode (tiles of 128 rows x 64 output columns, stream-K).
 * SWIGLU_DOWN_TILE=64|128|256|512 forces one of them (128: the decode kernel,
 * only for M <= 128); SWIGLU_DECODE_SPLITS=<j> forces the decode kernel's K
 * ranges per tile, SWIGLU_SK_PAIRS=<g> the number of pairs of the CTA-pair
 * kernel's stream-K over all tiles (ablations). The wide kernel also
 * has split forms (forced by SWIGLU_SCHEDULE=sk|sk-tail|sk-aligned): a split
 * tile is finished, 128 columns at a time, by whichever participant counts
 * in last on them, so no CTA waits for another and the sums are added in k
 * order whoever finishes.
 * ---------------------------------------------------------------------- */

/* Packed down-projection weight bytes: [KT][NB][256][64] BF16 values,
 * KT = ceil(K/256) tiles of 256 output columns, NB = ceil(N/64) k-blocks.
 * Returns 0 if N <= 0 or K <= 0. */
size_t swiglu_down_packed_weight_bytes(int64_t N, int64_t K);

/* Packs W3 (device, BF16, [N, K] row-major: out = Y x W3) into W3packed
 * (device, swiglu_down_packed_weight_bytes(N, K) bytes, any prior content):
 * element (j, b, r, i) = W3[64b + i][256j + r], zero padded. A permutation:
 * bit-exact. Requirements: N > 0, K > 0, N % 8 == 0, K % 8 == 0, pointers
 * non-null and 16-byte aligned, no overlap. Asynchronous on `stream`. */
int swiglu_pack_down_weights(const void *W3, int64_t N, int64_t K, void *W3packed,
                             void *stream);

/* The same from the nn.Linear layout of the down-projection weight: W3t
 * (device, BF16, [K, N] row-major, W3t[c][n] = W3[n][c]). Note the argument
 * order (K, N), the order of W3t's dimensions. Same packed result. */
int swiglu_pack_down_weights_nk(const void *W3t, int64_t K, int64_t N, void *W3packed,
                                void *stream);

/* Workspace bytes of swiglu_down_forward for (M, N, K) on the current device
 * (0: none needed). Same rules and layout as swiglu_workspace_bytes. */
size_t swiglu_down_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * out = Y x W3, the down-projection alone.
 *   Y         device, BF16, [M, N] row-major (e.g. swiglu_up_forward's Y)
 *   W3packed  device, output of swiglu_pack_down_weights for this (N, K)
 *   out       device, BF16, [M, K] row-major; fully overwritten
 *   workspace: as swiglu_up_forward, sized by swiglu_down_workspace_bytes
 * Requirements: M >= 1, N >= 8, K >= 8, N % 8 == 0, K % 8 == 0, M, N, K <
 * 2^31; pointers 16-byte aligned; out must not overlap Y, W3packed or the
 * workspace. SWIGLU_SCHEDULE=dp|sk|sk-tail forces a work split as for
 * swiglu_up_forward (split is not offered here and means the automatic
 * choice; sk-aligned, every tile cut into equal K ranges on as many pairs,
 * applies to the wide kernel only; the decode kernel takes dp as one K
 * range per tile and its own SWIGLU_DECODE_SPLITS); SWIGLU_DOWN_TILE=
 * 64|128|256|512 forces the kernel (see above); SWIGLU_FUSED_VARIANT does not
 * apply. Errors as swiglu_up_forward; SWIGLU_ERR_UNSUPPORTED also for a
 * forced decode split whose clusters cannot be launched on this device.
 */
int swiglu_down_forward(const void *Y, const void *W3packed, void *out,
                        int64_t M, int64_t N, int64_t K,
                        void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes of swiglu_mlp_forward: the larger of the two products'. */
size_t swiglu_mlp_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * out = (SiLU(A x W1) (.) (A x W2)) x W3: swiglu_up_forward into Y, then
 * swiglu_down_forward from Y, two launches on `stream` (the second starts
 * while the first finishes and waits for its results before reading Y).
 * The first lets the second start only after every earlier work on
 * `stream` has completed, so the second (the decode kernel, up to 128 rows)
 * may already load W3packed while the first finishes; as with any stream
 * order, W3packed must not be written by work still running on another
 * stream.
 *   A, Wpacked  as swiglu_up_forward; W3packed as swiglu_down_forward
 *   Y           device, BF16, [M, N]: the intermediate, caller-owned,
 *               overwritten (it holds the up-projection's output afterwards)
 *   out         device, BF16, [M, K]; fully overwritten
 *   workspace   shared by both launches, at least swiglu_mlp_workspace_bytes
 * Every argument of both launches is checked before the first is made.
 * Requirements: those of both entry points; out must not overlap A or
 * Wpacked, and Y must not overlap W3packed.
 */
int swiglu_mlp_forward(const void *A, const void *Wpacked, const void *W3packed, void *Y,
                       void *out, int64_t M, int64_t N, int64_t K,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Synchronizes `stream`, then reads and clears the current device's status
 * word. Every wait inside the kernels is bounded (about a second); a kernel
 * that gives up sets a bit in the word, releases its tensor memory and
 * exits instead of hanging. Returns SWIGLU_OK, SWIGLU_ERR_DEVICE_TIMEOUT
 * (and writes the raw word to *raw_word if non-NULL), or SWIGLU_ERR_CUDA.
 * raw_word (optional, may be NULL) is a diagnostic output beyond the status:
 * which role's wait ran out (bit 0 producer, 1 MMA issuer, 2 epilogue,
 * 3 the drain after an abort).
 */
int swiglu_check_device_status(void *stream, uint32_t *raw_word);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_GB300_H */
