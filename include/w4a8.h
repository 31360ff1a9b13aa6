/*
 * w4a8.h -- C ABI of the W4A8 (LiquidQuant) path of the library (NVIDIA GB300, sm_103a).
 *
 *   Y[m, n] = RNE_dtype( fp32( sum_k A_i8[m, k] * Q_i8[n, k] ) * s_a[m] * s_w[n] )
 *   Q_i8[n, k] = ((Q_u4[n, k] * s_u8[n, g] + a[n, g]) mod 256) XOR 0x80,  g = k / 128
 *
 * Source: "W4A8量化计算优化：提升LLM推理效率的关键技术"
 *   §2.1 -- two-level weights: int8 per channel (scale s_w), then 4-bit codes per group
 *           with an integer step s_u8 <= 16 and an offset a = 128 + min, so that
 *           dequantisation is one IMAD and one XOR per four weights (the congruence above);
 *   §3.1-3.2 -- dequantise in registers and feed the int8 multiply directly;
 *   §4.2 -- groups of 128 along K.
 * Activations are quantised per row to int8 (w4a8_quantize_act).  Products are summed
 * exactly in int32 and scaled in fp32 (two multiplies, in the order above), then
 * rounded once to the output dtype.
 *
 * On sm_103a the tcgen05 family has no int8 MMA (kind::i8 is rejected for this target)
 * and the int8 mma.sync runs at the rate of dp4a on the CUDA cores, so the int8 products
 * are computed exactly through the f16 mma.sync (int8 values are exact in fp16, and each
 * 128-K block's sum stays below 2^24) or by dp4a; see w4a8_gemm.
 *
 * Conventions are those of w4a16.h: device pointers on the current device, caller-owned
 * buffers, `stream` a cudaStream_t passed as void*, asynchronous calls, w4a16_status
 * return codes, and kernel-detected errors recorded in the device status word read by
 * w4a16_get_device_status().
 */
#ifndef W4A8_H_
#define W4A8_H_

#include <stddef.h>
#include <stdint.h>

#include "w4a16.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Size in bytes of the packed W4A8 blob for an N x K weight matrix, or 0 if the shape is
 * unsupported (N < 1, K < 128, K % 128 != 0, K > 131072).  Host-only.  Source: the
 * two-level format of "W4A8量化计算优化" §2.1 (4-bit codes, one step and one offset byte
 * per group, one fp32 channel scale), repacked into the kernel's order.  With Np = N
 * rounded up to a multiple of 16 the blob is
 *     128-byte header
 *   + (Np/16)*(K/128) blocks of 1056 bytes (1024 bytes of codes for 16 channels x 128 K
 *     in the MMA fragment order, then the channels' steps and offsets)
 *   + 4*Np bytes of fp32 channel scales.
 * The layout is private to this library and versioned by the header.
 */
size_t w4a8_packed_bytes(int N, int K);

/*
 * Offline repack of canonical W4A8 weights ("W4A8量化计算优化" §2.1) into the blob.
 *   qweight  device, uint32 [N][K/8], 16-byte aligned: nibble j of word w in row n is the
 *            code Q_u4[n, 8w + j] (0..15), the nibble order of w4a16_repack.
 *   s_u8     device, uint8 [N][K/128]: the group's integer step, 1..16.
 *   a        device, uint8 [N][K/128]: the group's offset (128 + the group's int8 minimum).
 *   s_w      device, float [N]: the per-channel scale of the first (int8) level.
 *   N, K     N >= 1; K a multiple of 128, at most 131072 (so that |sum| < 2^31).
 *   packed   device output, >= w4a8_packed_bytes(N, K) bytes (packed_bytes), 16-byte
 *            aligned, not overlapping the inputs.
 * Precondition of the format: every code satisfies Q_u4 * s_u8 + a <= 255 (the value of
 * a code stays in the int8 range, as the page's quantiser guarantees), so that the
 * kernel's one IMAD per four codes never carries between bytes.  Steps outside 1..16 or
 * codes that break the precondition are recorded as W4A16_ERR_INVALID_ARG in the device
 * status word (the blob is written anyway and its results are then undefined).
 * Errors returned directly: INVALID_ARG (null/misaligned pointer, capacity too small),
 * UNSUPPORTED (shape), CUDA (launch failure).
 */
int w4a8_repack(const uint32_t* qweight, const uint8_t* s_u8, const uint8_t* a,
                const float* s_w, int N, int K, void* packed, size_t packed_bytes,
                void* stream);

/*
 * Per-row int8 activations (the activation side of "W4A8量化计算优化" §2: 8-bit
 * activations, one scale per token).  For each row m of A:
 *     s_a[m] = max_k |A[m, k]| / 127   (fp32, rounded to nearest even; 1 for a zero row)
 *     A_i8[m, k] = clamp(rint(A[m, k] / s_a[m]), -127, 127)   (fp32 division, ties to even)
 *   A      device, dtype [M][K] row-major (fp16 or bf16), 16-byte aligned.
 *   M      rows, M == 0 is a no-op; K a multiple of 128.
 *   dtype  w4a16_dtype of A.
 *   A_i8   device output, int8 [M][K] row-major, 16-byte aligned (caller-owned).
 *   s_a    device output, float [M], 4-byte aligned (caller-owned).
 * Launched with programmatic dependent launch: it reads A only after the previous kernel
 * in the stream has finished.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int w4a8_quantize_act(const void* A, int M, int K, int dtype, int8_t* A_i8, float* s_a,
                      void* stream);

/*
 * The W4A8 GEMM: Y = the formula at the top of this header, with the int8 weights
 * dequantised in registers from `packed` by one IMAD per four codes and never written
 * back ("W4A8量化计算优化" §3.1-3.2).  For 3..16 rows the int8 products go through the f16
 * tensor-core mma.sync (int8 values carried exactly as fp16, each 128-K block summed
 * exactly in fp32, the blocks added in int32); for 1 or 2 rows through dp4a on the CUDA
 * cores.  The sum is exact either way.  This is a decode path: 1 <= M <= 16 (larger M
 * returns UNSUPPORTED).
 *   A_i8, s_a  device, as written by w4a8_quantize_act (A_i8 16-byte aligned).
 *   packed     device, blob written by w4a8_repack with the same N and K.
 *   M, N, K    M == 0 is a no-op; N, K as for w4a8_repack.
 *   dtype      w4a16_dtype of Y.
 *   Y          device output, dtype [M][N] row-major, 2-byte aligned.
 * Launched with programmatic dependent launch: the blob header and the first weight
 * blocks are read while the previous kernel in the stream may still run (so that kernel
 * must not write the blob; w4a8_repack ends with a launch that later kernels cannot
 * overlap), A_i8 and s_a only after it has finished.  On a header mismatch nothing is
 * written and W4A16_ERR_FORMAT is recorded in the device status word.
 * Errors returned directly: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int w4a8_gemm(const int8_t* A_i8, const float* s_a, const void* packed, int M, int N, int K,
              int dtype, void* Y, void* stream);

/*
 * Debug / parity only: the int8 weights Q_i8[N][K] (row-major, device, 16-byte aligned,
 * caller-owned) the GEMM multiplies, expanded from the blob with the GEMM's own
 * IMAD arithmetic and the XOR (the congruence of "W4A8量化计算优化" §2.1).  Header checked as in
 * w4a8_gemm.  Errors: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int w4a8_dequant_debug(const void* packed, int N, int K, int8_t* W_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A8_H_ */
