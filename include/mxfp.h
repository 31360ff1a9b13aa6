/*
 * mxfp.h -- C ABI of the MX block-scaled decode GEMM of the library (NVIDIA GB300,
 * sm_103a): MXFP4 weights times MXFP8 activations.
 *
 *   Y[m, n] = RNE_dtype( sum_k a[m, k] * w[n, k] ),
 *   w[n, k] = e2m1(Wc[n, k]) * 2^(Ws[n, k/32] - 127),
 *   a[m, k] = e4m3(Ac[m, k]) * 2^(As[m, k/32] - 127)
 *
 * Source: "量化开销对比：各家方案的矩阵乘账本与省账手段", end of §3 and the MXFP4 / NVFP4
 * row of the §5 overhead table: 4-bit floating-point weights and 8-bit floating-point
 * activations, one E8M0 exponent scale per block of 32 values, which Blackwell's
 * tensor cores apply in hardware.  This path decodes the elements with the conversion
 * instructions (cvt.rn.f16x2.e2m1x2 / .e4m3x2) and multiplies them with the f16
 * mma.sync, one 32-value scale block per MMA step, applying the two block scales to each
 * block's fp32 partial sum; it is NOT the native block-scaled MMA, whose encodings are
 * not documented in this build's sources.  It serves the pages' comparison of 4-bit
 * decode bandwidth between the integer (W4A16) and the floating-point (MXFP4) formats.
 *
 * Conventions are those of w4a16.h: device pointers on the current device, caller-owned
 * buffers, `stream` a cudaStream_t passed as void*, asynchronous calls, w4a16_status
 * return codes, kernel-detected errors in the device status word read by
 * w4a16_get_device_status().
 */
#ifndef MXFP_H_
#define MXFP_H_

#include <stddef.h>
#include <stdint.h>

#include "w4a16.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Size in bytes of the packed MXFP4 weight blob, or 0 if the shape is unsupported (N < 1,
 * K < 128, K % 128 != 0).  Host-only.  With Np = N rounded up to a multiple of 16:
 * 128-byte header + (Np/16)*(K/128) blocks of 1088 bytes (1024 bytes of codes for 16
 * channels x 128 K in the MMA fragment order, then 64 scale bytes).  Private layout,
 * versioned by the header.
 */
size_t mx_packed_bytes(int N, int K);

/*
 * Offline repack of canonical MXFP4 weights into the blob.
 *   w_codes   device, uint8 [N][K/2]: byte k/2 of row n holds the E2M1 code of K value k
 *             (even k in the low nibble, odd k in the high nibble).
 *   w_scales  device, uint8 [N][K/32]: the E8M0 scale code of each block of 32 values.
 *   N, K      N >= 1, K a multiple of 128.
 *   packed    device output, >= mx_packed_bytes(N, K) bytes (packed_bytes), 16-byte
 *             aligned.
 * Errors: INVALID_ARG (null/misaligned pointer, capacity), UNSUPPORTED (shape), CUDA.
 */
int mx_repack(const uint8_t* w_codes, const uint8_t* w_scales, int N, int K, void* packed,
              size_t packed_bytes, void* stream);

/*
 * The MXFP4 x MXFP8 decode GEMM, Y = the formula at the top of this header, fp32
 * accumulation, Y rounded to nearest-even into dtype.
 *   a_codes   device, uint8 [M][K] E4M3 codes, 16-byte aligned.
 *   a_scales  device, uint8 [M][K/32] E8M0 scale codes, 4-byte aligned.
 *   packed    device, blob written by mx_repack with the same N and K.
 *   M         1..16 (0 is a no-op; more returns UNSUPPORTED).
 *   dtype     w4a16_dtype of Y (fp16 or bf16).
 *   Y         device output, dtype [M][N] row-major, 2-byte aligned.
 * On a header mismatch nothing is written and W4A16_ERR_FORMAT is recorded in the device
 * status word.  Errors returned directly: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int mx_gemm(const uint8_t* a_codes, const uint8_t* a_scales, const void* packed, int M, int N,
            int K, int dtype, void* Y, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXFP_H_ */
