/*
 * w4a16.h -- C ABI of the W4A16 fused dequant-GEMM library for NVIDIA GB300 (sm_103a).
 *
 *   Y[M, N] = A[M, K] . W^T,   W[n, k] = s[k/g, n] * (q[n, k] - z[k/g, n])
 *
 * A is fp16 or bf16; W is stored as 4-bit nibbles q (8 per uint32), with one scale s
 * (same dtype as A) and one 4-bit zero z per group of g = 32, 64 or 128 weights along K.
 * The weights are dequantised only inside the GEMM kernel and are never written back
 * to device memory.
 *
 * Sources (web pages, cited by title and section):
 *   "W4A16 GEMM 算子浅析：INT4 权重反量化的计算流水线"
 *       section "计算流水线的核心哲学"  -- HBM(4-bit) -> SMEM -> registers: unpack,
 *           W = (W_int4 - Zero) * Scale, half2 -> tensor-core MMA with fp32 accumulate;
 *       section "Marlin 与 CUTLASS 中的寄存器解包黑魔法" -- 8 nibbles per uint32 and the
 *           0x6400 exponent-injection (magic bias) unpack.
 *   "量化开销对比：各家方案的矩阵乘账本与省账手段"
 *       §6.1-6.2 -- one launch, one pass over the weights, no materialised FP16 weights;
 *           the group scale is applied to the weight operand inside the k loop, the
 *           per-channel scale in the epilogue;
 *       §6.4 -- offline repack of weights, scales and zeros into the kernel's tile order;
 *       §6.5 -- weights stream from HBM exactly once, double-buffered with TMA.
 *
 * Conventions for every entry point:
 *   - Every pointer named "device" is a CUDA device pointer on the CURRENT device
 *     (cudaGetDevice()).  The caller owns every buffer; the library keeps no reference
 *     after the call returns.
 *   - "stream" is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Work is enqueued asynchronously on it; the call does not synchronise unless it
 *     says so.
 *   - Return values are w4a16_status codes (0 = success, negative = error).  Argument
 *     errors are detected on the host before anything is launched.  Errors detected by
 *     a kernel (packed-header mismatch, a pipeline wait that ran out) are recorded in a
 *     per-device status word read by w4a16_get_device_status().
 *   - Calls are thread-safe: the only library state is per-device, created on first use
 *     under a lock.
 */
#ifndef W4A16_H_
#define W4A16_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W4A16_ABI_VERSION 1

typedef enum w4a16_status {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = -1,    /* null pointer, negative size, misaligned pointer  */
    W4A16_ERR_UNSUPPORTED = -2,    /* shape or group the kernels do not handle         */
    W4A16_ERR_CUDA = -3,           /* a CUDA runtime/driver call failed                */
    W4A16_ERR_DEVICE_TIMEOUT = -4, /* a bounded in-kernel wait expired (device status) */
    W4A16_ERR_FORMAT = -5          /* packed blob header does not match the arguments  */
} w4a16_status;

typedef enum w4a16_dtype {
    W4A16_FP16 = 0,
    W4A16_BF16 = 1
} w4a16_dtype;

/* Kernel selection for w4a16_gemm_ex (w4a16_gemm always uses W4A16_KERNEL_AUTO). */
typedef enum w4a16_kernel {
    W4A16_KERNEL_AUTO = 0,  /* M == 1, N*K <= 26*2^20, N/128 <= SMs: SIMT; else TC   */
    W4A16_KERNEL_TC = 1,    /* TMA ring -> dequant warps -> tcgen05.mma (swap-AB)      */
    W4A16_KERNEL_SIMT = 2   /* CUDA-core FMA GEMV (cp.async ring), M <= 8              */
} w4a16_kernel;

/* Flags for w4a16_gemm_config.flags. */
/* Launch without programmatic dependent launch (the kernel then starts only after the
 * previous work in the stream has finished). */
#define W4A16_GEMM_NO_PDL 1
/* Read the packed blob only after the previous kernel in the stream has finished.  By
 * default the tensor-core kernel reads the blob header and its first weight stages
 * while that kernel is still running (weights are static between repacks), and reads A
 * and writes Y only after it has finished.  Set this flag if the kernel that runs right
 * before the GEMM in the same stream writes the packed blob itself; w4a16_repack needs
 * no flag (it ends with a launch that later kernels cannot overlap). */
#define W4A16_GEMM_NO_WEIGHT_PREFETCH 2
/* Unpack the weights through a 16-entry table in shared memory (nibble -> its value in
 * the activation dtype; then the group's zero and scale, one rounding) instead of the
 * exponent-injection unpack: "量化开销对比" §6.3 (16-entry LUT, then the group scale).
 * Results are bit-identical to the default path; it is a measured alternative and is
 * slower on this GPU.  Tensor-core kernel with 16- or 32-row tiles only: any other plan
 * (the SIMT kernel, tile_m > 32, or M > 32 under the heuristic) returns
 * W4A16_ERR_UNSUPPORTED. */
#define W4A16_GEMM_DEQUANT_LUT 4
/* Integer-operand variant: the MMA takes the exact integers (q - z) and each 128-K block's
 * fp32 partial sum is multiplied by its group scale before it is accumulated ("fine-grained
 * scaling" per group; the pages' alternative to scaling the weight operand, "量化开销对比"
 * §6.2 explains why the scale cannot simply move to the end).  The weights are then NOT
 * rounded to the activation dtype, so the results differ from the default path (they are
 * the exact product to fp32 accumulation).  Tensor-core kernel with 16-row tiles (M <= 16)
 * and groups of 128 only; anything else returns W4A16_ERR_UNSUPPORTED.  Exclusive with
 * W4A16_GEMM_DEQUANT_LUT (both set: W4A16_ERR_INVALID_ARG). */
#define W4A16_GEMM_DEQUANT_INT 8

typedef struct w4a16_gemm_config {
    int kernel;       /* w4a16_kernel; AUTO picks SIMT only if the three fields below
                         are all 0                                                       */
    int split_k;      /* TC: 0 = heuristic; else 1..8 K-slices reduced inside a CTA
                         cluster.  SIMT: 0 or 1                                          */
    int tile_m;       /* TC: 0 = heuristic; else 16, 32, 64, 128 or 256 rows of A per
                         tile.  SIMT: 0, 16 or 32 output channels per work unit          */
    int stages;       /* TC: 0 = heuristic; else depth of the shared-memory ring of A
                         tiles (2..16); the weight ring beside it is sized by the library.
                         SIMT: must be 0 (fixed 4-stage cp.async ring)                   */
    int flags;        /* W4A16_GEMM_* bits; 0 = defaults                                 */
    int reserved[3];  /* must be zero (w4a16_gemm_plan's output, TC plans: reserved[0] =
                         the weight ring depth, reserved[1] = the dequant warpgroups,
                         reserved[2] = 1 if each warpgroup unpacks whole 128-K blocks,
                         0 if they share every block; all 0 for SIMT)                   */
} w4a16_gemm_config;

/* Library ABI version (W4A16_ABI_VERSION). */
int w4a16_abi_version(void);

/* Static, human-readable text for a status code (never NULL). */
const char* w4a16_status_string(int status);

/*
 * Size in bytes of the packed blob that w4a16_repack writes for these arguments, or 0
 * if the shape is unsupported (see w4a16_repack).  Source: "量化开销对比" §6.4 (weights,
 * scales and zeros repacked offline into the kernel's tile order) and "W4A16 GEMM 算子浅析"
 * §"Marlin 与 CUTLASS 中的寄存器解包黑魔法" (eight 4-bit weights per uint32, hence K*N/2
 * bytes of nibbles).  Host-only: touches no device memory.  With Np = N and Kp = K rounded up to
 * multiples of 128, the blob is
 *     128-byte header
 *   + Kp*Np/2 bytes of nibbles
 *   + (Kp/group)*Np*2 bytes of scales
 *   + (Kp/group)*Np/2 bytes of zeros         (only if has_zeros)
 *   + 4*N bytes of fp32 per-channel factors  (only if has_channel_scale)
 * laid out in the kernel's tile order (128 output channels x 128 K per block, blocks of
 * one channel tile contiguous along K; nibbles interleaved within each word so that
 * one LOP3 per pair of halves unpacks them; the block's scales and zeros follow its
 * nibbles so that they arrive with the weights).  The format is private to this
 * library and versioned by the header.
 */
size_t w4a16_packed_bytes(int N, int K, int group, int has_zeros, int has_channel_scale);

/*
 * Offline repack ("量化开销对比" §6.4 / §6.7): reorder canonical quantised weights into
 * the packed blob.  Runs once per weight matrix; asynchronous on `stream`.
 *
 *   qweight        device, uint32 [N][K/8], row-major.  Nibble j (bits 4j..4j+3) of word
 *                  w in row n is q[n, 8w + j], an unsigned value 0..15.
 *   scales         device, dtype [K/group][N], row-major: s[gi, n] for group gi.
 *   qzeros         device, uint32 [K/group][N/8], row-major.  Nibble j of word w in row
 *                  gi is z[gi, 8w + j].  NULL = symmetric weights, every zero is 8.
 *   channel_scale  device, dtype [N]: optional factor c[n] applied to the fp32 result
 *                  of output channel n in the epilogue.  NULL = none.
 *   N, K, group    N, K > 0; N % 8 == 0 (zeros are packed along N); group in
 *                  {32, 64, 128} and K % group == 0.  N and K need not be multiples of
 *                  128: the blob is padded to whole 128 x 128 blocks (zero scales past N
 *                  or K, so the padded weights are exactly 0) and records the logical
 *                  N and K.
 *   dtype          w4a16_dtype of scales and channel_scale (and of A/Y at GEMM time).
 *   packed         device output, at least w4a16_packed_bytes(...) bytes, 16-byte
 *                  aligned, must not overlap the inputs.
 *   packed_bytes   capacity of `packed` in bytes.
 * Errors: INVALID_ARG (null/misaligned pointer, capacity too small), UNSUPPORTED
 * (shape/group/dtype), CUDA (launch failure).
 */
int w4a16_repack(const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                 const void* channel_scale, int N, int K, int group, int dtype,
                 void* packed, size_t packed_bytes, void* stream);

/*
 * The fused W4A16 GEMM ("W4A16 GEMM 算子浅析" §"计算流水线的核心哲学"; "量化开销对比"
 * §6.2): Y = A . W^T with W dequantised on the fly from `packed`; fp32 accumulation;
 * the per-channel factor (if the blob has one) applied to the fp32 result; Y rounded to
 * nearest-even into dtype.
 *
 *   A       device, dtype [M][K] row-major, 16-byte aligned.
 *   packed  device, blob written by w4a16_repack with the same N, K, group, dtype.
 *   M       rows of A and Y; M == 0 is a no-op that returns W4A16_OK.
 *   N, K, group, dtype   as for w4a16_repack.
 *   Y       device output, dtype [M][N] row-major, 16-byte aligned, must not overlap A
 *           or packed.
 * The kernel checks the blob header against (N, K, group, dtype); on a mismatch it
 * writes nothing to Y and records W4A16_ERR_FORMAT in the device status word.
 * Errors returned directly: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int w4a16_gemm(const void* A, const void* packed, int M, int N, int K, int group, int dtype,
               void* Y, void* stream);

/* Same as w4a16_gemm with explicit kernel/tiling choices (cfg may be NULL = AUTO).
 * Returns UNSUPPORTED for a combination the chosen kernel cannot run.  w4a16_gemm is
 * w4a16_gemm_ex with cfg = NULL: programmatic dependent launch and weight prefetch on
 * (see W4A16_GEMM_NO_WEIGHT_PREFETCH for the one case that needs them off). */
int w4a16_gemm_ex(const void* A, const void* packed, int M, int N, int K, int group,
                  int dtype, void* Y, const w4a16_gemm_config* cfg, void* stream);

/* Activation of the fused epilogue (w4a16_gemm_epilogue). */
typedef enum w4a16_act {
    W4A16_ACT_NONE = 0,
    W4A16_ACT_RELU = 1,  /* max(x, 0)                                                 */
    W4A16_ACT_SILU = 2   /* x / (1 + exp(-x))                                         */
} w4a16_act;

/*
 * The fused GEMM with a bias / activation / residual epilogue ("量化开销对比" §6.2: the
 * accumulator times the per-channel scale, plus bias, then the store; §6.6: bias and
 * residual / activation fused into the same kernel).  Per output element, in fp32 after
 * the fp32 k-sum and the per-channel factor c[n]:
 *     Y[m,n] = RNE_dtype( act( c[n] * sum_k A[m,k] W[n,k] + bias[n] ) + residual[m,n] )
 *   bias      device, dtype [N], 2-byte aligned, or NULL (no bias).
 *   residual  device, dtype [M][N] row-major, 2-byte aligned, or NULL.  It may be Y
 *             itself (in-place residual add: each element is read and then written by the
 *             same thread); any other overlap with Y, A or packed is not allowed.
 *   act       w4a16_act.
 * Everything else (arguments, kernel choice through cfg, header check, errors) as for
 * w4a16_gemm_ex; INVALID_ARG also for an unknown act or a misaligned bias / residual.
 */
int w4a16_gemm_epilogue(const void* A, const void* packed, int M, int N, int K, int group,
                        int dtype, const void* bias, const void* residual, int act, void* Y,
                        const w4a16_gemm_config* cfg, void* stream);

/*
 * The kernel and tiling that w4a16_gemm_ex(..., cfg, ...) would launch for this shape on
 * the current device (cfg may be NULL = AUTO), written to *out with every field resolved
 * (kernel TC or SIMT; split_k, tile_m, stages as used; flags as applied; reserved[0..2]
 * = a TC plan's weight ring depth, dequant warpgroups and whole-block flag).  Host-side
 * only: launches nothing, reads no device memory.  Errors: INVALID_ARG (M < 1, out NULL,
 * bad cfg fields), UNSUPPORTED, CUDA (no usable device).
 */
int w4a16_gemm_plan(int M, int N, int K, int group, int dtype, const w4a16_gemm_config* cfg,
                    w4a16_gemm_config* out);

/*
 * Debug / parity only: expand the packed blob to dtype W_out[N][K] (row-major, device)
 * with exactly the unpack + dequant arithmetic the GEMM kernels use, i.e. step 2 of the
 * pipeline in "W4A16 GEMM 算子浅析" §"计算流水线的核心哲学", W = (W_int4 - Zero) * Scale,
 * rounded once to nearest-even into dtype.  This is the materialised-weight path that
 * "量化开销对比" §6.1 warns against; it is never used by w4a16_gemm.
 *   packed  device, blob written by w4a16_repack with the same N, K, group, dtype.
 *   W_out   device output, dtype [N][K], 16-byte aligned (caller-owned).
 * The header is checked as in w4a16_gemm (W4A16_ERR_FORMAT in the status word, W_out
 * untouched).  Errors returned directly: INVALID_ARG, UNSUPPORTED, CUDA.
 */
int w4a16_dequant_debug(const void* packed, int N, int K, int group, int dtype,
                        void* W_out, void* stream);

/*
 * Library infrastructure (no passage of the pages describes it): the error channel of
 * the kernels' bounded waits and header checks.
 * Synchronises `stream`, then reads and clears the current device's status word.
 * Returns W4A16_OK, or the first error a kernel recorded since the last call
 * (W4A16_ERR_FORMAT, W4A16_ERR_DEVICE_TIMEOUT), or W4A16_ERR_CUDA if the stream itself
 * reports an error.
 */
int w4a16_get_device_status(void* stream);

/*
 * Failure-path check: launches one CTA that waits on an mbarrier nothing ever arrives
 * on, with the same bounded wait the GEMM pipeline uses, limited to `timeout_us`
 * microseconds (1..1000000).  The kernel records W4A16_ERR_DEVICE_TIMEOUT and returns;
 * the GPU context stays usable.  Follow with w4a16_get_device_status().
 */
int w4a16_debug_timeout_probe(unsigned int timeout_us, void* stream);

/*
 * Failure-path check of the split-K exchange (library infrastructure, no passage of the
 * pages describes it): runs the tensor-core GEMM with 16-row tiles and the launch
 * choice's split-K on these arguments (as w4a16_gemm_ex with kernel TC, tile_m 16), except
 * that cluster rank 0 of every tile pushes none of its fp32 partials.  The other ranks'
 * waits for those partials are bounded by `timeout_us` microseconds (1..1000000; every
 * other wait of the launch too): they run out, the kernel records W4A16_ERR_DEVICE_TIMEOUT,
 * every rank still leaves only after its peers have stopped pushing into it, and the GPU
 * context stays usable.  Y (device, dtype [M][N], 16-byte aligned) is written only where
 * a rank received all partials; treat its contents as undefined.  A, packed, M (1..16), N,
 * K, group and dtype as for w4a16_gemm.  Returns UNSUPPORTED if the shape gives no split
 * (K too short or N large enough to fill the GPU without it).  Follow with
 * w4a16_get_device_status().
 */
int w4a16_debug_splitk_timeout_probe(const void* A, const void* packed, int M, int N, int K,
                                     int group, int dtype, void* Y, unsigned int timeout_us,
                                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H_ */
