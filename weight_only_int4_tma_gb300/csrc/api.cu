// C-ABI entry points (include/w4a16.h): argument validation, per-device state, kernel
// selection and the device status word.
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "w4a16.h"
#include "w4a8.h"
#include "mxfp.h"
#include "format.cuh"
#include "launch.h"

namespace w4g {

// One status word per device (each device holds its own copy of a __device__ variable).
__device__ int g_status_word = 0;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_ctx_mutex;
DeviceCtx g_ctx[kMaxDevices];
bool g_ctx_ready[kMaxDevices] = {};

// Returns the current device's context, creating it on first use.
int get_ctx(const DeviceCtx** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return W4A16_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ctx_mutex);
    if (!g_ctx_ready[dev]) {
        DeviceCtx c{};
        c.device = dev;
        if (cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&c.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return W4A16_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return W4A16_ERR_CUDA;
        c.status = static_cast<int*>(p);
        uint64_t ms = 2000;
        if (const char* e = std::getenv("W4A16_WAIT_TIMEOUT_MS")) {
            const long v = std::strtol(e, nullptr, 10);
            if (v > 0) ms = static_cast<uint64_t>(v);
        }
        c.timeout_ns = ms * 1000000ull;
        g_ctx[dev] = c;
        g_ctx_ready[dev] = true;
    }
    *out = &g_ctx[dev];
    return W4A16_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shape(int N, int K, int group, int dtype) {
    if (N <= 0 || K <= 0) return W4A16_ERR_INVALID_ARG;
    if (dtype != W4A16_FP16 && dtype != W4A16_BF16) return W4A16_ERR_UNSUPPORTED;
    if (group != 32 && group != 64 && group != 128) return W4A16_ERR_UNSUPPORTED;
    // N: zeros are packed 8 per word along N; K: whole groups (hence a multiple of 32).
    // Anything else is padded to whole 128 x 128 blocks by the repack.
    if (N % 8 != 0 || K % group != 0) return W4A16_ERR_UNSUPPORTED;
    if (tiles_n(N) > 65535) return W4A16_ERR_UNSUPPORTED;  // grid.y limit
    return W4A16_OK;
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Kernel / tiling choice for a GEMM.
// heavy_epilogue: an activation or a residual is fused into the store (more epilogue
// work per output element, done by the dequant warps).
int make_plan(const DeviceCtx& ctx, int M, int N, int K, int group,
              const w4a16_gemm_config* cfg, GemmPlan* plan, bool heavy_epilogue = false) {
    int kernel = cfg ? cfg->kernel : W4A16_KERNEL_AUTO;
    // Single-row decode of a small matrix (N*K up to 26 Mi weights, at most one 128-channel
    // tile per SM): the CUDA-core GEMV beats the tensor-core kernel there (no split-K
    // exchange, a shorter start); larger matrices favour the tensor-core kernel (measured
    // over N 2048..19200, K 2048..14336: e.g. 5.5 vs 6.0 us at 4096 x 4096, 10.8 vs 9.1 us
    // at 11008 x 4096).
    int flags = 0;
    if (cfg) {
        for (int i = 0; i < 3; ++i)
            if (cfg->reserved[i] != 0) return W4A16_ERR_INVALID_ARG;
        if (cfg->flags &
            ~(W4A16_GEMM_NO_PDL | W4A16_GEMM_NO_WEIGHT_PREFETCH | W4A16_GEMM_DEQUANT_LUT |
              W4A16_GEMM_DEQUANT_INT))
            return W4A16_ERR_INVALID_ARG;
        flags = cfg->flags;
    }
    if ((flags & W4A16_GEMM_DEQUANT_LUT) && (flags & W4A16_GEMM_DEQUANT_INT))
        return W4A16_ERR_INVALID_ARG;
    plan->dequant = (flags & W4A16_GEMM_DEQUANT_LUT) ? 1 : (flags & W4A16_GEMM_DEQUANT_INT) ? 2 : 0;
    if (kernel == W4A16_KERNEL_AUTO && M == 1 &&
        static_cast<long long>(N) * K <= (26LL << 20) && tiles_n(N) <= ctx.num_sms &&
        !plan->dequant && !(cfg && (cfg->tile_m || cfg->split_k || cfg->stages)))
        kernel = W4A16_KERNEL_SIMT;
    plan->pdl = (flags & W4A16_GEMM_NO_PDL) == 0;
    plan->prefetch_weights = plan->pdl && (flags & W4A16_GEMM_NO_WEIGHT_PREFETCH) == 0;
    if (kernel == W4A16_KERNEL_SIMT && plan->dequant) return W4A16_ERR_UNSUPPORTED;
    if (plan->dequant == 2 && group != 128) return W4A16_ERR_UNSUPPORTED;
    if (kernel == W4A16_KERNEL_SIMT) {
        if (M > 8) return W4A16_ERR_UNSUPPORTED;
        if (cfg && (cfg->split_k > 1 || cfg->stages != 0)) return W4A16_ERR_UNSUPPORTED;
        int rows = cfg && cfg->tile_m ? cfg->tile_m : 0;
        if (rows == 0) rows = 16;  // channels per unit (measured best or equal everywhere)
        if (rows != 16 && rows != 32) return W4A16_ERR_UNSUPPORTED;
        plan->kernel = W4A16_KERNEL_SIMT;
        plan->tile_m = rows;
        plan->split_k = 1;
        plan->stages = 0;
        return W4A16_OK;
    }
    if (kernel != W4A16_KERNEL_AUTO && kernel != W4A16_KERNEL_TC) return W4A16_ERR_INVALID_ARG;
    plan->kernel = W4A16_KERNEL_TC;

    const int n_tiles = tiles_n(N);
    const int kblocks = blocks_k(K);
    int bm = cfg && cfg->tile_m ? cfg->tile_m : 0;
    if (bm == 0) {
        if (M <= 16) bm = 16;
        else if (M <= 32) bm = 32;
        else if (M <= 64) bm = 64;
        else if (M >= 256 && n_tiles * ceil_div(M, 256) >= ctx.num_sms) bm = 256;
        else bm = 128;
    }
    if (bm != 16 && bm != 32 && bm != 64 && bm != 128 && bm != 256) return W4A16_ERR_UNSUPPORTED;
    if (plan->dequant == 1 && bm > 32) return W4A16_ERR_UNSUPPORTED;  // table: decode tiles
    if (plan->dequant == 2 && bm != 16) return W4A16_ERR_UNSUPPORTED;  // integer: 16 rows
    const int m_tiles = ceil_div(M, bm);
    if (m_tiles > 65535) return W4A16_ERR_UNSUPPORTED;
    const int base = n_tiles * m_tiles;
    // 64-row tiles alone on an SM (four whole-block groups, two MMA issuers) where one
    // CTA per SM, with the K slices that fit, still fills at least 4/5 of the SMs; an odd
    // A ring forced by the caller keeps the shared-block arrangement (two issuers take
    // alternate A stages).
    bool il64 = false;
    if (bm == 64 && plan->dequant == 0 && !(cfg && cfg->stages % 2 != 0)) {
        int s1 = cfg && cfg->split_k ? cfg->split_k : ctx.num_sms / base;
        if (s1 > 8) s1 = 8;
        if (s1 > kblocks) s1 = kblocks;
        il64 = s1 >= 1 && base * s1 <= ctx.num_sms && base * s1 * 5 >= ctx.num_sms * 4;
    }
    // CTAs per SM the rings are sized for: decode tiles always pair up, 64-row tiles
    // unless they run alone (above); 128-row tiles pair up (shallower rings) when there
    // are enough tiles to fill two per SM.
    const int occ = bm <= 32 ? 2 : bm == 64 ? (il64 ? 1 : 2)
                  : (bm == 128 && base >= 2 * ctx.num_sms ? 2 : 1);

    int split = cfg && cfg->split_k ? cfg->split_k : 0;
    if (split == 0) {
        const int slots = ctx.num_sms * occ;
        if (base >= slots) split = 1;
        // 16-row tiles, more tiles than SMs but fewer than slots: one wave would give
        // some SMs two tiles and others one; two half-length waves balance the SMs
        // (measured: 37.7 vs 44.2 us at N = 28672, K = 8192; with 32-row tiles the
        // receive area costs a ring stage and the split loses).
        else if (bm == 16 && base > ctx.num_sms) split = 2;
        else {
            // Clusters are placed whole within a GPC, so not every slot takes a cluster
            // CTA: above ~6/7 of the slots (260 CTAs on 152 SMs) the launch ran in two
            // waves (measured, 16-row tiles, K 4096 / 8192: 48 tiles x 6 = 288 CTAs 11.7
            // us, 48 x 5 = 240 CTAs 7.6 us, 48 x 4 7.3 us).
            split = slots / base;
            const int fit = slots * 6 / 7 / base;
            if (split > 2 && fit < split) split = fit < 2 ? 2 : fit;
        }
        if (split > 8) split = 8;
        if (split > kblocks) split = kblocks;
        if (split < 1) split = 1;
        // the split-K receive area must leave room for rings of at least two stages each
        const size_t lim = occ == 2 ? 113 * 1024 : static_cast<size_t>(ctx.max_smem_optin);
        while (split > 1 && tc_layout(bm, M, group, split, 2, 2).smem > lim) --split;
    }
    if (split < 1 || split > 8 || split > kblocks) return W4A16_ERR_UNSUPPORTED;

    // Decode tiles: each dequant warpgroup unpacks whole 128-K blocks.  128-row tiles
    // alone on an SM: four whole-block groups, each owning every fourth weight slot
    // (measured N = K = 8192: M = 256 34.4 against 36.7 us, M = 128 with split-K 2 25.5
    // against 28.1 us, with the groups sharing every block).  64-row tiles two to an SM:
    // both arrangements measured equal (M = 64: 18.2 us), the shared one is kept; alone
    // on an SM (il64, above): four whole-block groups and two issuers (M = 64, N = K =
    // 8192, split-K 2: 15.3-15.7 us against 16.4-18.0 two to an SM; M = 40, N = 2432:
    // 8.5 against 10.1 us).
    plan->whole_blocks = bm <= 32;
    plan->nwg = 2;
    // Shared-block tiles: four warpgroups (16 dequant warps) hide more latency where one
    // CTA holds an SM: 128-row tiles (transition M = 128, N = K = 8192: 28.7-30.9 against
    // 30.8-32.1 us), and 256-row tiles whose epilogue applies an activation or a residual
    // (prefill M = 4096 with bias + SiLU: 311.9 against 338.0 us); for the plain 256-row
    // store two groups stay faster (273.0 against 280.2 us).  Four groups at two CTAs per
    // SM would exceed the register file.
    if ((bm == 128 && occ == 1) || (bm == 256 && heavy_epilogue) || il64) plan->nwg = 4;
    if ((bm == 128 && occ == 1) || il64) plan->whole_blocks = true;
    const int mult = tc_stage_multiple(bm, plan->whole_blocks, plan->nwg);
    const int amult = tc_a_stage_multiple(bm, plan->whole_blocks);

    // Rings: A stages are freed when their MMAs complete, weight stages as soon as they
    // are unpacked (into TMEM), so the weight ring needs only a few slots per reading
    // group.  Decode tiles favour weight stages (the HBM stream; their A tiles are small
    // and stay in L2), larger tiles A stages (up to 4; they feed the MMAs).
    const size_t limit = occ == 2 ? 113 * 1024 : static_cast<size_t>(ctx.max_smem_optin);
    auto fits = [&](int a, int w) { return tc_layout(bm, M, group, split, a, w).smem <= limit; };
    const int sw_min = mult > 2 ? mult : 2;
    const int sw_max = 2 * mult > 4 ? 2 * mult : 4;
    const int sa_fixed = cfg && cfg->stages ? cfg->stages : 0;
    // 64-row tiles alone on an SM: an 8-stage A ring (M = 64, N = K = 8192: 15.3-15.7 us
    // against 15.9-16.4 with 4 stages)
    const int sa_max = sa_fixed ? sa_fixed : (il64 ? 8 : 4), sa_min = sa_fixed ? sa_fixed : 2;
    int sa = 0, sw = 0;
    if (bm <= 32) {
        for (int w = sw_max; w >= sw_min && !sa; w -= mult)
            for (int a = sa_max; a >= sa_min; --a)
                if (a % amult == 0 && fits(a, w)) { sa = a; sw = w; break; }
    } else {
        // at least 3 weight stages where they fit (64-row tiles with a 4-stage A ring and
        // 2 weight stages measured 0.6 us slower than 3 + 3), then any
        for (int pass = 0; pass < 2 && !sa; ++pass) {
            const int wmin = pass == 0 && sw_min < 3 ? 3 : sw_min;
            for (int a = sa_max; a >= sa_min && !sa; --a)
                for (int w = sw_max; w >= wmin; w -= mult)
                    if (a % amult == 0 && fits(a, w)) { sa = a; sw = w; break; }
        }
    }
    if (!sa) return W4A16_ERR_UNSUPPORTED;
    // With split-K a rank first writes its own partials of every slice to the start of
    // the rings (then pushes them to the owners), so the rings must hold recv bytes.
    auto rings_hold_partials = [&](int a, int w) {
        const TcLayout L = tc_layout(bm, M, group, split, a, w);
        return L.recv_off >= L.part_bytes;
    };
    while (split > 1 && !rings_hold_partials(sa, sw) && sw + mult <= kTcMaxStages &&
           fits(sa, sw + mult))
        sw += mult;
    if (sa < 2 || sa > kTcMaxStages || sa % amult != 0 || sw < sw_min || sw > kTcMaxStages ||
        sw % mult != 0 ||
        !fits(sa, sw) || !rings_hold_partials(sa, sw))
        return W4A16_ERR_UNSUPPORTED;
    plan->tile_m = bm;
    plan->split_k = split;
    plan->stages = sa;
    plan->w_stages = sw;
    return W4A16_OK;
}

}  // namespace
}  // namespace w4g

using namespace w4g;

extern "C" {

int w4a16_abi_version(void) { return W4A16_ABI_VERSION; }

const char* w4a16_status_string(int status) {
    switch (status) {
        case W4A16_OK: return "ok";
        case W4A16_ERR_INVALID_ARG: return "invalid argument";
        case W4A16_ERR_UNSUPPORTED: return "unsupported shape or option";
        case W4A16_ERR_CUDA: return "CUDA error";
        case W4A16_ERR_DEVICE_TIMEOUT: return "in-kernel wait timed out";
        case W4A16_ERR_FORMAT: return "packed weight header does not match the arguments";
        default: return "unknown status";
    }
}

size_t w4a16_packed_bytes(int N, int K, int group, int has_zeros, int has_channel_scale) {
    if (check_shape(N, K, group, W4A16_FP16) != W4A16_OK) return 0;
    const size_t blocks = static_cast<size_t>(tiles_n(N)) * static_cast<size_t>(blocks_k(K));
    return kHeaderBytes + blocks * block_bytes(group, has_zeros != 0) +
           (has_channel_scale ? 4ull * static_cast<size_t>(N) : 0ull);
}

int w4a16_repack(const uint32_t* qweight, const void* scales, const uint32_t* qzeros,
                 const void* channel_scale, int N, int K, int group, int dtype, void* packed,
                 size_t packed_bytes, void* stream) {
    if (!qweight || !scales || !packed) return W4A16_ERR_INVALID_ARG;
    int rc = check_shape(N, K, group, dtype);
    if (rc != W4A16_OK) return rc;
    if (!aligned(qweight, 16) || !aligned(scales, 2) || !aligned(packed, 16) ||
        (qzeros && !aligned(qzeros, 4)) || (channel_scale && !aligned(channel_scale, 2)))
        return W4A16_ERR_INVALID_ARG;
    if (packed_bytes < w4a16_packed_bytes(N, K, group, qzeros != nullptr, channel_scale != nullptr))
        return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    return launch_repack(*ctx, qweight, scales, qzeros, channel_scale, N, K, group, dtype,
                         packed, static_cast<cudaStream_t>(stream));
}

namespace {
int gemm_common(const void* A, const void* packed, int M, int N, int K, int group, int dtype,
                void* Y, const w4a16_gemm_config* cfg, const EpilogueArgs& epi, void* stream) {
    if (M < 0) return W4A16_ERR_INVALID_ARG;
    int rc = check_shape(N, K, group, dtype);
    if (rc != W4A16_OK) return rc;
    if (M == 0) return W4A16_OK;
    if (!A || !packed || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(Y, 16) || !aligned(packed, 16)) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    GemmPlan plan{};
    const bool heavy = epi.act != kActNone || epi.residual != nullptr;
    if ((rc = make_plan(*ctx, M, N, K, group, cfg, &plan, heavy)) != W4A16_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan.kernel == W4A16_KERNEL_SIMT)
        return launch_simt_gemm(*ctx, A, packed, M, N, K, group, dtype, Y, plan, epi, s);
    return launch_tc_gemm(*ctx, A, packed, M, N, K, group, dtype, Y, plan, epi, s);
}
}  // namespace

int w4a16_gemm_ex(const void* A, const void* packed, int M, int N, int K, int group, int dtype,
                  void* Y, const w4a16_gemm_config* cfg, void* stream) {
    const EpilogueArgs none{nullptr, nullptr, kActNone};
    return gemm_common(A, packed, M, N, K, group, dtype, Y, cfg, none, stream);
}

int w4a16_gemm_epilogue(const void* A, const void* packed, int M, int N, int K, int group,
                        int dtype, const void* bias, const void* residual, int act, void* Y,
                        const w4a16_gemm_config* cfg, void* stream) {
    if (act != W4A16_ACT_NONE && act != W4A16_ACT_RELU && act != W4A16_ACT_SILU)
        return W4A16_ERR_INVALID_ARG;
    if (!aligned(bias, 2) || !aligned(residual, 2)) return W4A16_ERR_INVALID_ARG;
    const EpilogueArgs epi{static_cast<const uint16_t*>(bias),
                           static_cast<const uint16_t*>(residual), act};
    return gemm_common(A, packed, M, N, K, group, dtype, Y, cfg, epi, stream);
}

int w4a16_gemm_plan(int M, int N, int K, int group, int dtype, const w4a16_gemm_config* cfg,
                    w4a16_gemm_config* out) {
    if (M < 1 || !out) return W4A16_ERR_INVALID_ARG;
    int rc = check_shape(N, K, group, dtype);
    if (rc != W4A16_OK) return rc;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    GemmPlan plan{};
    if ((rc = make_plan(*ctx, M, N, K, group, cfg, &plan)) != W4A16_OK) return rc;
    w4a16_gemm_config r{};
    r.kernel = plan.kernel;
    r.split_k = plan.split_k;
    r.tile_m = plan.tile_m;
    r.stages = plan.stages;
    if (plan.kernel == W4A16_KERNEL_TC) {
        r.reserved[0] = plan.w_stages;
        r.reserved[1] = plan.nwg;
        r.reserved[2] = plan.whole_blocks ? 1 : 0;
    }
    r.flags = (plan.pdl ? 0 : W4A16_GEMM_NO_PDL) |
              (plan.prefetch_weights ? 0 : W4A16_GEMM_NO_WEIGHT_PREFETCH) |
              (plan.dequant == 1 ? W4A16_GEMM_DEQUANT_LUT : 0) |
              (plan.dequant == 2 ? W4A16_GEMM_DEQUANT_INT : 0);
    *out = r;
    return W4A16_OK;
}

int w4a16_gemm(const void* A, const void* packed, int M, int N, int K, int group, int dtype,
               void* Y, void* stream) {
    return w4a16_gemm_ex(A, packed, M, N, K, group, dtype, Y, nullptr, stream);
}

int w4a16_dequant_debug(const void* packed, int N, int K, int group, int dtype, void* W_out,
                        void* stream) {
    if (!packed || !W_out) return W4A16_ERR_INVALID_ARG;
    int rc = check_shape(N, K, group, dtype);
    if (rc != W4A16_OK) return rc;
    if (!aligned(packed, 16) || !aligned(W_out, 16)) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    return launch_dequant_debug(*ctx, packed, N, K, group, dtype, W_out,
                                static_cast<cudaStream_t>(stream));
}

int w4a16_get_device_status(void* stream) {
    const DeviceCtx* ctx = nullptr;
    int rc = get_ctx(&ctx);
    if (rc != W4A16_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return W4A16_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyAsync(&v, ctx->status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(ctx->status, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return W4A16_ERR_CUDA;
    return v;
}

int w4a16_debug_splitk_timeout_probe(const void* A, const void* packed, int M, int N, int K,
                                     int group, int dtype, void* Y, unsigned int timeout_us,
                                     void* stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return W4A16_ERR_INVALID_ARG;
    if (M < 1 || M > 16) return W4A16_ERR_INVALID_ARG;
    int rc = check_shape(N, K, group, dtype);
    if (rc != W4A16_OK) return rc;
    if (!A || !packed || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(Y, 16) || !aligned(packed, 16)) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    w4a16_gemm_config cfg{};
    cfg.kernel = W4A16_KERNEL_TC;
    cfg.tile_m = 16;
    GemmPlan plan{};
    if ((rc = make_plan(*ctx, M, N, K, group, &cfg, &plan)) != W4A16_OK) return rc;
    if (plan.split_k < 2) return W4A16_ERR_UNSUPPORTED;
    return launch_tc_splitk_probe(*ctx, A, packed, M, N, K, group, dtype, Y, plan,
                                  static_cast<uint64_t>(timeout_us) * 1000ull,
                                  static_cast<cudaStream_t>(stream));
}

int w4a16_debug_timeout_probe(unsigned int timeout_us, void* stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    int rc = get_ctx(&ctx);
    if (rc != W4A16_OK) return rc;
    return launch_timeout_probe(*ctx, static_cast<uint64_t>(timeout_us) * 1000ull,
                                static_cast<cudaStream_t>(stream));
}

// ---- W4A8 (include/w4a8.h) ------------------------------------------------------------

namespace {
int w4a8_check_shape(int N, int K) {
    if (N < 1 || K < 1) return W4A16_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > 131072) return W4A16_ERR_UNSUPPORTED;
    if ((static_cast<long long>(N) + 31) / 32 * (K / 128) > 0x7FFFFFFFLL) return W4A16_ERR_UNSUPPORTED;
    return W4A16_OK;
}
}  // namespace

size_t w4a8_packed_bytes(int N, int K) {
    if (w4a8_check_shape(N, K) != W4A16_OK) return 0;
    return w4a8_blob_bytes(N, K);
}

int w4a8_repack(const uint32_t* qweight, const uint8_t* s_u8, const uint8_t* a,
                const float* s_w, int N, int K, void* packed, size_t packed_bytes,
                void* stream) {
    if (!qweight || !s_u8 || !a || !s_w || !packed) return W4A16_ERR_INVALID_ARG;
    int rc = w4a8_check_shape(N, K);
    if (rc != W4A16_OK) return rc;
    if (!aligned(qweight, 16) || !aligned(s_w, 4) || !aligned(packed, 16))
        return W4A16_ERR_INVALID_ARG;
    if (packed_bytes < w4a8_blob_bytes(N, K)) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    return launch_w4a8_repack(*ctx, qweight, s_u8, a, s_w, N, K, packed,
                              static_cast<cudaStream_t>(stream));
}

int w4a8_quantize_act(const void* A, int M, int K, int dtype, int8_t* A_i8, float* s_a,
                      void* stream) {
    if (M < 0 || K < 1) return W4A16_ERR_INVALID_ARG;
    if (dtype != W4A16_FP16 && dtype != W4A16_BF16) return W4A16_ERR_UNSUPPORTED;
    if (K % 128 != 0 || K > 131072) return W4A16_ERR_UNSUPPORTED;
    if (M == 0) return W4A16_OK;
    if (!A || !A_i8 || !s_a) return W4A16_ERR_INVALID_ARG;
    if (!aligned(A, 16) || !aligned(A_i8, 16) || !aligned(s_a, 4)) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    int rc = get_ctx(&ctx);
    if (rc != W4A16_OK) return rc;
    return launch_w4a8_quantize(*ctx, A, M, K, dtype, A_i8, s_a,
                                static_cast<cudaStream_t>(stream));
}

int w4a8_gemm(const int8_t* A_i8, const float* s_a, const void* packed, int M, int N, int K,
              int dtype, void* Y, void* stream) {
    if (M < 0) return W4A16_ERR_INVALID_ARG;
    int rc = w4a8_check_shape(N, K);
    if (rc != W4A16_OK) return rc;
    if (dtype != W4A16_FP16 && dtype != W4A16_BF16) return W4A16_ERR_UNSUPPORTED;
    if (M > 16) return W4A16_ERR_UNSUPPORTED;
    if (M == 0) return W4A16_OK;
    if (!A_i8 || !s_a || !packed || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(A_i8, 16) || !aligned(s_a, 4) || !aligned(packed, 16) || !aligned(Y, 2))
        return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    return launch_w4a8_gemm(*ctx, A_i8, s_a, packed, M, N, K, dtype, Y,
                            static_cast<cudaStream_t>(stream));
}

int w4a8_dequant_debug(const void* packed, int N, int K, int8_t* W_out, void* stream) {
    if (!packed || !W_out) return W4A16_ERR_INVALID_ARG;
    int rc = w4a8_check_shape(N, K);
    if (rc != W4A16_OK) return rc;
    if (!aligned(packed, 16) || !aligned(W_out, 16)) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    if ((rc = get_ctx(&ctx)) != W4A16_OK) return rc;
    return launch_w4a8_dequant_debug(*ctx, packed, N, K, W_out,
                                     static_cast<cudaStream_t>(stream));
}

// ---- MX block-scaled decode GEMM (include/mxfp.h) ---------------------------------------

size_t mx_packed_bytes(int N, int K) {
    if (N < 1 || K < 128 || K % 128 != 0) return 0;
    return mx_blob_bytes(N, K);
}

int mx_repack(const uint8_t* w_codes, const uint8_t* w_scales, int N, int K, void* packed,
              size_t packed_bytes, void* stream) {
    if (!w_codes || !w_scales || !packed) return W4A16_ERR_INVALID_ARG;
    if (N < 1 || K < 1) return W4A16_ERR_INVALID_ARG;
    if (K % 128 != 0) return W4A16_ERR_UNSUPPORTED;
    if (!aligned(packed, 16) || packed_bytes < mx_blob_bytes(N, K)) return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    int rc = get_ctx(&ctx);
    if (rc != W4A16_OK) return rc;
    return launch_mx_repack(*ctx, w_codes, w_scales, N, K, packed,
                            static_cast<cudaStream_t>(stream));
}

int mx_gemm(const uint8_t* a_codes, const uint8_t* a_scales, const void* packed, int M, int N,
            int K, int dtype, void* Y, void* stream) {
    if (M < 0 || N < 1 || K < 1) return W4A16_ERR_INVALID_ARG;
    if (K % 128 != 0) return W4A16_ERR_UNSUPPORTED;
    if (dtype != W4A16_FP16 && dtype != W4A16_BF16) return W4A16_ERR_UNSUPPORTED;
    if (M > 16) return W4A16_ERR_UNSUPPORTED;
    if (M == 0) return W4A16_OK;
    if (!a_codes || !a_scales || !packed || !Y) return W4A16_ERR_INVALID_ARG;
    if (!aligned(a_codes, 16) || !aligned(a_scales, 4) || !aligned(packed, 16) || !aligned(Y, 2))
        return W4A16_ERR_INVALID_ARG;
    const DeviceCtx* ctx = nullptr;
    int rc = get_ctx(&ctx);
    if (rc != W4A16_OK) return rc;
    return launch_mx_gemm(*ctx, a_codes, a_scales, packed, M, N, K, dtype, Y,
                          static_cast<cudaStream_t>(stream));
}

}  // extern "C"
