// The fused W4A16 GEMM on the 5th-generation tensor cores (tcgen05), swap-AB form.
//
// One CTA computes a 128-channel x BM-row tile of Y^T = W . A^T over a K slice:
//
//   HBM --TMA bulk copy--> SMEM ring stage: [A tile BM x 128 (128B swizzle) | packed block]
//        (weights stream once, evict-first; "量化开销对比" §6.5; "W4A16 GEMM 算子浅析"
//         §"计算流水线的核心哲学", the HBM -> SMEM step)
//   SMEM --dequant warps: LOP3 magic-bias unpack, sub/mul per pair--> TMEM (A operand)
//        ("W4A16 GEMM 算子浅析" §"寄存器解包黑魔法"; the group scale is applied here, on the
//         weight operand, as "量化开销对比" §6.2 requires)
//   tcgen05.mma.kind::f16 D[128 x BM] (fp32, TMEM) += W_tile[128 x 16] (TMEM) . A[BM x 16]^T
//        (the FP16 x FP16 -> FP32 MMA of the pipeline diagram; weights are the 128-row M
//         operand so that a decode batch of 1..16 tokens only pads the narrow N side)
//   epilogue: tcgen05.ld -> (split-K: partials reduced over the CTA cluster through
//        distributed shared memory) -> x per-channel factor -> round to dtype -> Y
//        ("量化开销对比" §6.2 "最后：累加器 × s_x → +bias → 写出", §6.7 folding)
//
// Warp roles: warp 0 = TMA producer, warp 1 = TMEM allocator + single-thread MMA issuer,
// warps 2.. = dequant warps (4 per warpgroup; warp w may only touch TMEM lanes
// 32*(w%4)..+31, so each warpgroup covers all 128 lanes) which also run the epilogue.
// Every mbarrier wait is bounded; on expiry the CTA records a timeout, drains what it
// issued and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "dequant.cuh"
#include "format.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4g {

namespace {

constexpr int kMaxStages = 16;
constexpr int kCtrlBytes = 1024;

#ifdef W4A16_TRACE
// Development-only timeline (built with -DW4A16_TRACE, never in the product library):
// globaltimer stamps per CTA for the first kTraceCtas CTAs.
constexpr int kTraceCtas = 1024;
constexpr int kTraceSlots = 64;
__device__ unsigned long long g_w4a16_trace[kTraceCtas * kTraceSlots];
#define W4G_TRACE(slot, value)                                                         \
    do {                                                                              \
        const unsigned cta_ = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z); \
        const int slot_ = (slot);                                                     \
        if (cta_ < kTraceCtas && slot_ >= 0 && slot_ < kTraceSlots)                   \
            g_w4a16_trace[cta_ * kTraceSlots + slot_] = (value);                      \
    } while (0)
#define W4G_NOW() globaltimer_ns()
#else
#define W4G_TRACE(slot, value) do { } while (0)
#define W4G_NOW() 0ull
#endif

struct TcArgs {
    const uint8_t* packed;
    void* Y;
    int* status;
    int M, N, K, group;
    int kblocks;        // K / 128
    int splits;         // K slices = cluster size along x
    int stages;         // ring depth
    uint32_t stage_bytes;
    uint64_t timeout_ns;
};

template <int BM>
struct TcShape {
    static constexpr int kABoxBytes = BM * 128;            // BM rows x 64 K (128 bytes)
    static constexpr int kATileBytes = 2 * kABoxBytes;     // 128 K per stage
    static constexpr int kTBuf = BM >= 256 ? 2 : (BM >= 128 ? 2 : 3);  // TMEM W buffers
    static constexpr int kACol0 = BM < 64 ? 64 : BM;       // first W staging column
    static constexpr int kColsUsed = kACol0 + kTBuf * 64;
    static constexpr int kTmemCols = kColsUsed <= 32 ? 32 : kColsUsed <= 64 ? 64
                                   : kColsUsed <= 128 ? 128 : kColsUsed <= 256 ? 256 : 512;
};

template <int DT>
__device__ __forceinline__ uint16_t f32_to_dtype(float v) {
    if constexpr (DT == 0) return __half_as_ushort(__float2half_rn(v));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int BM, int NWG, int DT>
__global__ void __launch_bounds__(64 + 128 * NWG, 1)
w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const TcArgs args) {
    using S = TcShape<BM>;
    constexpr int kTBuf = S::kTBuf;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw);
    const uint32_t ring_bytes = static_cast<uint32_t>(args.stages) * args.stage_bytes;
    const uint32_t ctrl = base + ring_bytes;
    uint8_t* ctrl_ptr = base_ptr + ring_bytes;
    // control block: full[16] empty[16] tfull[4] tempty[4] accum, then scalars
    const uint32_t full0 = ctrl, empty0 = ctrl + 128, tfull0 = ctrl + 256, tempty0 = ctrl + 288;
    const uint32_t accum_bar = ctrl + 320;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl_ptr + 328);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ctrl_ptr + 332);
    int* info = reinterpret_cast<int*>(ctrl_ptr + 336);  // [0] flags or -1, [1] block bytes
    const float** cs_slot = reinterpret_cast<const float**>(ctrl_ptr + 352);

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int split = static_cast<int>(blockIdx.x);
    const int n_tile = static_cast<int>(blockIdx.y);
    const int m_tile = static_cast<int>(blockIdx.z);
    const int kb_per = args.kblocks / args.splits, kb_rem = args.kblocks % args.splits;
    const int kb0 = split * kb_per + (split < kb_rem ? split : kb_rem);
    const int nkb = kb_per + (split < kb_rem ? 1 : 0);

    if (threadIdx.x == 0) {
        W4G_TRACE(0, W4G_NOW());
        const PackedHeader* h = reinterpret_cast<const PackedHeader*>(args.packed);
        const int flags = check_header(h, args.N, args.K, args.group, DT);
        info[0] = flags;
        info[1] = flags < 0 ? 0 : static_cast<int>(h->block_bytes);
        *cs_slot = (flags >= 0 && (flags & kFlagChannelScale))
                       ? reinterpret_cast<const float*>(args.packed + h->cscale_offset)
                       : nullptr;
        if (flags < 0 && split == 0 && n_tile == 0 && m_tile == 0)
            record_status(args.status, kStatusFormat);
        *abort_flag = 0;
        for (int s = 0; s < args.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int t = 0; t < kTBuf; ++t) {
            mbar_init(tfull0 + 8 * t, 4 * NWG);
            mbar_init(tempty0 + 8 * t, 1);
        }
        mbar_init(accum_bar, 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) prefetch_tensormap(&tmap_a);
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), S::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = *tmem_slot;
#ifdef W4A16_TRACE
    if (threadIdx.x == 0) {
        W4G_TRACE(1, W4G_NOW());
        unsigned smid_;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid_));
        W4G_TRACE(56, smid_);
    }
#endif
    const int flags = info[0];
    const bool run = flags >= 0 && nkb > 0;
    const bool has_z = flags >= 0 && (flags & kFlagZeros) != 0;
    const uint32_t bb = static_cast<uint32_t>(info[1]);
    const float* cscale = *cs_slot;
    const uint64_t tlim = args.timeout_ns;

    if (run && warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            const uint8_t* src = args.packed + kHeaderBytes +
                                 (static_cast<size_t>(n_tile) * args.kblocks + kb0) * bb;
            const int m0 = m_tile * BM;
            int issued = 0;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % args.stages;
                const uint32_t ph = static_cast<uint32_t>(i / args.stages) & 1u;
                if (i >= args.stages &&
                    !mbar_wait_bounded(empty0 + 8 * s, ph ^ 1u, abort_flag, args.status, tlim))
                    break;
                const uint32_t st = base + static_cast<uint32_t>(s) * args.stage_bytes;
                const uint32_t fb = full0 + 8 * s;
                mbar_arrive_expect_tx(fb, bb + S::kATileBytes);
                tma_bulk_g2s(st + S::kATileBytes, src + static_cast<size_t>(i) * bb, bb, fb, pol_w);
                const int kc = (kb0 + i) * kTileK;
                tma_tensor_2d_g2s(st, &tmap_a, kc, m0, fb, pol_a);
                tma_tensor_2d_g2s(st + S::kABoxBytes, &tmap_a, kc + 64, m0, fb, pol_a);
                W4G_TRACE(2 + (i < 16 ? i : 15), W4G_NOW());
                ++issued;
            }
            if (issued < nkb || *abort_flag) {
                // Drain: every issued copy must land before the CTA may exit.
                const int first = issued > args.stages ? issued - args.stages : 0;
                for (int i = first; i < issued; ++i) {
                    const int s = i % args.stages;
                    const uint32_t ph = static_cast<uint32_t>(i / args.stages) & 1u;
                    int dummy = 0;
                    (void)mbar_wait_bounded(full0 + 8 * s, ph, &dummy, nullptr, tlim);
                }
            }
        }
    } else if (run && warp == 1) {
        // ---------------- MMA issuer (one thread) ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16(DT, 128, BM);
            bool ok = true;
            for (int i = 0; i < nkb && ok; ++i) {
                const int s = i % args.stages;
                const uint32_t ph = static_cast<uint32_t>(i / args.stages) & 1u;
                const int t = i % kTBuf;
                const uint32_t tph = static_cast<uint32_t>(i / kTBuf) & 1u;
                ok = mbar_wait_bounded(full0 + 8 * s, ph, abort_flag, args.status, tlim) &&
                     mbar_wait_bounded(tfull0 + 8 * t, tph, abort_flag, args.status, tlim);
                if (!ok) break;
                if (i < 6) W4G_TRACE(57 + i, W4G_NOW());
                tc_fence_after();
                const uint32_t st = base + static_cast<uint32_t>(s) * args.stage_bytes;
#pragma unroll
                for (int j = 0; j < kTileK / 16; ++j) {
                    const uint32_t a_t = tmem + S::kACol0 + t * 64 + j * 8;
                    const uint64_t bd = sw128_desc(st + (j >> 2) * S::kABoxBytes + (j & 3) * 32);
                    tc_mma_ts(tmem, a_t, bd, idesc, (i | j) != 0 ? 1u : 0u);
                }
                tc_commit(empty0 + 8 * s);
                tc_commit(tempty0 + 8 * t);
            }
            tc_commit(accum_bar);
            W4G_TRACE(50, W4G_NOW());
            if (!ok) {  // make sure no MMA is still reading TMEM/SMEM when the CTA exits
                int dummy = 0;
                (void)mbar_wait_bounded(accum_bar, 0, &dummy, nullptr, tlim);
            }
        }
    } else if (run) {
        // ---------------- dequant warps ----------------
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int wg = (warp - 2) >> 2;         // dequant warpgroup
        const int r = q * 32 + lane;            // weight row of the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t zoff = kNibbleBytes + scale_bytes(args.group);
        for (int i = 0; i < nkb; ++i) {
            const int s = i % args.stages;
            const uint32_t ph = static_cast<uint32_t>(i / args.stages) & 1u;
            const int t = i % kTBuf;
            const uint32_t tph = static_cast<uint32_t>(i / kTBuf) & 1u;
            if (!mbar_wait_warp(full0 + 8 * s, ph, abort_flag, args.status, tlim)) break;
            if (warp == 2 && lane == 0 && i < 16) W4G_TRACE(18 + i, W4G_NOW());
            if (i >= kTBuf &&
                !mbar_wait_warp(tempty0 + 8 * t, tph ^ 1u, abort_flag, args.status, tlim))
                break;
            const uint8_t* wb = base_ptr + static_cast<size_t>(s) * args.stage_bytes + S::kATileBytes;
#pragma unroll
            for (int c = wg; c < 4; c += NWG) {
                const int gi = (c * kChunkK) / args.group;
                const uint32_t sbits =
                    reinterpret_cast<const uint16_t*>(wb + kNibbleBytes)[gi * kTileN + r];
                uint32_t z = 8;
                if (has_z) z = (wb[zoff + gi * (kTileN / 2) + (r >> 1)] >> ((r & 1) * 4)) & 0xFu;
                const uint32_t zp = zero_pair<DT>(z), sp = scale_pair(sbits);
                const uint4 v = *reinterpret_cast<const uint4*>(wb + c * 2048 + r * 16);
                uint32_t out[16];
                dequant_word<DT>(v.x, zp, sp, out + 0);
                dequant_word<DT>(v.y, zp, sp, out + 4);
                dequant_word<DT>(v.z, zp, sp, out + 8);
                dequant_word<DT>(v.w, zp, sp, out + 12);
                tmem_st16(tmem + lane_base + S::kACol0 + t * 64 + c * 16, out);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tfull0 + 8 * t);
            if (warp == 2 && lane == 0 && i < 16) W4G_TRACE(34 + i, W4G_NOW());
        }

        // ---------------- epilogue ----------------
        if (mbar_wait_warp(accum_bar, 0, abort_flag, args.status, tlim)) {
            if (warp == 2 && lane == 0) W4G_TRACE(51, W4G_NOW());
            tc_fence_after();
            const int n = n_tile * kTileN + r;
            const float cs = cscale ? cscale[n] : 1.0f;
            uint16_t* Y = static_cast<uint16_t*>(args.Y);
            float* part = reinterpret_cast<float*>(base_ptr);  // [BM][128] when split
#pragma unroll 1
            for (int e = wg; e < BM / 16; e += NWG) {
                uint32_t v[16];
                tmem_ld16(tmem + lane_base + e * 16, v);
                tmem_wait_ld();
                if (args.splits == 1) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int m = m_tile * BM + e * 16 + j;
                        if (m < args.M)
                            Y[static_cast<size_t>(m) * args.N + n] =
                                f32_to_dtype<DT>(__uint_as_float(v[j]) * cs);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) part[(e * 16 + j) * kTileN + r] = __uint_as_float(v[j]);
                }
            }
        }
    }

    // ---------------- split-K reduction across the cluster ----------------
    __syncwarp();
    if (warp == 2 && lane == 0) W4G_TRACE(52, W4G_NOW());
    if (args.splits > 1) {
        cluster_sync_all();
        if (threadIdx.x == 0) W4G_TRACE(53, W4G_NOW());
        if (run && !*abort_flag) {
            const uint32_t rank = cluster_ctarank();
            const int S_ = args.splits;
            const int rows_per = (kTileN + S_ - 1) / S_;
            const int r0 = static_cast<int>(rank) * rows_per;
            const int r1 = min(kTileN, r0 + rows_per);
            const int nr = r1 - r0;
            const int mvalid = min(BM, args.M - m_tile * BM);
            uint16_t* Y = static_cast<uint16_t*>(args.Y);
            for (int e = static_cast<int>(threadIdx.x); nr > 0 && e < nr * mvalid;
                 e += static_cast<int>(blockDim.x)) {
                const int ml = e / nr;
                const int rl = r0 + e % nr;
                const uint32_t off = base + static_cast<uint32_t>((ml * kTileN + rl) * 4);
                float acc = 0.0f;
                for (int p = 0; p < S_; ++p) acc += ld_dsmem_f32(map_to_rank(off, p));
                const int n = n_tile * kTileN + rl;
                if (cscale) acc *= cscale[n];
                Y[static_cast<size_t>(m_tile * BM + ml) * args.N + n] = f32_to_dtype<DT>(acc);
            }
        }
        if (threadIdx.x == 0) W4G_TRACE(54, W4G_NOW());
        cluster_sync_all();
    }
    if (threadIdx.x == 0) W4G_TRACE(55, W4G_NOW());

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, S::kTmemCols);
    }
}

// ---- host side ---------------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

template <int BM, int NWG, int DT>
int launch_tc_instance(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                       int K, int group, void* Y, const GemmPlan& plan, cudaStream_t stream) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return -3;
    CUtensorMap map;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(BM)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult cr = enc(&map, DT == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      2, const_cast<void*>(A), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return -3;

    TcArgs args;
    args.packed = static_cast<const uint8_t*>(packed);
    args.Y = Y;
    args.status = ctx.status;
    args.M = M;
    args.N = N;
    args.K = K;
    args.group = group;
    args.kblocks = K / kTileK;
    args.splits = plan.split_k;
    args.stages = plan.stages;
    args.stage_bytes = tc_stage_bytes(BM, group);
    args.timeout_ns = ctx.timeout_ns;

    const size_t smem = static_cast<size_t>(plan.stages) * args.stage_bytes + kCtrlBytes + 1024;
    auto kern = w4a16_tc_kernel<BM, NWG, DT>;
    {   // raise the dynamic shared-memory limit once per device (not a stream operation,
        // but kept out of the steady state so that launches can be graph-captured cheaply)
        static std::mutex mu;
        static size_t configured[64] = {};
        std::lock_guard<std::mutex> lock(mu);
        const int d = ctx.device < 64 ? ctx.device : 63;
        if (configured[d] < smem) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(smem)) != cudaSuccess)
                return -3;
            configured[d] = smem;
        }
    }

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.split_k), static_cast<unsigned>(N / kTileN),
                       static_cast<unsigned>((M + BM - 1) / BM));
    cfg.blockDim = dim3(64 + 128 * NWG, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int nattr = 0;
    if (plan.split_k > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(plan.split_k);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        nattr = 1;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, map, args);
    return e == cudaSuccess ? 0 : -3;
}

}  // namespace

#ifdef W4A16_TRACE
extern "C" int w4a16_trace_read(void* host, size_t bytes) {
    if (bytes > sizeof(g_w4a16_trace)) bytes = sizeof(g_w4a16_trace);
    return cudaMemcpyFromSymbol(host, g_w4a16_trace, bytes) == cudaSuccess ? 0 : -3;
}
extern "C" int w4a16_trace_clear(void) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_w4a16_trace) != cudaSuccess) return -3;
    return cudaMemset(p, 0, sizeof(g_w4a16_trace)) == cudaSuccess ? 0 : -3;
}
#endif

uint32_t tc_stage_bytes(int tile_m, int group) {
    const uint32_t raw = static_cast<uint32_t>(tile_m) * 256u + block_bytes(group, true);
    return (raw + 1023u) & ~1023u;
}

int tc_max_stages(int tile_m, int group, int smem_budget) {
    const int avail = smem_budget - kCtrlBytes - 1024;
    int s = avail / static_cast<int>(tc_stage_bytes(tile_m, group));
    return s > kMaxStages ? kMaxStages : s;
}

int launch_tc_gemm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                   int K, int group, int dtype, void* Y, const GemmPlan& plan,
                   cudaStream_t stream) {
#define W4G_TC_CASE(BMV, NWGV)                                                            \
    case BMV:                                                                            \
        return dtype == 0                                                                \
                   ? launch_tc_instance<BMV, NWGV, 0>(ctx, A, packed, M, N, K, group, Y, \
                                                      plan, stream)                      \
                   : launch_tc_instance<BMV, NWGV, 1>(ctx, A, packed, M, N, K, group, Y, \
                                                      plan, stream);
    switch (plan.tile_m) {
        W4G_TC_CASE(16, 2)
        W4G_TC_CASE(32, 2)
        W4G_TC_CASE(64, 2)
        W4G_TC_CASE(128, 2)
        W4G_TC_CASE(256, 1)
        default:
            return -2;
    }
#undef W4G_TC_CASE
}

}  // namespace w4g
