// CUDA-core variant of the fused W4A16 GEMM for small M (1..8 rows of A).
//
// Same packed blob and the same unpack + dequant arithmetic as the tensor-core kernel
// (one RNE rounding of (q - z) * s per weight, "W4A16 GEMM 算子浅析"
// §"计算流水线的核心哲学"); the products are accumulated with mixed-precision
// fma.rn.f32.{f16,bf16} on the CUDA cores instead of tcgen05, so neither the TMEM round
// trip of the dequantised tile nor the fixed issue cost of a narrow MMA bounds the rate.
//
// Work split.  A unit is ROWS (16 or 32) consecutive output channels over the whole K
// range.  The grid is persistent (at most as many CTAs as fit on the GPU at once); CTA b
// takes units b, b + grid, ...  Its 8 warps form 256 / ROWS K slots (a slot is ROWS
// lanes); slot p handles the 128-K blocks p, p + slots, ... of every unit, so partial
// sums never leave the CTA.  A thread owns one channel of its slot and streams, per
// block, its 64 bytes of nibbles (four 16-byte pieces, one per 32-K chunk) and the 4-byte
// words holding its scale and zero into a private ring of kGemvStages shared-memory
// stages with per-thread cp.async copies; completion is tracked per thread with
// cp.async commit groups (cp.async.wait_group), so no thread waits on another and there
// is no mbarrier.  The ring is refilled with the thread's next block -- across unit
// boundaries, so the stream never drains between units.  A is read through the L1 cache
// with broadcast 128-bit loads.  At the end of a unit the slots' fp32 partials are
// combined in shared memory in slot order (deterministic) and stored as Y.
//
// With programmatic dependent launch the header check and the first ring stages run
// before the dependency wait (the packed weights do not depend on the previous kernel);
// A is read and Y written only after it.  The kernel has no spin-wait: cp.async
// completion waits end when the thread's own copies land.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "epilogue.cuh"
#include "format.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4g {
namespace {

constexpr int kGemvWarps = 8;

// acc += lo(w) * lo(a) + hi(w) * hi(a), each product and sum rounded once in fp32.
template <int DT>
__device__ __forceinline__ float fma_pair(uint32_t w, uint32_t a, float acc) {
    if constexpr (DT == 0) {
        asm("{\n\t.reg .f16 wl, wh, al, ah;\n\t"
            "mov.b32 {wl, wh}, %1;\n\tmov.b32 {al, ah}, %2;\n\t"
            "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %0, wh, ah, %0;\n\t}"
            : "+f"(acc) : "r"(w), "r"(a));
    } else {
        asm("{\n\t.reg .b16 wl, wh, al, ah;\n\t"
            "mov.b32 {wl, wh}, %1;\n\tmov.b32 {al, ah}, %2;\n\t"
            "fma.rn.f32.bf16 %0, wl, al, %0;\n\tfma.rn.f32.bf16 %0, wh, ah, %0;\n\t}"
            : "+f"(acc) : "r"(w), "r"(a));
    }
    return acc;
}

template <int DT>
__device__ __forceinline__ uint16_t f32_to_dtype_s(float v) {
    if constexpr (DT == 0) return __half_as_ushort(__float2half_rn(v));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

constexpr int kGemvStages = 4;       // ring depth (blocks in flight per thread)
constexpr int kGemvThreads = kGemvWarps * 32;

// Asynchronous global -> shared copies of the issuing thread (cp.async, completion tracked
// per thread by commit groups).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// acc[m][i] += the products of one 16-byte chunk (32 K values) with A, word position i in
// chain i.  a_chunk: A row 0 at the chunk's first K value (read through L1); row m is K
// values further.
template <int MM, int DT>
__device__ __forceinline__ void chunk_fma(const uint4 v, uint32_t zp, uint32_t sp, uint32_t zp16,
                                          uint32_t sp16, bool x16, const uint16_t* a_chunk,
                                          int K, int M, float (&acc)[MM][4]) {
    uint32_t wd[16];
    if (DT == 0 && x16) {
        dequant_word_f16_x16(v.x, zp, sp, zp16, sp16, wd + 0);
        dequant_word_f16_x16(v.y, zp, sp, zp16, sp16, wd + 4);
        dequant_word_f16_x16(v.z, zp, sp, zp16, sp16, wd + 8);
        dequant_word_f16_x16(v.w, zp, sp, zp16, sp16, wd + 12);
    } else {
        dequant_word<DT>(v.x, zp, sp, wd + 0);
        dequant_word<DT>(v.y, zp, sp, wd + 4);
        dequant_word<DT>(v.z, zp, sp, wd + 8);
        dequant_word<DT>(v.w, zp, sp, wd + 12);
    }
#pragma unroll
    for (int m = 0; m < MM; ++m) {
        if (m < M) {
            const uint4* ap = reinterpret_cast<const uint4*>(a_chunk + static_cast<size_t>(m) * K);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 a = __ldg(ap + i);
                float t = acc[m][i];
                t = fma_pair<DT>(wd[4 * i + 0], a.x, t);
                t = fma_pair<DT>(wd[4 * i + 1], a.y, t);
                t = fma_pair<DT>(wd[4 * i + 2], a.z, t);
                t = fma_pair<DT>(wd[4 * i + 3], a.w, t);
                acc[m][i] = t;
            }
        }
    }
}

// One 128-K block of this thread's channel from its ring stage: w_s = its 64 nibble bytes
// (chunk c at + c * 4 KB), sz_s = its scale / zero words (group gi at + 8 gi).
// kChunks = 4: a full block (no per-chunk test); 0: only the first nck chunks.
template <int MM, int DT, int kChunks>
__device__ __forceinline__ void block_fma(uint32_t w_s, uint32_t sz_s, int gshift, bool has_z,
                                          int r, const uint16_t* a_blk, int K, int M,
                                          float (&acc)[MM][4], int nck = 4) {
    uint32_t zp = 0, sp = 0, zp16 = 0, sp16 = 0;
    bool x16 = false;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (kChunks == 0 && c >= nck) break;
        // the chunk starts a new group: c == 0 always, c == 2 for groups of 64 or 32,
        // odd c for groups of 32
        const bool fresh = c == 0 || (c == 2 && gshift <= 1) || ((c & 1) && gshift == 0);
        if (fresh) {
            const int gi = c >> gshift;
            const uint32_t sw = lds_u32(sz_s + gi * 8);
            const uint32_t sbits = (sw >> ((r & 1) * 16)) & 0xFFFFu;
            uint32_t z = 8;
            if (has_z) z = (lds_u32(sz_s + gi * 8 + 4) >> (((r >> 1) & 3) * 8 + (r & 1) * 4)) & 0xFu;
            zp = zero_pair<DT>(z);
            sp = scale_pair(sbits);
            if constexpr (DT == 0) {
                zp16 = zero_pair_x16(z);
                sp16 = scale_pair_div16(sp);
                x16 = f16_div16_exact(sp, sp16);
            }
        }
        const uint4 v = lds_v4(w_s + c * (kGemvThreads * 16));
        chunk_fma<MM, DT>(v, zp, sp, zp16, sp16, x16, a_blk + c * kChunkK, K, M, acc);
    }
}

template <int MM, int DT, int ROWS>
__global__ void __launch_bounds__(kGemvThreads, 2) w4a16_gemv_kernel(
    const uint16_t* __restrict__ A, const uint8_t* __restrict__ packed,
    uint16_t* __restrict__ Y, int* status, int M, int N, int K, int group, int prefetch_w,
    const EpilogueArgs epi) {
    constexpr int kSub = 32 / ROWS;            // K slots per warp
    constexpr int kSlots = kGemvWarps * kSub;
    // Ring stage s: nibbles [4 chunks][threads][16 B], then per thread and group of the
    // block the 4-byte words holding its scale and its zero: [threads][G][2][4 B].
    extern __shared__ __align__(16) uint8_t ring_smem[];
    __shared__ float red[2][kSlots][MM][ROWS];
    __shared__ int s_flags;
    __shared__ const float* s_cs;

    const int tid = static_cast<int>(threadIdx.x);
    const int warp = tid >> 5, lane = tid & 31;
    const int rl = lane % ROWS;                // channel within the unit
    const int slot = warp * kSub + lane / ROWS;

    if (tid == 0) {
        if (!prefetch_w) grid_dep_wait();
        const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed);
        const int f = check_header(h, N, K, group, DT);
        s_flags = f;
        s_cs = (f >= 0 && (f & kFlagChannelScale))
                   ? reinterpret_cast<const float*>(packed + h->cscale_offset)
                   : nullptr;
        if (f < 0 && blockIdx.x == 0) record_status(status, kStatusFormat);
    }
    __syncthreads();
    const int flags = s_flags;
    if (flags < 0) return;
    if (tid == 0) grid_dep_launch();

    const bool has_z = (flags & kFlagZeros) != 0;
    const uint32_t bb = block_bytes(group, has_z);
    const uint32_t zoff = kNibbleBytes + scale_bytes(group);
    const int G = groups_per_block(group);
    const int gshift = group == 128 ? 2 : (group == 64 ? 1 : 0);
    const int kblocks = blocks_k(K);
    const int units = tiles_n(N) * (kTileN / ROWS);
    const int grid = static_cast<int>(gridDim.x);
    const int u0 = static_cast<int>(blockIdx.x);
    const int nbs = slot < kblocks ? (kblocks - 1 - slot) / kSlots + 1 : 0;  // blocks per unit
    const int my_units = u0 < units ? (units - 1 - u0) / grid + 1 : 0;
    const int total = my_units * nbs;  // items of this thread: (unit, block) pairs in order

    const uint32_t stage_bytes = static_cast<uint32_t>(kGemvThreads) * (64u + 8u * G);
    const uint32_t ring = smem_addr(ring_smem);
    const uint32_t my_w = ring + static_cast<uint32_t>(tid) * 16u;              // + s*stage + c*4 KB
    const uint32_t my_sz = ring + 4u * kGemvThreads * 16u + static_cast<uint32_t>(tid) * 8u * G;

    // Load cursor: the next item is block slot + lj * kSlots of unit u0 + lu * grid.
    int lu = 0, lj = 0, ls = 0;
    auto issue_next = [&]() {
        const int n0 = (u0 + lu * grid) * ROWS;
        const int r = n0 % kTileN + rl;
        const uint8_t* blk = packed + kHeaderBytes +
                             (static_cast<size_t>(n0 / kTileN) * kblocks + slot + lj * kSlots) * bb;
        const uint32_t so = static_cast<uint32_t>(ls) * stage_bytes;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            cp_async16(my_w + so + c * (kGemvThreads * 16), blk + c * 2048 + r * 16);
        for (int gi = 0; gi < G; ++gi) {
            cp_async4(my_sz + so + gi * 8, blk + kNibbleBytes + gi * 256 + (r & ~1) * 2);
            if (has_z) cp_async4(my_sz + so + gi * 8 + 4, blk + zoff + gi * (kTileN / 2) + ((r >> 1) & ~3));
        }
        if (++lj == nbs) { lj = 0; ++lu; }
        if (++ls == kGemvStages) ls = 0;
    };
    int issued = 0;
#pragma unroll
    for (int i = 0; i < kGemvStages - 1; ++i) {
        if (issued < total) { issue_next(); ++issued; }
        cp_async_commit();  // empty groups keep the group count uniform
    }

    grid_dep_wait();  // A and Y belong to the previous kernel until here
    const float* cs = s_cs;
    int cs_stage = 0;  // ring stage of the next item to consume
    for (int ui = 0; ui < my_units; ++ui) {
        const int n0 = (u0 + ui * grid) * ROWS;
        const int r = n0 % kTileN + rl;
        float acc[MM][4];
#pragma unroll
        for (int m = 0; m < MM; ++m)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[m][i] = 0.0f;
        for (int j = 0; j < nbs; ++j) {
            cp_async_wait<kGemvStages - 2>();  // this thread's copies of the item have landed
            const uint32_t so = static_cast<uint32_t>(cs_stage) * stage_bytes;
            const int kb = slot + j * kSlots;
            const uint16_t* a_blk = A + kb * kTileK;
            // chunks of the block inside K (all 4 except in a padded last block, whose
            // chunks past K have zero weights and must not read A)
            const int nck = (kb + 1) * kTileK <= K ? 4 : (K - kb * kTileK) / kChunkK;
            if (nck == 4)
                block_fma<MM, DT, 4>(my_w + so, my_sz + so, gshift, has_z, r, a_blk, K, M, acc);
            else
                block_fma<MM, DT, 0>(my_w + so, my_sz + so, gshift, has_z, r, a_blk, K, M, acc,
                                     nck);
            // refill the stage consumed one item ago (its shared-memory reads are done)
            if (issued < total) { issue_next(); ++issued; }
            cp_async_commit();
            if (++cs_stage == kGemvStages) cs_stage = 0;
        }
        // Unit done: the slots' partials are summed in slot order.
#pragma unroll
        for (int m = 0; m < MM; ++m)
            red[ui & 1][slot][m][rl] = (acc[m][0] + acc[m][1]) + (acc[m][2] + acc[m][3]);
        __syncthreads();  // one barrier per unit: red is double-buffered by unit parity
        for (int e = tid; e < MM * ROWS; e += kGemvThreads) {
            const int m = e / ROWS, jr = e - (e / ROWS) * ROWS;
            if (m < M && n0 + jr < N) {  // channels past N are padding
                float sum = 0.0f;
#pragma unroll
                for (int p = 0; p < kSlots; ++p) sum += red[ui & 1][p][m][jr];
                const int n = n0 + jr;
                if (cs) sum *= cs[n];
                const float bias_n = epi.bias ? dtype_to_f32<DT>(epi.bias[n]) : 0.0f;
                const size_t o = static_cast<size_t>(m) * N + n;
                Y[o] = f32_to_dtype_s<DT>(apply_epilogue<DT>(sum, bias_n, epi, o));
            }
        }
    }
    cp_async_wait<0>();
}

template <int MM, int DT, int ROWS>
int launch_gemv_instance(const DeviceCtx& ctx, const void* A, const void* packed, int M,
                         int N, int K, int group, void* Y, const GemmPlan& plan,
                         const EpilogueArgs& epi, cudaStream_t stream) {
    auto kern = w4a16_gemv_kernel<MM, DT, ROWS>;
    const int G = groups_per_block(group);
    const size_t smem = static_cast<size_t>(kGemvStages) * kGemvThreads * (64 + 8 * G);
    static int configured_device = -1;  // attributes set once per device and instance
    static int occ[3] = {0, 0, 0};      // CTAs per SM for groups of 128, 64, 32
    const int gidx = G == 1 ? 0 : (G == 2 ? 1 : 2);
    if (configured_device != ctx.device) {
        cudaFuncAttributes fa;
        if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess ||
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 ctx.max_smem_optin - static_cast<int>(fa.sharedSizeBytes)) !=
                cudaSuccess)
            return -3;
        occ[0] = occ[1] = occ[2] = 0;
        configured_device = ctx.device;
    }
    if (occ[gidx] == 0 &&
        (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[gidx], kern, kGemvThreads, smem) !=
             cudaSuccess || occ[gidx] < 1)) {
        occ[gidx] = 0;
        return -3;
    }
    const int units = tiles_n(N) * (kTileN / ROWS);
    const int slots = occ[gidx] * ctx.num_sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units < slots ? units : slots), 1, 1);
    cfg.blockDim = dim3(kGemvThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (plan.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = static_cast<unsigned>(na);
    const cudaError_t e = cudaLaunchKernelEx(
        &cfg, kern, static_cast<const uint16_t*>(A), static_cast<const uint8_t*>(packed),
        static_cast<uint16_t*>(Y), ctx.status, M, N, K, group, plan.prefetch_weights ? 1 : 0,
        epi);
    return e == cudaSuccess ? 0 : -3;
}

template <int MM>
int launch_gemv_mm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                   int K, int group, int dtype, void* Y, const GemmPlan& plan,
                   const EpilogueArgs& epi, cudaStream_t stream) {
    if (plan.tile_m == 16)
        return dtype == 0 ? launch_gemv_instance<MM, 0, 16>(ctx, A, packed, M, N, K, group, Y, plan, epi, stream)
                          : launch_gemv_instance<MM, 1, 16>(ctx, A, packed, M, N, K, group, Y, plan, epi, stream);
    return dtype == 0 ? launch_gemv_instance<MM, 0, 32>(ctx, A, packed, M, N, K, group, Y, plan, epi, stream)
                      : launch_gemv_instance<MM, 1, 32>(ctx, A, packed, M, N, K, group, Y, plan, epi, stream);
}

}  // namespace

int launch_simt_gemm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                     int K, int group, int dtype, void* Y, const GemmPlan& plan,
                     const EpilogueArgs& epi, cudaStream_t stream) {
    if (M <= 1) return launch_gemv_mm<1>(ctx, A, packed, M, N, K, group, dtype, Y, plan, epi, stream);
    if (M <= 2) return launch_gemv_mm<2>(ctx, A, packed, M, N, K, group, dtype, Y, plan, epi, stream);
    if (M <= 4) return launch_gemv_mm<4>(ctx, A, packed, M, N, K, group, dtype, Y, plan, epi, stream);
    if (M <= 8) return launch_gemv_mm<8>(ctx, A, packed, M, N, K, group, dtype, Y, plan, epi, stream);
    return -2;
}

}  // namespace w4g
