// CUDA-core variant of the fused W4A16 GEMM for very small M (1..8 rows of A).
//
// Same packed blob and the same unpack + dequant arithmetic as the tensor-core kernel
// (one RNE rounding of (q - z) * s per weight, "W4A16 GEMM 算子浅析"
// §"计算流水线的核心哲学"), but the products are accumulated with mixed-precision
// fma.rn.f32.{f16,bf16} instead of tcgen05.  Each CTA owns 32 output channels (a
// quarter of a 128-channel tile, so one warp's 128-bit loads of a chunk cover 512
// contiguous bytes) and splits K over its 8 warps; the warps' fp32 partials are summed
// in shared memory.  No inter-CTA reduction, no global scratch.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "format.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace w4g {
namespace {

constexpr int kWarps = 8;

__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

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

template <int MM, int DT>
__global__ void __launch_bounds__(kWarps * 32) w4a16_simt_kernel(
    const uint16_t* __restrict__ A, const uint8_t* __restrict__ packed,
    uint16_t* __restrict__ Y, int* status, int M, int N, int K, int group) {
    __shared__ int s_flags;
    __shared__ const float* s_cs;
    __shared__ float red[kWarps][MM][32];
    if (threadIdx.x == 0) {
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
    const bool has_z = (flags & kFlagZeros) != 0;
    const uint32_t bb = block_bytes(group, has_z);
    const uint32_t zoff = kNibbleBytes + scale_bytes(group);

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    const int tile = static_cast<int>(blockIdx.x >> 2);
    const int r = static_cast<int>(blockIdx.x & 3) * 32 + lane;
    const int n = tile * kTileN + r;
    const int kblocks = K / kTileK;
    const uint8_t* tile_base = packed + kHeaderBytes + static_cast<size_t>(tile) * kblocks * bb;

    float acc[MM];
#pragma unroll
    for (int m = 0; m < MM; ++m) acc[m] = 0.0f;

    const int nchunks = K / kChunkK;
#pragma unroll 2
    for (int ch = warp; ch < nchunks; ch += kWarps) {
        const int kb = ch >> 2, c = ch & 3;
        const uint8_t* blk = tile_base + static_cast<size_t>(kb) * bb;
        const uint4 v = ldg_stream_v4(blk + c * 2048 + r * 16);
        const int gi = (c * kChunkK) / group;
        const uint32_t sbits = __ldg(reinterpret_cast<const uint16_t*>(blk + kNibbleBytes) + gi * kTileN + r);
        uint32_t z = 8;
        if (has_z) z = (__ldg(blk + zoff + gi * (kTileN / 2) + (r >> 1)) >> ((r & 1) * 4)) & 0xFu;
        const uint32_t zp = zero_pair<DT>(z), sp = scale_pair(sbits);
        uint32_t w[16];
        dequant_word<DT>(v.x, zp, sp, w + 0);
        dequant_word<DT>(v.y, zp, sp, w + 4);
        dequant_word<DT>(v.z, zp, sp, w + 8);
        dequant_word<DT>(v.w, zp, sp, w + 12);
        const int k0 = kb * kTileK + c * kChunkK;
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            if (m < M) {
                const uint4* ap = reinterpret_cast<const uint4*>(A + static_cast<size_t>(m) * K + k0);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 a = __ldg(ap + i);
                    acc[m] = fma_pair<DT>(w[4 * i + 0], a.x, acc[m]);
                    acc[m] = fma_pair<DT>(w[4 * i + 1], a.y, acc[m]);
                    acc[m] = fma_pair<DT>(w[4 * i + 2], a.z, acc[m]);
                    acc[m] = fma_pair<DT>(w[4 * i + 3], a.w, acc[m]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MM; ++m) red[warp][m][lane] = acc[m];
    __syncthreads();
    if (warp == 0) {
        const float cs = s_cs ? s_cs[n] : 1.0f;
#pragma unroll
        for (int m = 0; m < MM; ++m) {
            if (m < M) {
                float s = 0.0f;
#pragma unroll
                for (int w2 = 0; w2 < kWarps; ++w2) s += red[w2][m][lane];
                Y[static_cast<size_t>(m) * N + n] = f32_to_dtype_s<DT>(s * cs);
            }
        }
    }
}

template <int MM>
int launch_simt_mm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                   int K, int group, int dtype, void* Y, cudaStream_t stream) {
    const unsigned grid = static_cast<unsigned>(N / 32);
    const uint16_t* a = static_cast<const uint16_t*>(A);
    const uint8_t* p = static_cast<const uint8_t*>(packed);
    uint16_t* y = static_cast<uint16_t*>(Y);
    if (dtype == 0)
        w4a16_simt_kernel<MM, 0><<<grid, kWarps * 32, 0, stream>>>(a, p, y, ctx.status, M, N, K, group);
    else
        w4a16_simt_kernel<MM, 1><<<grid, kWarps * 32, 0, stream>>>(a, p, y, ctx.status, M, N, K, group);
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

int launch_simt_gemm(const DeviceCtx& ctx, const void* A, const void* packed, int M, int N,
                     int K, int group, int dtype, void* Y, const GemmPlan& plan,
                     cudaStream_t stream) {
    (void)plan;
    if (M <= 1) return launch_simt_mm<1>(ctx, A, packed, M, N, K, group, dtype, Y, stream);
    if (M <= 2) return launch_simt_mm<2>(ctx, A, packed, M, N, K, group, dtype, Y, stream);
    if (M <= 4) return launch_simt_mm<4>(ctx, A, packed, M, N, K, group, dtype, Y, stream);
    if (M <= 8) return launch_simt_mm<8>(ctx, A, packed, M, N, K, group, dtype, Y, stream);
    return -2;
}

}  // namespace w4g
