// MX block-scaled decode GEMM: MXFP4 (E2M1) weights times MXFP8 (E4M3) activations, one
// E8M0 scale per block of 32 values along K on each side ("量化开销对比" §3 end and the
// MXFP4 / NVFP4 row of the §5 table).  The elements are decoded to fp16 by the
// conversion instructions (cvt.rn.f16x2.e2m1x2 / .e4m3x2, exact: every E2M1 and E4M3
// value is an fp16 value) and multiplied with the f16 mma.sync; each MMA step stays
// inside one 32-value scale block, so the two block scales multiply that block's fp32
// partial sum before it is accumulated.  This is not the native block-scaled MMA (its
// instruction and scale-factor encodings are not documented in this build's sources).
//
// Packed blob (private, versioned by its header):
//   [0, 128)          header (MxHeader)
//   blocks            one per (16-channel tile t, 128-K block kb), tiles in order, blocks
//                     of one tile contiguous along K; kMxBlockBytes each:
//     [0, 1024)       codes: lane l = 4g + i owns 32 bytes at 32 l, one word per MMA step
//                     j = 2c + h (scale block c, half h); the word's bytes hold the E2M1
//                     pairs (K, K + 1) and (K + 2, K + 3) of channel g, then the same of
//                     channel g + 8, for K = 32c + 8i + 4h (low nibble = the even K).
//     [1024, 1088)    word r: the four E8M0 scale codes of channel r (scale blocks 0..3).
// N is padded to a multiple of 16 (codes 0, scale code 127: weights 0); K must be a
// multiple of 128.
//
// In MMA step j the MMA's K index 2i + e stands for K value 32c + 8i + 4h + e and
// 8 + 2i + e for 32c + 8i + 4h + 2 + e, for weights and activations alike.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.h"
#include "ptx.cuh"

namespace w4g {
namespace {

constexpr uint32_t kMxMagic = 0x3446584Du;  // "MXF4"
constexpr uint32_t kMxVersion = 1;
constexpr int kMxBlockK = 128;
constexpr int kMxTileN = 16;
constexpr uint32_t kMxCodeBytes = 1024;
constexpr uint32_t kMxBlockBytes = kMxCodeBytes + 64;  // 1088
constexpr int kMxThreads = 256;
constexpr int kMxWarps = kMxThreads / 32;  // K slots of a GEMM CTA

struct MxHeader {
    uint32_t magic;
    uint32_t version;
    int32_t N;
    int32_t K;
    uint32_t block_bytes;
    uint32_t reserved0;
    uint64_t body_offset;
    uint64_t total_bytes;
    uint32_t reserved[22];
};
static_assert(sizeof(MxHeader) == 128, "header must be 128 bytes");

__host__ __device__ constexpr int mx_tiles(int N) { return (N + kMxTileN - 1) / kMxTileN; }

__device__ __forceinline__ bool mx_header_ok(const uint8_t* packed, int N, int K) {
    const MxHeader* h = reinterpret_cast<const MxHeader*>(packed);
    return h->magic == kMxMagic && h->version == kMxVersion && h->N == N && h->K == K &&
           h->block_bytes == kMxBlockBytes && h->body_offset == 128;
}

// One CTA per (tile, block); thread (j, l) = (tid / 32, tid % 32) writes word j of lane l
// (two bytes of each of its two channels, copied from the canonical rows); the first 16
// threads also write their channel's four scale codes.
__global__ void __launch_bounds__(256) mx_repack_kernel(const uint8_t* __restrict__ wc,
                                                        const uint8_t* __restrict__ ws, int N,
                                                        int K, uint8_t* __restrict__ packed) {
    const int kblocks = K / kMxBlockK;
    const int t = static_cast<int>(blockIdx.x) / kblocks;
    const int kb = static_cast<int>(blockIdx.x) - t * kblocks;
    const int j = static_cast<int>(threadIdx.x) >> 5, l = static_cast<int>(threadIdx.x) & 31;
    const int g = l >> 2, i = l & 3, c = j >> 1, h = j & 1;
    uint8_t* blk = packed + 128 + static_cast<size_t>(blockIdx.x) * kMxBlockBytes;
    const int k0 = kb * kMxBlockK + 32 * c + 8 * i + 4 * h;  // even
    uint32_t word = 0;
#pragma unroll
    for (int q = 0; q < 2; ++q) {  // channel g, then g + 8
        const int n = t * kMxTileN + g + 8 * q;
        if (n < N) {
            const uint8_t* row = wc + static_cast<size_t>(n) * (K / 2) + k0 / 2;
            word |= (static_cast<uint32_t>(row[0]) | (static_cast<uint32_t>(row[1]) << 8)) << (16 * q);
        }
    }
    *reinterpret_cast<uint32_t*>(blk + 32 * l + 4 * j) = word;
    if (threadIdx.x < kMxTileN) {
        const int r = static_cast<int>(threadIdx.x);
        const int n = t * kMxTileN + r;
        uint32_t sc = 0x7F7F7F7Fu;  // padded channels: scale 1 (their codes are 0)
        if (n < N) {
            const uint8_t* s = ws + static_cast<size_t>(n) * (K / 32) + kb * 4;
            sc = static_cast<uint32_t>(s[0]) | (static_cast<uint32_t>(s[1]) << 8) |
                 (static_cast<uint32_t>(s[2]) << 16) | (static_cast<uint32_t>(s[3]) << 24);
        }
        *reinterpret_cast<uint32_t*>(blk + kMxCodeBytes + 4 * r) = sc;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        MxHeader hd{};
        hd.magic = kMxMagic;
        hd.version = kMxVersion;
        hd.N = N;
        hd.K = K;
        hd.block_bytes = kMxBlockBytes;
        hd.body_offset = 128;
        hd.total_bytes = 128ull + static_cast<uint64_t>(mx_tiles(N)) * kblocks * kMxBlockBytes;
        *reinterpret_cast<MxHeader*>(packed) = hd;
    }
}

// A later kernel launched with programmatic dependent launch may start while this one
// still runs; this empty kernel keeps it from overlapping the repack itself.
__global__ void mx_fence_kernel() {}

__device__ __forceinline__ uint4 mx_ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Four E2M1 pairs of a word -> four fp16 pairs: bytes 0, 1 (channel g) to a0, a2 and
// bytes 2, 3 (channel g + 8) to a1, a3; the low nibble goes to the low half.
__device__ __forceinline__ void e2m1_word_to_f16(uint32_t x, uint32_t& a0, uint32_t& a1,
                                                 uint32_t& a2, uint32_t& a3) {
    asm("{\n\t.reg .b16 h0, h1;\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "mov.b32 {h0, h1}, %4;\n\tmov.b16 {t0, t1}, h0;\n\tmov.b16 {t2, t3}, h1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, t0;\n\tcvt.rn.f16x2.e2m1x2 %2, t1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, t2;\n\tcvt.rn.f16x2.e2m1x2 %3, t3;\n\t}"
        : "=r"(a0), "=r"(a1), "=r"(a2), "=r"(a3)
        : "r"(x));
}

// Four E4M3 values (K, K + 1, K + 2, K + 3) -> two fp16 pairs.
__device__ __forceinline__ void e4m3_word_to_f16(uint32_t x, uint32_t& b0, uint32_t& b1) {
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
        : "=r"(b0), "=r"(b1)
        : "r"(x));
}

__device__ __forceinline__ void mx_mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                       uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// E8M0 scale code -> 2^(e - 127) as an fp32 value (2^-127 is subnormal; 255 is NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
    if (e == 0) return __uint_as_float(0x00400000u);
    if (e == 255) return __uint_as_float(0x7FC00000u);
    return __uint_as_float(e << 23);
}

template <int DT>
__device__ __forceinline__ uint16_t mx_f32_to_dtype(float v) {
    if constexpr (DT == 0) return __half_as_ushort(__float2half_rn(v));
    else return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

struct MxCodes {
    uint4 w0, w1;    // words 0..3 and 4..7 of the lane
    uint32_t sa, sb; // scale codes of channels g and g + 8 (scale blocks in bytes 0..3)
};

// Activations of one block for a lane: for each group t, the 8 E4M3 codes of row 8t + g
// at K = 32c + 8i .. + 7 of every scale block c, and the scale words of rows 8t + 2i and
// 8t + 2i + 1 (the D columns the lane holds).
template <int NT>
struct MxActs {
    uint2 x[NT][4];
    uint32_t s0[NT], s1[NT];
};

template <int NT>
__device__ __forceinline__ void mx_block(const MxCodes& cw, const MxActs<NT>& xa,
                                         float (&acc)[NT][4]) {
    const uint32_t w[8] = {cw.w0.x, cw.w0.y, cw.w0.z, cw.w0.w, cw.w1.x, cw.w1.y, cw.w1.z, cw.w1.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        float d[NT][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) d[t][e] = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t a0, a1, a2, a3;
            e2m1_word_to_f16(w[2 * c + h], a0, a1, a2, a3);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                uint32_t b0, b1;
                e4m3_word_to_f16(h ? xa.x[t][c].y : xa.x[t][c].x, b0, b1);
                mx_mma(d[t], a0, a1, a2, a3, b0, b1);
            }
        }
        const float fw0 = e8m0_to_f32((cw.sa >> (8 * c)) & 0xFFu);
        const float fw1 = e8m0_to_f32((cw.sb >> (8 * c)) & 0xFFu);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float fa0 = e8m0_to_f32((xa.s0[t] >> (8 * c)) & 0xFFu);
            const float fa1 = e8m0_to_f32((xa.s1[t] >> (8 * c)) & 0xFFu);
            // D: (channel g, row 2i), (g, 2i + 1), (g + 8, 2i), (g + 8, 2i + 1)
            acc[t][0] += (d[t][0] * fw0) * fa0;
            acc[t][1] += (d[t][1] * fw0) * fa1;
            acc[t][2] += (d[t][2] * fw1) * fa0;
            acc[t][3] += (d[t][3] * fw1) * fa1;
        }
    }
}

// Work split as in the W4A8 GEMM: a CTA owns one 16-channel tile over the whole K range,
// its 8 warps are K slots (blocks slot, slot + 8, ...), codes and activations travel in
// registers ahead of their use (two blocks for 8 rows, one for 16), and the warps' fp32
// partials are summed in shared memory in slot order.
template <int MT, int DT>
__global__ void __launch_bounds__(kMxThreads, 3) mx_gemm_kernel(
    const uint8_t* __restrict__ ac, const uint8_t* __restrict__ as,
    const uint8_t* __restrict__ packed, uint16_t* __restrict__ Y, int* status, int M, int N,
    int K) {
    constexpr int NT = MT / 8;
    __shared__ float red[kMxWarps][kMxTileN][MT];
    __shared__ int s_ok;
    const int tid = static_cast<int>(threadIdx.x);
    const int slot = tid >> 5, l = tid & 31;
    const int g = l >> 2, i = l & 3;
    const int tile = static_cast<int>(blockIdx.x);
    if (tid == 0) {
        const int ok = mx_header_ok(packed, N, K);
        s_ok = ok;
        if (!ok && blockIdx.x == 0) record_status(status, kStatusFormat);
    }
    __syncthreads();
    if (!s_ok) return;
    if (tid == 0) grid_dep_launch();

    const int kblocks = K / kMxBlockK;
    const uint8_t* tile_p = packed + 128 + static_cast<size_t>(tile) * kblocks * kMxBlockBytes;
    auto load = [&](int kb, MxCodes& cw) {
        const uint8_t* blk = tile_p + static_cast<size_t>(kb) * kMxBlockBytes;
        cw.w0 = mx_ld_stream16(blk + 32 * l);
        cw.w1 = mx_ld_stream16(blk + 32 * l + 16);
        cw.sa = __ldg(reinterpret_cast<const unsigned int*>(blk + kMxCodeBytes + 4 * g));
        cw.sb = __ldg(reinterpret_cast<const unsigned int*>(blk + kMxCodeBytes + 4 * (g + 8)));
    };
    auto load_a = [&](int kb, MxActs<NT>& xa) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int row = 8 * t + g, r0 = 8 * t + 2 * i, r1 = r0 + 1;
#pragma unroll
            for (int c = 0; c < 4; ++c)
                xa.x[t][c] = row < M ? __ldg(reinterpret_cast<const uint2*>(
                                           ac + static_cast<size_t>(row) * K + kb * kMxBlockK +
                                           32 * c + 8 * i))
                                     : make_uint2(0u, 0u);
            xa.s0[t] = r0 < M ? __ldg(reinterpret_cast<const unsigned int*>(
                                    as + static_cast<size_t>(r0) * (K / 32) + kb * 4))
                              : 0x7F7F7F7Fu;
            xa.s1[t] = r1 < M ? __ldg(reinterpret_cast<const unsigned int*>(
                                    as + static_cast<size_t>(r1) * (K / 32) + kb * 4))
                              : 0x7F7F7F7Fu;
        }
    };

    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[t][e] = 0.0f;
    MxCodes ca, cb;
    if (slot < kblocks) load(slot, ca);
    if (slot + kMxWarps < kblocks) load(slot + kMxWarps, cb);
    grid_dep_wait();  // the activations (and Y) belong to the previous kernel until here
    MxActs<NT> xa;
    if constexpr (NT == 1) {
        MxActs<NT> xb;
        if (slot < kblocks) load_a(slot, xa);
        if (slot + kMxWarps < kblocks) load_a(slot + kMxWarps, xb);
        for (int kb = slot; kb < kblocks; kb += 2 * kMxWarps) {
            mx_block<NT>(ca, xa, acc);
            if (kb + 2 * kMxWarps < kblocks) {
                load(kb + 2 * kMxWarps, ca);
                load_a(kb + 2 * kMxWarps, xa);
            }
            if (kb + kMxWarps < kblocks) {
                mx_block<NT>(cb, xb, acc);
                if (kb + 3 * kMxWarps < kblocks) {
                    load(kb + 3 * kMxWarps, cb);
                    load_a(kb + 3 * kMxWarps, xb);
                }
            }
        }
    } else {  // 16 rows: activations one block ahead, in one set of registers
        if (slot < kblocks) load_a(slot, xa);
        for (int kb = slot; kb < kblocks; kb += 2 * kMxWarps) {
            mx_block<NT>(ca, xa, acc);
            if (kb + kMxWarps < kblocks) load_a(kb + kMxWarps, xa);
            if (kb + 2 * kMxWarps < kblocks) load(kb + 2 * kMxWarps, ca);
            if (kb + kMxWarps < kblocks) {
                mx_block<NT>(cb, xa, acc);
                if (kb + 2 * kMxWarps < kblocks) load_a(kb + 2 * kMxWarps, xa);
                if (kb + 3 * kMxWarps < kblocks) load(kb + 3 * kMxWarps, cb);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) red[slot][g + 8 * (e >> 1)][8 * t + 2 * i + (e & 1)] = acc[t][e];
    __syncthreads();
    for (int e = tid; e < kMxTileN * M; e += kMxThreads) {
        const int m = e / kMxTileN, r = e % kMxTileN;
        const int n = tile * kMxTileN + r;
        if (n < N) {
            float sum = 0.0f;
#pragma unroll
            for (int q = 0; q < kMxWarps; ++q) sum += red[q][r][m];
            Y[static_cast<size_t>(m) * N + n] = mx_f32_to_dtype<DT>(sum);
        }
    }
}

template <int MT, int DT>
int launch_mx_instance(const DeviceCtx& ctx, const uint8_t* ac, const uint8_t* as,
                       const void* packed, int M, int N, int K, void* Y, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(mx_tiles(N)), 1, 1);
    cfg.blockDim = dim3(kMxThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, mx_gemm_kernel<MT, DT>, ac, as,
                                             static_cast<const uint8_t*>(packed),
                                             static_cast<uint16_t*>(Y), ctx.status, M, N, K);
    return e == cudaSuccess ? 0 : -3;
}

}  // namespace

size_t mx_blob_bytes(int N, int K) {
    return 128ull + static_cast<size_t>(mx_tiles(N)) * (K / kMxBlockK) * kMxBlockBytes;
}

int launch_mx_repack(const DeviceCtx& ctx, const uint8_t* w_codes, const uint8_t* w_scales,
                     int N, int K, void* packed, cudaStream_t stream) {
    (void)ctx;
    const unsigned blocks = static_cast<unsigned>(mx_tiles(N) * (K / kMxBlockK));
    mx_repack_kernel<<<blocks, 256, 0, stream>>>(w_codes, w_scales, N, K,
                                                  static_cast<uint8_t*>(packed));
    if (cudaGetLastError() != cudaSuccess) return -3;
    mx_fence_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int launch_mx_gemm(const DeviceCtx& ctx, const uint8_t* a_codes, const uint8_t* a_scales,
                   const void* packed, int M, int N, int K, int dtype, void* Y,
                   cudaStream_t stream) {
    if (M <= 8)
        return dtype == 0 ? launch_mx_instance<8, 0>(ctx, a_codes, a_scales, packed, M, N, K, Y, stream)
                          : launch_mx_instance<8, 1>(ctx, a_codes, a_scales, packed, M, N, K, Y, stream);
    if (M <= 16)
        return dtype == 0 ? launch_mx_instance<16, 0>(ctx, a_codes, a_scales, packed, M, N, K, Y, stream)
                          : launch_mx_instance<16, 1>(ctx, a_codes, a_scales, packed, M, N, K, Y, stream);
    return -2;
}

}  // namespace w4g
